"""ZeRO-1 optimizer step across ranks: one process and one GPU per rank.

llm.c walk-through ch. 04 "Multi-GPU and mixed precision":
  §3.2  ZeRO-1: every rank holds the full gradients; a reduce-scatter
        (average) leaves each rank the average of its own contiguous 1/N
        shard; each rank updates only its shard's m, v and master weights;
        an all-gather puts the new bf16 weights back together on every rank.
        The parameter count must divide by the number of ranks.
  §3.3  the collectives run on their own stream, ordered against the
        compute stream by events, so the host never waits.
  §4    under ZeRO-1 the gradient norm sums the squares of the local shard
        only; the per-rank sums are then combined across ranks.
CMU 11-667 lecture 13 notes §5.2: ZeRO-1 computes what data parallelism
computes, with 1/N of the optimizer state per rank.

One step, per rank, in stream order:
  1. reduce-scatter (average) of the bf16 gradients     comm stream
  2. sum of squares of the rank's shard (mp_grad_sumsq)  compute stream
  3. all-gather of the per-rank sums (one double each)   comm stream
  4. norm and clip scale from the sums in rank order (mp_clip_scale_from_sumsq)
  5. AdamW + stochastic rounding of the shard at its global offset
     (mp_adamw_step: decay flags and rounding draws keyed on global indices)
  6. all-gather of the new bf16 weights, in place         comm stream
Every arithmetic step of the optimizer runs in the library's kernels; the
collectives are torch.distributed calls (NCCL on GPUs). The per-rank sums
are gathered rather than all-reduced, so each rank adds the same values in
the same order and every rank derives the same clip scale, bit for bit.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Tuple

import torch
import torch.distributed as dist


@dataclasses.dataclass(frozen=True)
class ShardLayout:
    """The contiguous equal shard of one rank: [offset, offset + size)."""
    n_total: int
    world: int
    rank: int

    def __post_init__(self):
        if self.world < 1 or not 0 <= self.rank < self.world:
            raise ValueError(f"rank {self.rank} of world {self.world}")
        if self.n_total % self.world:
            # llm.c ch. 04 §3.2 and §6: ZeRO-1 needs the parameter count to
            # divide by the number of ranks
            raise ValueError(f"{self.n_total} parameters do not divide into {self.world} equal shards")

    @property
    def size(self) -> int:
        return self.n_total // self.world

    @property
    def offset(self) -> int:
        return self.rank * self.size

    def slice(self) -> slice:
        return slice(self.offset, self.offset + self.size)


class LibraryKernels:
    """The library's entry points the ZeRO-1 step calls."""

    def __init__(self):
        from . import mp_adamw_step, mp_clip_scale_from_sumsq, mp_grad_norm_workspace_bytes, mp_grad_sumsq
        self.grad_sumsq = mp_grad_sumsq
        self.clip_scale_from_sumsq = mp_clip_scale_from_sumsq
        self.adamw_step = mp_adamw_step
        self.workspace_bytes = mp_grad_norm_workspace_bytes


class Zero1Optimizer:
    """The ZeRO-1 step of one rank.

    params, grads: the full flat bf16 buffers (every rank holds both);
    master, m, v: this rank's shard of the fp32 state (layout.size elements,
    for global indices layout.slice()). step() enqueues the six stages above
    and does not synchronise; the bf16 weights are whole again on every rank
    once the compute stream reaches the end of the call.
    """

    def __init__(self, table_entries: Sequence[Tuple[int, int, int]], *, lr: float, beta1: float, beta2: float,
                 eps: float, weight_decay: float, clip: float, device=None, group=None, schedule=None,
                 kernels=None):
        from . import TensorTable
        self.group = group
        self.table = TensorTable(table_entries)
        self.layout = ShardLayout(self.table.total, dist.get_world_size(group), dist.get_rank(group))
        self.hyper = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay)
        self.clip = clip
        self.schedule = schedule
        self.kernels = kernels if kernels is not None else LibraryKernels()
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.device = dev
        per, world = self.layout.size, self.layout.world
        self.grad_shard = torch.empty(per, dtype=torch.bfloat16, device=dev)
        self.sumsq_local = torch.zeros(1, dtype=torch.float64, device=dev)
        self.sumsq_all = torch.zeros(world, dtype=torch.float64, device=dev)
        self.workspace = torch.empty(max(8, self.kernels.workspace_bytes(per)), dtype=torch.uint8, device=dev)
        self.d_norm = torch.zeros(1, dtype=torch.float32, device=dev)
        self.d_scale = torch.zeros(1, dtype=torch.float32, device=dev)
        self.d_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.comm_stream = torch.cuda.Stream(dev) if dev.type == "cuda" else None

    def make_shard_state(self, master_full: Optional[torch.Tensor] = None, with_master: bool = True):
        """Zeroed m and v for this rank's shard, and its slice of a full fp32
        master (copied) when with_master."""
        per = self.layout.size
        st = dict(m=torch.zeros(per, dtype=torch.float32, device=self.device),
                  v=torch.zeros(per, dtype=torch.float32, device=self.device))
        if with_master:
            if master_full is None:
                raise ValueError("with_master needs the full fp32 master to take the shard from")
            st["master"] = master_full[self.layout.slice()].to(self.device, torch.float32, copy=True)
        return st

    def _collective(self, compute, fn):
        """Runs fn (a collective) on the comm stream after the compute
        stream's work so far; the compute stream then waits for it."""
        if self.comm_stream is None:
            fn()
            return
        self.comm_stream.wait_stream(compute)
        with torch.cuda.stream(self.comm_stream):
            fn()
        compute.wait_stream(self.comm_stream)

    def step(self, params: torch.Tensor, grads: torch.Tensor, master: Optional[torch.Tensor], m: torch.Tensor,
             v: torch.Tensor, t: int, seed: int, stream=None) -> None:
        L, K, g = self.layout, self.kernels, self.group
        if params.numel() != L.n_total or grads.numel() != L.n_total:
            raise ValueError("params and grads must be the full flat buffers")
        compute = None
        if self.comm_stream is not None:
            compute = stream if stream is not None else torch.cuda.current_stream(self.device)
        sl = L.slice()
        hyper = dict(self.hyper)
        if self.schedule is not None:
            hyper["lr"] = self.schedule.lr(t)
        # 1. each rank receives the average of its shard of everyone's gradients
        self._collective(compute, lambda: dist.reduce_scatter_tensor(self.grad_shard, grads,
                                                                     op=dist.ReduceOp.AVG, group=g))
        # 2. the local share of the norm
        K.grad_sumsq(self.grad_shard, self.workspace, self.sumsq_local, n=L.size, stream=compute)
        # 3. every rank's share, in rank order
        self._collective(compute, lambda: dist.all_gather_into_tensor(self.sumsq_all, self.sumsq_local, group=g))
        # 4. the global norm and clip scale (the same bits on every rank)
        K.clip_scale_from_sumsq(self.sumsq_all, self.clip, self.d_norm, self.d_scale, count=L.world,
                                stream=compute)
        # 5. the shard's update, keyed on global indices
        K.adamw_step(params[sl], self.grad_shard, master, m, v, self.table, d_grad_scale=self.d_scale, t=t,
                     seed=seed, global_offset=L.offset, n=L.size, d_status=self.d_status, stream=compute, **hyper)
        # 6. the new bf16 weights from every rank, in place
        self._collective(compute, lambda: dist.all_gather_into_tensor(params, params[sl], group=g))

    def take_status(self) -> int:
        """Device status of the steps since the last call (0 or
        MP_ERR_NONFINITE); clears it. Synchronises."""
        st = int(self.d_status.item())
        if st != 0:
            self.d_status.zero_()
        return st
