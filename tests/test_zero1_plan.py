"""The ZeRO-1 step on CPU ranks (gloo, world size 2): its collective plan,
and its results against plain data parallelism.

llm.c walk-through ch. 04 §3.2-§3.3 and §4: a reduce-scatter (average) of
the full gradients, each rank's sum of squares of its own shard, those sums
combined across ranks, the shard update at its global offset, an all-gather
of the new bf16 weights. Here the library's kernels are replaced by stubs
that only record their arguments and write tags (none of the optimizer's
arithmetic), and the collectives are real gloo collectives; the test checks
what each rank received and sent. A second test puts the oracle's arithmetic
behind the same calls and requires ZeRO-1 to give data parallelism's weights
and state bit for bit (CMU 11-667 lecture 13 notes §5.2: max difference 0).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mproc

N = 4096 * 6  # 24,576 parameters: two shards of 12,288
TABLE = [(0, 8192, 1), (8192, 1000, 0), (9192, N - 9192, 1)]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class StubKernels:
    """Records every call; writes only rank tags (no arithmetic)."""

    def __init__(self, rank):
        self.rank = rank
        self.log = []

    def workspace_bytes(self, n):
        return 64

    def grad_sumsq(self, grads, workspace, d_sumsq, n=None, stream=None):
        self.log.append(("sumsq", n, grads.float().unique().tolist()))
        d_sumsq.fill_(100.0 + self.rank)

    def clip_scale_from_sumsq(self, d_sumsq, clip, d_norm, d_scale, count=None, stream=None):
        self.log.append(("scale", count, d_sumsq.tolist(), clip))
        d_scale.fill_(0.25)

    def adamw_step(self, params, grads, master, m, v, table, *, d_grad_scale, t, seed, global_offset, n,
                   d_status, stream, lr, beta1, beta2, eps, weight_decay):
        self.log.append(("step", global_offset, n, params.numel(), grads.numel(), m.numel(), t, seed, lr,
                         float(d_grad_scale.item()), table.n_tensors))
        params.fill_(float(self.rank + 1))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixed_precision_adamw_gb300 import LRSchedule
        from mixed_precision_adamw_gb300.zero1 import Zero1Optimizer
        stub = StubKernels(rank)
        sched = LRSchedule("cosine", lr_max=1e-3, lr_min=1e-4, warmup=2, total=10)
        opt = Zero1Optimizer(TABLE, lr=5e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0,
                             device="cpu", kernels=stub, schedule=sched)
        st = opt.make_shard_state(torch.zeros(N, dtype=torch.float32))
        params = torch.zeros(N, dtype=torch.bfloat16)
        # rank r's gradients are all r + 1: the average of every shard is 1.5
        grads = torch.full((N,), float(rank + 1), dtype=torch.bfloat16)
        opt.step(params, grads, st["master"], st["m"], st["v"], t=3, seed=77)
        q.put((rank, opt.layout.offset, opt.layout.size, stub.log, params.float().tolist()[::4096],
               sched.lr(3)))
    finally:
        dist.destroy_process_group()


def test_zero1_collective_plan_gloo():
    world = 2
    port = _free_port()
    ctx = mproc.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    per = N // world
    for rank, offset, size, log, params, lr3 in out:
        assert (offset, size) == (rank * per, per)
        kinds = [e[0] for e in log]
        assert kinds == ["sumsq", "scale", "step"]
        # reduce-scatter with the average: the shard holds (1 + 2) / 2
        assert log[0][1] == per and log[0][2] == [1.5]
        # the per-rank sums gathered in rank order, the same on every rank
        assert log[1][1] == world and log[1][2] == [100.0, 101.0] and log[1][3] == 1.0
        # the shard step: global offset, shard-sized arrays, the full table,
        # the device clip scale, the scheduled learning rate of step 3
        _, goff, n, np_, ng, nm, t, seed, lr, scale, ntab = log[2]
        assert (goff, n, np_, ng, nm) == (rank * per, per, per, per, per)
        assert (t, seed, scale, ntab) == (3, 77, 0.25, len(TABLE))
        assert lr == pytest.approx(lr3) and lr < 1e-3
        # the in-place all-gather: every rank now holds each rank's shard
        assert params == [1.0] * (per // 4096) + [2.0] * (per // 4096)


def test_shard_layout_rules():
    from mixed_precision_adamw_gb300.zero1 import ShardLayout
    L = ShardLayout(1_557_686_400, 8, 3)  # GPT-2 1.5B over 8 ranks
    assert (L.size, L.offset) == (194_710_800, 3 * 194_710_800)
    assert ShardLayout(8_030_261_248, 8, 7).offset == 7 * 1_003_782_656
    with pytest.raises(ValueError):
        ShardLayout(10, 3, 0)  # must divide (llm.c ch. 04 §3.2)
    with pytest.raises(ValueError):
        ShardLayout(12, 3, 3)


class OracleKernels:
    """The oracle's arithmetic behind the ZeRO-1 driver's three kernel calls,
    on CPU tensors (test-only: it checks the driver's plumbing with real
    arithmetic, not the CUDA kernels)."""

    def __init__(self):
        import oracle
        self.o = oracle

    def workspace_bytes(self, n):
        return 64

    @staticmethod
    def _u16(t):
        import numpy as np
        return t.view(torch.int16).numpy().view(np.uint16)

    def grad_sumsq(self, grads, workspace, d_sumsq, n=None, stream=None):
        d_sumsq.fill_(self.o.sumsq(self._u16(grads)))

    def clip_scale_from_sumsq(self, d_sumsq, clip, d_norm, d_scale, count=None, stream=None):
        _, nrm, sc = self.o.norm_from_parts(d_sumsq.numpy(), clip)
        d_norm.fill_(float(nrm))
        d_scale.fill_(float(sc))

    def adamw_step(self, params, grads, master, m, v, table, *, d_grad_scale, t, seed, global_offset, n,
                   d_status, stream, lr, beta1, beta2, eps, weight_decay):
        entries = [(table.ctypes_array[i].offset, table.ctypes_array[i].size, table.ctypes_array[i].decay)
                   for i in range(table.n_tensors)]
        st = self.o.adamw_step(self._u16(params), self._u16(grads), master.numpy() if master is not None else None,
                               m.numpy(), v.numpy(), global_offset, entries, lr, beta1, beta2, eps, weight_decay,
                               float(d_grad_scale.item()), t, seed)
        assert st == 0


def _pow2_grads(rank, step, n):
    """+-2^k gradients (k in [-12, -5]): the two ranks' average (the
    collective's own bf16 arithmetic, the same in the reduce-scatter and the
    all-reduce) has few significant bits and a narrow range, so every sum of
    its squares is exact in fp64 and the ZeRO-1 and data-parallel norms
    agree exactly."""
    g = torch.Generator().manual_seed(1000 * step + rank)
    k = torch.randint(-12, -4, (n,), generator=g).float()
    s = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0)
    return (s * torch.exp2(k)).to(torch.bfloat16)


def _dp_worker(rank, world, port, q, with_master=True):
    """Three steps of ZeRO-1 (the driver, oracle arithmetic) and of plain data
    parallelism (all-reduce average, every rank the whole buffer) from the
    same state: the weights must agree bit for bit (CMU 11-667 lecture 13
    notes §5.2: maximum difference 0)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from mixed_precision_adamw_gb300.zero1 import Zero1Optimizer
        H = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
        gen = torch.Generator().manual_seed(5)
        master0 = torch.randn(N, generator=gen) * 0.02
        zopt = Zero1Optimizer(TABLE, clip=1.0, device="cpu", kernels=OracleKernels(), **H)
        z = zopt.make_shard_state(master0, with_master=with_master)
        z_params = master0.to(torch.bfloat16)
        d_params, d_master = master0.to(torch.bfloat16), (master0.clone() if with_master else None)
        d_m, d_v = torch.zeros(N), torch.zeros(N)
        u16 = OracleKernels._u16
        for t in (1, 2, 3):
            g = _pow2_grads(rank, t, N)
            zopt.step(z_params, g.clone(), z.get("master"), z["m"], z["v"], t=t, seed=100 + t)
            avg = g.clone()
            dist.all_reduce(avg, op=dist.ReduceOp.AVG)
            _, _, sc = oracle.grad_norm(u16(avg), 1.0)
            assert oracle.adamw_step(u16(d_params), u16(avg), d_master.numpy() if with_master else None,
                                     d_m.numpy(), d_v.numpy(), 0, TABLE,
                                     H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], float(sc), t,
                                     100 + t) == 0
        sl = zopt.layout.slice()
        q.put((rank, torch.equal(z_params.view(torch.int16), d_params.view(torch.int16)),
               torch.equal(z["master"], d_master[sl]) if with_master else True,
               torch.equal(z["m"], d_m[sl]), torch.equal(z["v"], d_v[sl])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("with_master", [True, False])
def test_zero1_equals_data_parallel_bit_for_bit_gloo(with_master):
    world = 2
    port = _free_port()
    ctx = mproc.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_dp_worker, args=(r, world, port, q, with_master)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, params_eq, master_eq, m_eq, v_eq in out:
        assert params_eq and master_eq and m_eq and v_eq, (rank, params_eq, master_eq, m_eq, v_eq)
