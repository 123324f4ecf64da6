"""mixed_precision_adamw_gb300 — Python binding of libmpadamw.so.

A thin ctypes layer over the C ABI in include/mp_adamw.h: it checks tensor
dtypes, devices and sizes, passes raw device pointers and the current CUDA
stream, and raises MpError on a non-OK status. Every step of the optimizer
runs in the library's CUDA kernels; there is no fallback of any kind, and
importing this package fails if the compiled library is missing.

PyTorch is used only for device memory and streams. bf16 arrays are passed
as torch.bfloat16 (or int16/uint16) tensors holding the raw patterns.
"""
from __future__ import annotations

import ctypes
import os
from contextlib import nullcontext as _nullcontext
from typing import Iterable, Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmpadamw.so")

MP_OK = 0
MP_ERR_NULL = 1
MP_ERR_ALIGN = 2
MP_ERR_TABLE = 3
MP_ERR_RANGE = 4
MP_ERR_NONFINITE = 5
MP_ERR_CUDA = 6
MP_ERR_WORKSPACE = 7
MP_SKIPPED_OUTLIER = 8
MP_ERR_ACCESS = 9


class MpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}"
                         + (f" (cudaError {last_cuda_error()})" if status == MP_ERR_CUDA else ""))


class MpTensor(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_uint64), ("size", ctypes.c_uint64),
                ("decay", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class MpHyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("clip", ctypes.c_float)]


class MpLaunch(ctypes.Structure):
    """mp_launch_t: one kernel launch of a step (mp_step_launches)."""
    _fields_ = [("offset", ctypes.c_uint64), ("size", ctypes.c_uint64), ("segments", ctypes.c_uint32),
                ("first_decay", ctypes.c_uint32)]


class MpLrSchedule(ctypes.Structure):
    """mp_lr_schedule_t: a learning-rate schedule (mp_lr_at)."""
    _fields_ = [("kind", ctypes.c_int32), ("reserved", ctypes.c_int32), ("warmup", ctypes.c_int64),
                ("total", ctypes.c_int64), ("lr_max", ctypes.c_float), ("lr_min", ctypes.c_float),
                ("decay_frac", ctypes.c_float), ("reserved2", ctypes.c_float)]


class MpStepState(ctypes.Structure):
    """mp_step_state_t: the device step counter of replayable steps (32 B)."""
    _fields_ = [("t", ctypes.c_int32), ("seed_base", ctypes.c_uint32), ("lr", ctypes.c_float),
                ("reserved0", ctypes.c_uint32), ("seed", ctypes.c_uint32), ("bc1", ctypes.c_float),
                ("bc2", ctypes.c_float), ("reserved1", ctypes.c_uint32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python mixed_precision_adamw_gb300/build.py` "
            "(nvcc, sm_103a). There is no fallback path.")
    L = ctypes.CDLL(LIB_PATH)
    vp, u64, u32, i32, f32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_float
    L.mp_abi_version.restype = ctypes.c_int
    L.mp_abi_version.argtypes = []
    L.mp_status_string.restype = ctypes.c_char_p
    L.mp_status_string.argtypes = [ctypes.c_int]
    L.mp_last_cuda_error.restype = ctypes.c_int
    L.mp_last_cuda_error.argtypes = []
    L.mp_grad_norm_workspace_bytes.restype = ctypes.c_size_t
    L.mp_grad_norm_workspace_bytes.argtypes = [u64]
    L.mp_grad_norm.restype = ctypes.c_int
    L.mp_grad_norm.argtypes = [vp, u64, f32, vp, ctypes.c_size_t, vp, vp, vp, vp]
    L.mp_grad_sumsq.restype = ctypes.c_int
    L.mp_grad_sumsq.argtypes = [vp, u64, vp, ctypes.c_size_t, vp, vp]
    L.mp_clip_scale_from_sumsq.restype = ctypes.c_int
    L.mp_clip_scale_from_sumsq.argtypes = [vp, i32, f32, vp, vp, vp, vp]
    L.mp_lr_at.restype = ctypes.c_int
    L.mp_lr_at.argtypes = [ctypes.POINTER(MpLrSchedule), ctypes.c_int64, ctypes.POINTER(ctypes.c_float)]
    L.mp_copy_from_host.restype = ctypes.c_int
    L.mp_copy_from_host.argtypes = [vp, vp, u64, i32, vp]
    L.mp_adamw_step.restype = ctypes.c_int
    L.mp_adamw_step.argtypes = [vp, vp, vp, vp, vp, u64, u64, ctypes.POINTER(MpTensor), i32,
                                f32, f32, f32, f32, f32, vp, i32, u32, vp, vp]
    L.mp_stochastic_round.restype = ctypes.c_int
    L.mp_stochastic_round.argtypes = [vp, vp, u64, u64, u32, vp]
    L.mp_stochastic_round_fp16.restype = ctypes.c_int
    L.mp_stochastic_round_fp16.argtypes = [vp, vp, u64, u64, u32, vp]
    L.mp_accumulate_sr.restype = ctypes.c_int
    L.mp_accumulate_sr.argtypes = [vp, vp, u64, u64, u32, vp]
    L.mp_noise_u32.restype = ctypes.c_int
    L.mp_noise_u32.argtypes = [vp, u64, u64, u32, vp]
    L.mp_outlier_state_bytes.restype = ctypes.c_size_t
    L.mp_outlier_state_bytes.argtypes = []
    L.mp_outlier_reset.restype = ctypes.c_int
    L.mp_outlier_reset.argtypes = [vp, vp]
    L.mp_outlier_check.restype = ctypes.c_int
    L.mp_outlier_check.argtypes = [vp, vp, f32, vp, vp, vp, vp]
    L.mp_optimizer_step.restype = ctypes.c_int
    L.mp_optimizer_step.argtypes = [vp, vp, vp, vp, vp, vp, u64, ctypes.POINTER(MpTensor), i32,
                                    ctypes.POINTER(MpHyper), i32, u32, vp, ctypes.c_size_t, vp, f32, vp,
                                    vp, vp, vp, vp, vp]
    L.mp_grad_norm_noalloc.restype = ctypes.c_int
    L.mp_grad_norm_noalloc.argtypes = [vp, u64, f32, vp, vp, vp, vp]
    L.mp_step_launches.restype = ctypes.c_int
    L.mp_step_launches.argtypes = [u64, u64, ctypes.POINTER(MpTensor), i32, vp, ctypes.c_int64,
                                   ctypes.POINTER(ctypes.c_int64)]
    L.mp_bias_table_len.restype = ctypes.c_int64
    L.mp_bias_table_len.argtypes = [f32, f32]
    L.mp_bias_table.restype = ctypes.c_int
    L.mp_bias_table.argtypes = [f32, f32, ctypes.c_int64, vp]
    L.mp_optimizer_step_graph.restype = ctypes.c_int
    L.mp_optimizer_step_graph.argtypes = [vp, vp, vp, vp, vp, vp, u64, ctypes.POINTER(MpTensor), i32,
                                          ctypes.POINTER(MpHyper), vp, vp, ctypes.c_int64, vp, ctypes.c_size_t,
                                          vp, f32, vp, vp, vp, vp, vp, vp]
    return L


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def abi_version() -> int:
    return int(_lib.mp_abi_version())


def status_string(status: int) -> str:
    return _lib.mp_status_string(status).decode()


def last_cuda_error() -> int:
    return int(_lib.mp_last_cuda_error())


def _check(status: int, what: str):
    if status != MP_OK:
        raise MpError(status, what)


_BF16_LIKE = (torch.bfloat16, torch.int16, torch.uint16)


def _ptr(t: Optional[torch.Tensor], dtypes, name: str, n: Optional[int] = None) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if n is not None and t.numel() < n:
        raise ValueError(f"{name}: {t.numel()} elements < {n}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class TensorTable:
    """The flat parameter buffer's tensor table, packed once for reuse.

    entries: iterable of (offset, size, decay) with global element offsets.
    """

    def __init__(self, entries: Iterable[Tuple[int, int, int]]):
        entries = list(entries)
        self.n_tensors = len(entries)
        self._arr = (MpTensor * max(1, self.n_tensors))()
        for i, (off, size, decay) in enumerate(entries):
            self._arr[i].offset = int(off)
            self._arr[i].size = int(size)
            self._arr[i].decay = int(decay)
            self._arr[i].reserved = 0
        self.total = (entries[-1][0] + entries[-1][1]) if entries else 0

    @property
    def ctypes_array(self):
        return self._arr


def mp_grad_norm_workspace_bytes(n: int) -> int:
    return int(_lib.mp_grad_norm_workspace_bytes(n))


def mp_grad_norm(grads: torch.Tensor, clip: float, workspace: torch.Tensor, d_norm: torch.Tensor,
                 d_scale: torch.Tensor, d_sumsq: Optional[torch.Tensor] = None, n: Optional[int] = None,
                 stream=None) -> None:
    """Enqueue the global gradient norm and clip scale (device outputs)."""
    n = grads.numel() if n is None else n
    st = _lib.mp_grad_norm(
        _ptr(grads, _BF16_LIKE, "grads", n), n, clip,
        _ptr(workspace, (torch.uint8, torch.float64, torch.int64), "workspace"),
        workspace.numel() * workspace.element_size(),
        _ptr(d_norm, (torch.float32,), "d_norm", 1), _ptr(d_scale, (torch.float32,), "d_scale", 1),
        _ptr(d_sumsq, (torch.float64,), "d_sumsq", 1), _stream(stream))
    _check(st, "mp_grad_norm")


def mp_grad_sumsq(grads: torch.Tensor, workspace: torch.Tensor, d_sumsq: torch.Tensor, n: Optional[int] = None,
                  stream=None) -> None:
    """Enqueue the sum of squares of grads (mp_grad_norm's, bit for bit)
    into the device double d_sumsq: one rank's share of a ZeRO-1 norm."""
    n = grads.numel() if n is None else n
    st = _lib.mp_grad_sumsq(
        _ptr(grads, _BF16_LIKE, "grads", n), n,
        _ptr(workspace, (torch.uint8, torch.float64, torch.int64), "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(d_sumsq, (torch.float64,), "d_sumsq", 1),
        _stream(stream))
    _check(st, "mp_grad_sumsq")


def mp_clip_scale_from_sumsq(d_sumsq: torch.Tensor, clip: float, d_norm: torch.Tensor, d_scale: torch.Tensor,
                             d_total: Optional[torch.Tensor] = None, count: Optional[int] = None,
                             stream=None) -> None:
    """Enqueue the norm and clip scale from `count` per-rank sums of squares
    (device float64, rank order), added left to right in fp64."""
    count = d_sumsq.numel() if count is None else count
    st = _lib.mp_clip_scale_from_sumsq(
        _ptr(d_sumsq, (torch.float64,), "d_sumsq", count), count, clip,
        _ptr(d_norm, (torch.float32,), "d_norm", 1), _ptr(d_scale, (torch.float32,), "d_scale", 1),
        _ptr(d_total, (torch.float64,), "d_total", 1), _stream(stream))
    _check(st, "mp_clip_scale_from_sumsq")


LR_KINDS = {"constant": 0, "cosine": 1, "linear": 2, "wsd": 3}


class LRSchedule:
    """A learning-rate schedule of the library (mp_lr_at): linear warm-up,
    then constant, cosine, linear or WSD (warm-up, stable, decay)."""

    def __init__(self, kind: str, *, lr_max: float, lr_min: float = 0.0, warmup: int = 0, total: int = 0,
                 decay_frac: float = 0.0):
        if kind not in LR_KINDS:
            raise ValueError(f"kind: one of {sorted(LR_KINDS)}")
        self.kind = kind
        self._s = MpLrSchedule(LR_KINDS[kind], 0, int(warmup), int(total), float(lr_max), float(lr_min),
                               float(decay_frac), 0.0)
        self.lr(max(1, int(warmup) + 1))  # validates the schedule

    def lr(self, t: int) -> float:
        """Learning rate of the 1-based step t."""
        out = ctypes.c_float()
        _check(_lib.mp_lr_at(ctypes.byref(self._s), int(t), ctypes.byref(out)), "mp_lr_at")
        return out.value


def mp_copy_from_host(dst: torch.Tensor, host_src: torch.Tensor, nbytes: Optional[int] = None,
                      blocks_per_sm: int = 1, stream=None) -> None:
    """Enqueue a host-to-device copy of page-locked host memory done by the
    SMs (blocks_per_sm blocks of 256 threads per SM)."""
    if not isinstance(dst, torch.Tensor) or not dst.is_cuda or not dst.is_contiguous():
        raise ValueError("dst: contiguous CUDA tensor expected")
    if not isinstance(host_src, torch.Tensor) or host_src.is_cuda or not host_src.is_contiguous():
        raise ValueError("host_src: contiguous host tensor expected")
    if dst.device.index != torch.cuda.current_device():
        raise ValueError(f"dst: on {dst.device}, but the current device is cuda:{torch.cuda.current_device()}")
    avail = min(dst.numel() * dst.element_size(), host_src.numel() * host_src.element_size())
    nbytes = host_src.numel() * host_src.element_size() if nbytes is None else nbytes
    if nbytes > avail:
        raise ValueError(f"nbytes {nbytes} > {avail} bytes available")
    _check(_lib.mp_copy_from_host(dst.data_ptr(), host_src.data_ptr(), nbytes, blocks_per_sm, _stream(stream)),
           "mp_copy_from_host")


def mp_grad_norm_noalloc(grads: torch.Tensor, clip: float, d_norm: torch.Tensor, d_scale: torch.Tensor,
                         d_sumsq: Optional[torch.Tensor] = None, n: Optional[int] = None, stream=None) -> None:
    """mp_grad_norm for callers that cannot allocate device memory: no
    workspace; the partial sums live in a small scratch array inside the
    library. Calls that overlap on one GPU race on that scratch."""
    n = grads.numel() if n is None else n
    st = _lib.mp_grad_norm_noalloc(
        _ptr(grads, _BF16_LIKE, "grads", n), n, clip, _ptr(d_norm, (torch.float32,), "d_norm", 1),
        _ptr(d_scale, (torch.float32,), "d_scale", 1), _ptr(d_sumsq, (torch.float64,), "d_sumsq", 1),
        _stream(stream))
    _check(st, "mp_grad_norm_noalloc")


def mp_adamw_step(params: torch.Tensor, grads: torch.Tensor, master: Optional[torch.Tensor],
                  m: torch.Tensor, v: torch.Tensor, table: TensorTable, *, lr: float, beta1: float,
                  beta2: float, eps: float, weight_decay: float, d_grad_scale: Optional[torch.Tensor],
                  t: int, seed: int, global_offset: int = 0, n: Optional[int] = None,
                  d_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Enqueue one AdamW + stochastic-rounding step over [global_offset, global_offset + n)."""
    n = m.numel() if n is None else n
    st = _lib.mp_adamw_step(
        _ptr(params, _BF16_LIKE, "params", n), _ptr(grads, _BF16_LIKE, "grads", n),
        _ptr(master, (torch.float32,), "master", n), _ptr(m, (torch.float32,), "m", n),
        _ptr(v, (torch.float32,), "v", n), global_offset, n, table.ctypes_array, table.n_tensors,
        lr, beta1, beta2, eps, weight_decay, _ptr(d_grad_scale, (torch.float32,), "d_grad_scale", 1),
        t, seed & 0xFFFFFFFF, _ptr(d_status, (torch.int32,), "d_status", 1), _stream(stream))
    _check(st, "mp_adamw_step")


def mp_stochastic_round(out: torch.Tensor, inp: torch.Tensor, seed: int, global_offset: int = 0,
                        n: Optional[int] = None, stream=None) -> None:
    """Enqueue out[i] = SR(inp[i], global_offset + i, seed)."""
    n = inp.numel() if n is None else n
    st = _lib.mp_stochastic_round(_ptr(out, _BF16_LIKE, "out", n), _ptr(inp, (torch.float32,), "in", n),
                                  global_offset, n, seed & 0xFFFFFFFF, _stream(stream))
    _check(st, "mp_stochastic_round")


_FP16_LIKE = (torch.float16, torch.int16, torch.uint16)


def mp_stochastic_round_fp16(out: torch.Tensor, inp: torch.Tensor, seed: int, global_offset: int = 0,
                             n: Optional[int] = None, stream=None) -> None:
    """Enqueue out[i] = fp16 stochastic rounding of inp[i] (draws keyed on
    global_offset + i and seed, as the bf16 rounding)."""
    n = inp.numel() if n is None else n
    st = _lib.mp_stochastic_round_fp16(_ptr(out, _FP16_LIKE, "out", n), _ptr(inp, (torch.float32,), "in", n),
                                       global_offset, n, seed & 0xFFFFFFFF, _stream(stream))
    _check(st, "mp_stochastic_round_fp16")


def mp_accumulate_sr(acc: torch.Tensor, delta: torch.Tensor, seed: int, global_offset: int = 0,
                     n: Optional[int] = None, stream=None) -> None:
    """Enqueue acc[i] = SR((float)acc[i] + delta[i], global_offset + i, seed),
    in place on the bf16 tensor acc."""
    n = delta.numel() if n is None else n
    st = _lib.mp_accumulate_sr(_ptr(acc, _BF16_LIKE, "acc", n), _ptr(delta, (torch.float32,), "delta", n),
                               global_offset, n, seed & 0xFFFFFFFF, _stream(stream))
    _check(st, "mp_accumulate_sr")


def mp_noise_u32(out: torch.Tensor, first_index: int, seed: int, n: Optional[int] = None, stream=None) -> None:
    """Enqueue out[i] = noise(first_index + i, seed) (the rounding draws)."""
    n = out.numel() if n is None else n
    st = _lib.mp_noise_u32(_ptr(out, (torch.int32, torch.uint32), "out", n), first_index, n,
                           seed & 0xFFFFFFFF, _stream(stream))
    _check(st, "mp_noise_u32")


def _host_ptr(t: Optional[torch.Tensor], dtypes, name: str, n: Optional[int] = None) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name}: must be a host (CPU) tensor")
    if t.dtype not in dtypes or not t.is_contiguous():
        raise TypeError(f"{name}: contiguous tensor of {dtypes} expected")
    if n is not None and t.numel() < n:
        raise ValueError(f"{name}: {t.numel()} elements < {n}")
    return t.data_ptr()


def mp_optimizer_step(params: torch.Tensor, grads: torch.Tensor, master: Optional[torch.Tensor], m: torch.Tensor,
                      v: torch.Tensor, table: "TensorTable", hyper: MpHyper, *, t: int, seed: int,
                      workspace: torch.Tensor, d_norm: torch.Tensor, d_scale: torch.Tensor,
                      d_status: Optional[torch.Tensor] = None, outlier_state: Optional[torch.Tensor] = None,
                      outlier_z: float = 0.0, d_z: Optional[torch.Tensor] = None,
                      host_grads: Optional[torch.Tensor] = None,
                      host_norm: Optional[torch.Tensor] = None, n: Optional[int] = None, stream=None) -> None:
    """Enqueue the whole step: norm + clip scale, optional outlier check, AdamW + SR.
    host_grads (pinned CPU bf16) is read by the norm kernel, which fills `grads`."""
    n = m.numel() if n is None else n
    st = _lib.mp_optimizer_step(
        _ptr(params, _BF16_LIKE, "params", n), _ptr(grads, _BF16_LIKE, "grads", n),
        _host_ptr(host_grads, _BF16_LIKE, "host_grads", n),
        _ptr(master, (torch.float32,), "master", n), _ptr(m, (torch.float32,), "m", n),
        _ptr(v, (torch.float32,), "v", n), n, table.ctypes_array, table.n_tensors, ctypes.byref(hyper), t,
        seed & 0xFFFFFFFF, _ptr(workspace, (torch.uint8, torch.float64, torch.int64), "workspace"),
        workspace.numel() * workspace.element_size(),
        _ptr(outlier_state, (torch.uint8, torch.float64), "outlier_state"), outlier_z,
        _ptr(d_z, (torch.float64,), "d_z", 1), _ptr(d_norm, (torch.float32,), "d_norm", 1), _ptr(d_scale, (torch.float32,), "d_scale", 1),
        _ptr(d_status, (torch.int32,), "d_status", 1), _host_ptr(host_norm, (torch.float32,), "host_norm", 1),
        _stream(stream))
    _check(st, "mp_optimizer_step")


def mp_step_launches(global_offset: int, n: int, table: "TensorTable"):
    """How mp_adamw_step splits [global_offset, global_offset + n) into kernel
    launches: a list of (offset, size, segments, first_decay). Host only."""
    count = ctypes.c_int64()
    _check(_lib.mp_step_launches(global_offset, n, table.ctypes_array, table.n_tensors, None, 0,
                                 ctypes.byref(count)), "mp_step_launches")
    out = (MpLaunch * max(1, count.value))()
    _check(_lib.mp_step_launches(global_offset, n, table.ctypes_array, table.n_tensors, out, count.value,
                                 ctypes.byref(count)), "mp_step_launches")
    return [(x.offset, x.size, x.segments, x.first_decay) for x in out[:count.value]]


def mp_bias_table_len(beta1: float, beta2: float) -> int:
    """Entries the bias-correction table needs (0: betas out of range)."""
    return int(_lib.mp_bias_table_len(beta1, beta2))


def mp_bias_table(beta1: float, beta2: float, length: Optional[int] = None) -> torch.Tensor:
    """The host-computed bias corrections (bc1(t), bc2(t)) for t = 1..length
    as a CPU float32 tensor of 2*length values (mp_bias_table)."""
    length = mp_bias_table_len(beta1, beta2) if length is None else length
    out = torch.empty(2 * max(1, length), dtype=torch.float32)
    _check(_lib.mp_bias_table(beta1, beta2, length, out.data_ptr()), "mp_bias_table")
    return out


def mp_optimizer_step_graph(params: torch.Tensor, grads: torch.Tensor, master: Optional[torch.Tensor],
                            m: torch.Tensor, v: torch.Tensor, table: "TensorTable", hyper: MpHyper, *,
                            d_state: torch.Tensor, d_bias: torch.Tensor, workspace: torch.Tensor,
                            d_norm: torch.Tensor, d_scale: torch.Tensor, d_status: Optional[torch.Tensor] = None,
                            outlier_state: Optional[torch.Tensor] = None, outlier_z: float = 0.0,
                            d_z: Optional[torch.Tensor] = None, host_grads: Optional[torch.Tensor] = None,
                            host_norm: Optional[torch.Tensor] = None, n: Optional[int] = None,
                            stream=None) -> None:
    """mp_optimizer_step with t, seed and lr taken from the device step state
    (d_state: 32 bytes of device memory holding an mp_step_state_t), so one
    captured CUDA graph of this call serves every later step."""
    n = m.numel() if n is None else n
    if d_state.numel() * d_state.element_size() < ctypes.sizeof(MpStepState):
        raise ValueError("d_state: smaller than mp_step_state_t")
    st = _lib.mp_optimizer_step_graph(
        _ptr(params, _BF16_LIKE, "params", n), _ptr(grads, _BF16_LIKE, "grads", n),
        _host_ptr(host_grads, _BF16_LIKE, "host_grads", n),
        _ptr(master, (torch.float32,), "master", n), _ptr(m, (torch.float32,), "m", n),
        _ptr(v, (torch.float32,), "v", n), n, table.ctypes_array, table.n_tensors, ctypes.byref(hyper),
        _ptr(d_state, (torch.uint8, torch.int32), "d_state"), _ptr(d_bias, (torch.float32,), "d_bias", 2),
        d_bias.numel() // 2, _ptr(workspace, (torch.uint8, torch.float64, torch.int64), "workspace"),
        workspace.numel() * workspace.element_size(),
        _ptr(outlier_state, (torch.uint8, torch.float64), "outlier_state"), outlier_z,
        _ptr(d_z, (torch.float64,), "d_z", 1), _ptr(d_norm, (torch.float32,), "d_norm", 1),
        _ptr(d_scale, (torch.float32,), "d_scale", 1), _ptr(d_status, (torch.int32,), "d_status", 1),
        _host_ptr(host_norm, (torch.float32,), "host_norm", 1), _stream(stream))
    _check(st, "mp_optimizer_step_graph")


def mp_outlier_state_bytes() -> int:
    return int(_lib.mp_outlier_state_bytes())


def mp_outlier_reset(d_state: torch.Tensor, stream=None) -> None:
    _check(_lib.mp_outlier_reset(_ptr(d_state, (torch.uint8, torch.float64), "d_state", None), _stream(stream)),
           "mp_outlier_reset")


def mp_outlier_check(d_state: torch.Tensor, d_norm: torch.Tensor, z_threshold: float, d_scale: torch.Tensor,
                     d_z: Optional[torch.Tensor] = None, d_status: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    """Enqueue the grad-norm z-score check; a skip sets *d_scale to NaN."""
    if d_state.numel() * d_state.element_size() < mp_outlier_state_bytes():
        raise ValueError("d_state: smaller than mp_outlier_state_bytes()")
    st = _lib.mp_outlier_check(
        _ptr(d_state, (torch.uint8, torch.float64), "d_state"), _ptr(d_norm, (torch.float32,), "d_norm", 1),
        z_threshold, _ptr(d_scale, (torch.float32,), "d_scale", 1), _ptr(d_z, (torch.float64,), "d_z", 1),
        _ptr(d_status, (torch.int32,), "d_status", 1), _stream(stream))
    _check(st, "mp_outlier_check")


class OutlierDetector:
    """Device state of the grad-norm outlier check (window of 128 norms)."""

    def __init__(self, z_threshold: float, device=None):
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.z_threshold = float(z_threshold)
        self.state = torch.zeros(mp_outlier_state_bytes(), dtype=torch.uint8, device=dev)
        self.d_z = torch.full((1,), float("nan"), dtype=torch.float64, device=dev)

    def check(self, d_norm, d_scale, d_status=None, stream=None):
        mp_outlier_check(self.state, d_norm, self.z_threshold, d_scale, self.d_z, d_status, stream=stream)


class Optimizer:
    """The device state of the optimizer step: workspace, norm/scale/status
    scalars, the packed tensor table and (with outlier_z) the outlier window.

    step() makes one mp_optimizer_step call on the given (default: current)
    stream — norm and clip scale, the optional outlier check, the AdamW + SR
    update — and does not synchronise (up to 32,768 parameters the library
    runs it as one cluster launch, otherwise as the norm, finalize and update
    kernels; the results are the same). take_status() (which synchronises)
    tells whether a step was refused for a non-finite norm or skipped as an
    outlier; check_status() raises MpError instead.

    For CUDA graphs, init_device_clock() moves the step count, rounding seed
    and learning rate into device memory and step_graph() takes the next step
    from there (mp_optimizer_step_graph): capture one step_graph() call and
    replay the graph once per training step.
    """

    def __init__(self, table_entries: Sequence[Tuple[int, int, int]], *, lr: float, beta1: float,
                 beta2: float, eps: float, weight_decay: float, clip: float, device=None,
                 outlier_z: Optional[float] = None, schedule: Optional[LRSchedule] = None):
        self.table = TensorTable(table_entries)
        self.schedule = schedule
        self.n = self.table.total
        self.hyper = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay)
        self.clip = clip
        self.hyper_struct = MpHyper(lr, beta1, beta2, eps, weight_decay, clip)
        dev = torch.device("cuda") if device is None else torch.device(device)
        nbytes = mp_grad_norm_workspace_bytes(self.n)
        self.workspace = torch.empty(max(8, nbytes), dtype=torch.uint8, device=dev)
        self.d_norm = torch.zeros(1, dtype=torch.float32, device=dev)
        self.d_scale = torch.zeros(1, dtype=torch.float32, device=dev)
        self.d_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.outlier = OutlierDetector(outlier_z, device=dev) if outlier_z is not None else None
        self.d_state = None  # device step state of replayable steps (init_device_clock)
        self.d_bias = None

    def step(self, params, grads, master, m, v, t: int, seed: int, host_grads=None, host_norm=None, stream=None):
        """One native call (mp_optimizer_step). With host_grads (pinned CPU
        bf16), `grads` is the device buffer that receives them. With a
        schedule, step t uses the schedule's learning rate for t."""
        if self.schedule is not None:
            self.hyper_struct.lr = self.schedule.lr(t)
        mp_optimizer_step(params, grads, master, m, v, self.table, self.hyper_struct, t=t, seed=seed,
                          workspace=self.workspace, d_norm=self.d_norm, d_scale=self.d_scale,
                          d_status=self.d_status,
                          outlier_state=self.outlier.state if self.outlier is not None else None,
                          outlier_z=self.outlier.z_threshold if self.outlier is not None else 0.0,
                          d_z=self.outlier.d_z if self.outlier is not None else None,
                          host_grads=host_grads, host_norm=host_norm, n=self.n, stream=stream)

    # --- replayable steps: the step count lives on the device -------------
    def init_device_clock(self, t: int = 0, seed_base: int = 0, lr: Optional[float] = None, stream=None):
        """Creates the device step state (t = steps already taken, step t
        rounds with seed seed_base + t) and the bias-correction table for
        this optimizer's betas; step_graph() then needs no per-step host
        arguments. Call again to reset or resume."""
        st = MpStepState(int(t), int(seed_base) & 0xFFFFFFFF, float(self.hyper["lr"] if lr is None else lr),
                         0, 0, 0.0, 0.0, 0)
        raw = torch.frombuffer(bytearray(ctypes.string_at(ctypes.addressof(st), ctypes.sizeof(st))),
                               dtype=torch.int32)
        dev = self.d_norm.device
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            if self.d_state is None:
                self.d_state = torch.empty(8, dtype=torch.int32, device=dev)
                self.d_bias = mp_bias_table(self.hyper["beta1"], self.hyper["beta2"]).to(dev)
            self.d_state.copy_(raw)

    def _need_clock(self):
        if self.d_state is None:
            raise RuntimeError("call init_device_clock() before the replayable-step methods")

    def set_lr(self, lr: float, stream=None):
        """Stream-ordered write of the next steps' learning rate into the
        device step state (between replays of a captured step)."""
        self._need_clock()
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            self.d_state[2:3].view(torch.float32).fill_(float(lr))

    def device_clock(self) -> dict:
        """The device step state (synchronises): t, seed_base, lr, and the
        seed and bias corrections of the last step taken."""
        self._need_clock()
        raw = self.d_state.cpu().numpy().tobytes()
        st = MpStepState.from_buffer_copy(raw)
        return dict(t=st.t, seed_base=st.seed_base, lr=st.lr, seed=st.seed, bc1=st.bc1, bc2=st.bc2)

    def step_graph(self, params, grads, master, m, v, host_grads=None, host_norm=None, stream=None):
        """One mp_optimizer_step_graph call: the next step of the device
        clock. Capturable: record it once in a CUDA graph and replay it."""
        self._need_clock()
        mp_optimizer_step_graph(params, grads, master, m, v, self.table, self.hyper_struct, d_state=self.d_state,
                                d_bias=self.d_bias, workspace=self.workspace, d_norm=self.d_norm,
                                d_scale=self.d_scale, d_status=self.d_status,
                                outlier_state=self.outlier.state if self.outlier is not None else None,
                                outlier_z=self.outlier.z_threshold if self.outlier is not None else 0.0,
                                d_z=self.outlier.d_z if self.outlier is not None else None,
                                host_grads=host_grads, host_norm=host_norm, n=self.n, stream=stream)

    def take_status(self) -> int:
        """Device status of the steps since the last call (0, MP_ERR_NONFINITE
        or MP_SKIPPED_OUTLIER; the first one recorded wins); clears it."""
        st = int(self.d_status.item())
        if st != MP_OK:
            self.d_status.zero_()
        return st

    def check_status(self) -> None:
        st = self.take_status()
        if st != MP_OK:
            raise MpError(st, "mp_adamw_step (device)")


class HostGradPipeline:
    """Optimizer steps whose gradients arrive in page-locked host memory,
    with each step's host-to-device copy overlapped with the previous step's
    update.

    Two device gradient buffers alternate: step t's copy (on its own stream)
    fills buffer t % 2 while the compute stream still runs step t - 1 on the
    other one; the step waits for its copy (an event), and a copy waits for
    the step that last read its buffer. transfer="kernel" (the default) copies
    with mp_copy_from_host (one block per SM, beside the update kernel);
    transfer="engine" with a copy engine (cudaMemcpyAsync). Every step is one
    Optimizer.step call (mp_optimizer_step) on the compute stream; the norm
    can be copied back to a page-locked host float each step. Nothing here
    synchronises the host, so a host buffer passed to step() must not be
    rewritten before its copy has run: wait on last_copy() (an event) first.
    Below SMALL_N parameters a copy takes less time than this bookkeeping, so
    each step is instead one Optimizer.step call whose norm kernel reads the
    host gradients itself (the same results).
    """

    SMALL_N = 1 << 20

    def __init__(self, opt: "Optimizer", device=None, transfer: str = "kernel"):
        if transfer not in ("kernel", "engine"):
            raise ValueError("transfer: 'kernel' or 'engine'")
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.opt = opt
        self.transfer = transfer
        self.buffers = [torch.empty(opt.n, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(dev)
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.used = [torch.cuda.Event() for _ in range(2)]  # after the last step that read each buffer
        self.k = 0
        self.small = opt.n <= self.SMALL_N

    def step(self, params, host_grads: torch.Tensor, master, m, v, t: int, seed: int, host_norm=None,
             stream=None):
        if host_grads.is_cuda or not host_grads.is_pinned():
            raise ValueError("host_grads: page-locked host memory expected")
        if host_grads.dtype not in _BF16_LIKE or host_grads.numel() != self.opt.n or not host_grads.is_contiguous():
            raise ValueError(f"host_grads: {self.opt.n} contiguous bf16 values expected")
        compute = stream if stream is not None else torch.cuda.current_stream(self.buffers[0].device)
        b = self.k % 2
        self.k += 1
        buf = self.buffers[b]
        if self.small:
            self.opt.step(params, buf, master, m, v, t, seed, host_grads=host_grads, host_norm=host_norm,
                          stream=compute)
            self.copied[b].record(compute)
            return
        with torch.cuda.stream(self.copy_stream):
            if self.k > 2:  # the buffer's previous reader, two steps back
                self.copy_stream.wait_event(self.used[b])
            if self.transfer == "kernel":
                mp_copy_from_host(buf, host_grads, stream=self.copy_stream)
            else:
                buf.copy_(host_grads.view(buf.dtype), non_blocking=True)
            self.copied[b].record(self.copy_stream)
        compute.wait_event(self.copied[b])
        self.opt.step(params, buf, master, m, v, t, seed, stream=compute)
        if host_norm is not None:
            with torch.cuda.stream(compute):
                host_norm.copy_(self.opt.d_norm, non_blocking=True)
        self.used[b].record(compute)

    def last_copy(self) -> torch.cuda.Event:
        """The event recorded after the latest step's host-to-device copy: once
        it has completed (.synchronize() or .query()), that host buffer may be
        rewritten."""
        return self.copied[(self.k - 1) % 2]


__all__ = [
    "MpError", "MpTensor", "MpHyper", "TensorTable", "Optimizer", "OutlierDetector", "lib", "abi_version",
    "status_string", "last_cuda_error", "mp_grad_norm_workspace_bytes", "mp_grad_norm", "mp_grad_norm_noalloc",
    "mp_adamw_step", "mp_optimizer_step", "mp_outlier_state_bytes", "mp_outlier_reset", "mp_outlier_check",
    "mp_stochastic_round", "mp_stochastic_round_fp16", "mp_accumulate_sr", "mp_noise_u32", "mp_bias_table_len", "mp_bias_table", "mp_optimizer_step_graph",
    "MpStepState", "MpLaunch", "mp_step_launches", "LIB_PATH", "mp_grad_sumsq", "mp_clip_scale_from_sumsq",
    "LRSchedule", "MpLrSchedule", "LR_KINDS", "HostGradPipeline", "mp_copy_from_host",
]
