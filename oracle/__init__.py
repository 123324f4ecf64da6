"""ctypes wrapper of the CPU oracle (mp_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and
by bench.py's CPU-baseline leg, never by the product package. Arrays are
numpy arrays; bf16 values are their raw uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_c_u16p = ctypes.POINTER(ctypes.c_uint16)
_c_u32p = ctypes.POINTER(ctypes.c_uint32)
_c_f32p = ctypes.POINTER(ctypes.c_float)
_c_f64p = ctypes.POINTER(ctypes.c_double)


class OracleTensor(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_uint64), ("size", ctypes.c_uint64),
                ("decay", ctypes.c_int32), ("pad", ctypes.c_int32)]


OUTLIER_WINDOW = 128


class OracleOutlier(ctypes.Structure):
    _fields_ = [("window", ctypes.c_double * OUTLIER_WINDOW), ("count", ctypes.c_uint64)]


_lib = None


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle build from `path` with its function signatures set."""
    L = ctypes.CDLL(path)
    L.oracle_noise_u32.restype = ctypes.c_uint32
    L.oracle_noise_u32.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
    L.oracle_noise_fill.restype = None
    L.oracle_noise_fill.argtypes = [_c_u32p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
    L.oracle_sr_with_rand.restype = ctypes.c_uint16
    L.oracle_sr_with_rand.argtypes = [ctypes.c_float, ctypes.c_uint32]
    L.oracle_sr.restype = ctypes.c_uint16
    L.oracle_sr.argtypes = [ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32]
    L.oracle_stochastic_round.restype = None
    L.oracle_stochastic_round.argtypes = [_c_u16p, _c_f32p, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_uint32]
    L.oracle_sr_fp16_with_rand.restype = ctypes.c_uint16
    L.oracle_sr_fp16_with_rand.argtypes = [ctypes.c_float, ctypes.c_uint32]
    L.oracle_stochastic_round_fp16.restype = None
    L.oracle_stochastic_round_fp16.argtypes = [_c_u16p, _c_f32p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
    L.oracle_accumulate_sr.restype = None
    L.oracle_accumulate_sr.argtypes = [_c_u16p, _c_f32p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
    L.oracle_sumsq.restype = ctypes.c_double
    L.oracle_sumsq.argtypes = [_c_u16p, ctypes.c_uint64]
    L.oracle_sumsq_from.restype = ctypes.c_double
    L.oracle_sumsq_from.argtypes = [ctypes.c_double, _c_u16p, ctypes.c_uint64]
    L.oracle_norm_from_parts.restype = None
    L.oracle_norm_from_parts.argtypes = [_c_f64p, ctypes.c_int32, ctypes.c_float, _c_f64p, _c_f32p, _c_f32p]
    L.oracle_lr.restype = ctypes.c_float
    L.oracle_lr.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                            ctypes.c_float, ctypes.c_int64]
    L.oracle_clip_scale.restype = ctypes.c_float
    L.oracle_clip_scale.argtypes = [ctypes.c_float, ctypes.c_float]
    L.oracle_grad_norm.restype = None
    L.oracle_grad_norm.argtypes = [_c_u16p, ctypes.c_uint64, ctypes.c_float,
                                   _c_f64p, _c_f32p, _c_f32p]
    L.oracle_bias_corrections.restype = None
    L.oracle_bias_corrections.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int32,
                                          _c_f32p, _c_f32p]
    L.oracle_adamw_step.restype = ctypes.c_int
    L.oracle_adamw_step.argtypes = [
        _c_u16p, _c_u16p, _c_f32p, _c_f32p, _c_f32p,
        ctypes.c_uint64, ctypes.c_uint64,
        ctypes.POINTER(OracleTensor), ctypes.c_int32,
        ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
        ctypes.c_float, ctypes.c_float, ctypes.c_int32, ctypes.c_uint32]
    L.oracle_outlier_check.restype = ctypes.c_int
    L.oracle_outlier_check.argtypes = [ctypes.POINTER(OracleOutlier), ctypes.c_float, ctypes.c_float,
                                       _c_f32p, _c_f64p]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def _ptr(a, ctype, dtype):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.dtype == dtype and a.flags["C_CONTIGUOUS"], \
        f"expected a C-contiguous {dtype} array"
    return a.ctypes.data_as(ctype)


def noise_u32(k: int, seed: int) -> int:
    return int(lib().oracle_noise_u32(k, seed))


def noise_fill(first: int, n: int, seed: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    lib().oracle_noise_fill(_ptr(out, _c_u32p, np.uint32), first, n, seed)
    return out


def sr_with_rand(x: float, rand16: int) -> int:
    return int(lib().oracle_sr_with_rand(x, rand16))


def sr(x: float, k: int, seed: int) -> int:
    return int(lib().oracle_sr(x, k, seed))


def stochastic_round(x: np.ndarray, global_offset: int, seed: int) -> np.ndarray:
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_stochastic_round(_ptr(out, _c_u16p, np.uint16), _ptr(x, _c_f32p, np.float32),
                                  global_offset, x.size, seed)
    return out


def sr_fp16_with_rand(x: float, rand16: int) -> int:
    return int(lib().oracle_sr_fp16_with_rand(x, rand16))


def stochastic_round_fp16(x: np.ndarray, global_offset: int, seed: int) -> np.ndarray:
    """fp16 patterns (uint16) of the stochastic rounding of fp32 x."""
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_stochastic_round_fp16(_ptr(out, _c_u16p, np.uint16), _ptr(x, _c_f32p, np.float32),
                                       global_offset, x.size, seed)
    return out


def accumulate_sr(acc: np.ndarray, delta: np.ndarray, global_offset: int, seed: int) -> None:
    """In place: acc[i] = SR((float)acc[i] + delta[i], global_offset + i, seed)
    (acc holds raw bf16 patterns as uint16)."""
    assert acc.size == delta.size
    lib().oracle_accumulate_sr(_ptr(acc, _c_u16p, np.uint16), _ptr(delta, _c_f32p, np.float32),
                               global_offset, acc.size, seed)


def sumsq(grads: np.ndarray) -> float:
    return float(lib().oracle_sumsq(_ptr(grads, _c_u16p, np.uint16), grads.size))


def sumsq_from(s: float, grads: np.ndarray) -> float:
    """s plus the squares of grads added one by one in index order."""
    return float(lib().oracle_sumsq_from(s, _ptr(grads, _c_u16p, np.uint16), grads.size))


def norm_from_parts(parts, clip: float):
    """ZeRO-1 norm from per-rank sums of squares added in rank order.
    Returns (sumsq: float64, norm: float32, scale: float32)."""
    arr = np.ascontiguousarray(parts, dtype=np.float64)
    s = ctypes.c_double()
    nrm = ctypes.c_float()
    sc = ctypes.c_float()
    lib().oracle_norm_from_parts(_ptr(arr, _c_f64p, np.float64), arr.size, clip, ctypes.byref(s),
                                 ctypes.byref(nrm), ctypes.byref(sc))
    return s.value, np.float32(nrm.value), np.float32(sc.value)


LR_CONSTANT, LR_COSINE, LR_LINEAR, LR_WSD = 0, 1, 2, 3


def lr(kind: int, warmup: int, total: int, lr_max: float, lr_min: float, decay_frac: float, t: int) -> np.float32:
    """Learning rate of the 1-based step t (NaN for invalid arguments)."""
    return np.float32(lib().oracle_lr(kind, warmup, total, lr_max, lr_min, decay_frac, t))


def clip_scale(norm: float, clip: float) -> float:
    return float(lib().oracle_clip_scale(norm, clip))


def grad_norm(grads: np.ndarray, clip: float):
    """Returns (sumsq: float64, norm: float32, scale: float32)."""
    s = ctypes.c_double()
    nrm = ctypes.c_float()
    sc = ctypes.c_float()
    lib().oracle_grad_norm(_ptr(grads, _c_u16p, np.uint16), grads.size, clip,
                           ctypes.byref(s), ctypes.byref(nrm), ctypes.byref(sc))
    return s.value, np.float32(nrm.value), np.float32(sc.value)


def bias_corrections(beta1: float, beta2: float, t: int):
    b1 = ctypes.c_float()
    b2 = ctypes.c_float()
    lib().oracle_bias_corrections(beta1, beta2, t, ctypes.byref(b1), ctypes.byref(b2))
    return np.float32(b1.value), np.float32(b2.value)


def make_table(entries):
    """entries: iterable of (offset, size, decay)."""
    entries = list(entries)
    arr = (OracleTensor * max(1, len(entries)))()
    for i, (off, size, decay) in enumerate(entries):
        arr[i].offset, arr[i].size, arr[i].decay, arr[i].pad = off, size, int(decay), 0
    return arr, len(entries)


def adamw_step(params, grads, master, m, v, global_offset, table_entries,
               lr, beta1, beta2, eps, weight_decay, scale, t, seed) -> int:
    """In-place step on numpy arrays (params/grads uint16, master/m/v float32).
    master=None selects the no-master variant. Returns the oracle status."""
    tab, nt = make_table(table_entries)
    n = m.size
    for a, dt in ((params, np.uint16), (grads, np.uint16), (m, np.float32), (v, np.float32)):
        assert a.size == n and a.dtype == dt
    if master is not None:
        assert master.size == n and master.dtype == np.float32
    return int(lib().oracle_adamw_step(
        _ptr(params, _c_u16p, np.uint16), _ptr(grads, _c_u16p, np.uint16),
        _ptr(master, _c_f32p, np.float32), _ptr(m, _c_f32p, np.float32),
        _ptr(v, _c_f32p, np.float32), global_offset, n, tab, nt,
        lr, beta1, beta2, eps, weight_decay, scale, t, seed))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 patterns (test-side convenience)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


class OutlierCheck:
    """Stateful wrapper of oracle_outlier_check (window of 128 finite norms)."""

    def __init__(self):
        self.state = OracleOutlier()

    def check(self, norm: float, z_threshold: float, scale: float):
        """Returns (status, z, scale_after)."""
        sc = ctypes.c_float(scale)
        z = ctypes.c_double()
        st = lib().oracle_outlier_check(ctypes.byref(self.state), norm, z_threshold, ctypes.byref(sc),
                                        ctypes.byref(z))
        return int(st), z.value, sc.value
