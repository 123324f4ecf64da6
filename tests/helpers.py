"""Shared test utilities: host copies of device tensors and the parity bars.

Tolerances (against the CPU oracle, on identical inputs):
  fp32 master / m / v    max relative error <= 1e-6
  grad norm              relative error <= 1e-6 against the fp64 sum;
                         bit-identical across GPU runs
  stochastic rounding    bit-exact
  bf16 params            <= 1e-6 of elements differ, by at most 1 bf16 ulp
The kernels follow the same fp32 operation order as the oracle, so the step
is expected to be bit-exact as well; tests check both.
"""
import numpy as np
import torch


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bits32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_f32_close(gpu: np.ndarray, ref: np.ndarray, name: str, rtol: float = 1e-6):
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    assert gpu.shape == ref.shape
    same_nan = np.isnan(gpu) == np.isnan(ref)
    assert same_nan.all(), f"{name}: NaN positions differ"
    fin = ~np.isnan(ref)
    err = np.abs(gpu[fin].astype(np.float64) - ref[fin].astype(np.float64))
    bound = rtol * np.abs(ref[fin].astype(np.float64))
    bad = err > bound
    assert not bad.any(), (f"{name}: {int(bad.sum())} elements beyond rel {rtol}; "
                           f"worst rel {float((err / np.maximum(bound / rtol, 1e-45)).max()):.3e}")


def assert_bf16_close(gpu: np.ndarray, ref: np.ndarray, name: str, max_frac: float = 1e-6):
    gpu = np.asarray(gpu, np.uint16).astype(np.int64)
    ref = np.asarray(ref, np.uint16).astype(np.int64)
    diff = gpu != ref
    frac = float(diff.mean()) if diff.size else 0.0
    allowed = int(np.floor(max_frac * diff.size))
    assert int(diff.sum()) <= allowed, f"{name}: {int(diff.sum())} of {diff.size} bf16 values differ (frac {frac:.2e})"
    if diff.any():
        # same sign, adjacent patterns = one bf16 ulp apart
        assert np.all(((gpu[diff] ^ ref[diff]) & 0x8000) == 0), f"{name}: sign differs"
        assert np.all(np.abs(gpu[diff] - ref[diff]) <= 1), f"{name}: differs by more than 1 ulp"


def assert_bit_equal(gpu: np.ndarray, ref: np.ndarray, name: str):
    if gpu.dtype == np.float32:
        gpu, ref = bits32(gpu), bits32(ref)
    neq = gpu != ref
    assert not neq.any(), f"{name}: {int(neq.sum())} of {neq.size} elements differ bitwise (first at {int(np.argmax(neq))})"


def rel_err(a: float, b: float) -> float:
    return abs(a - b) / abs(b) if b != 0 else abs(a - b)


def assert_f32_bits_or_both_nan(gpu: np.ndarray, ref: np.ndarray, name: str):
    """Bit equality, except that NaNs need only sit at the same positions:
    arithmetic NaNs carry different payloads on the GPU and on host CPUs."""
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    gn, rn = np.isnan(gpu), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{name}: NaN positions differ ({int(gn.sum())} vs {int(rn.sum())})"
    ok = ~gn
    neq = bits32(gpu[ok]) != bits32(ref[ok])
    assert not neq.any(), f"{name}: {int(neq.sum())} non-NaN elements differ bitwise"
