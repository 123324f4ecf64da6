"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every test runs the library's kernels on a GB300 and compares element by
element with the oracle on the same seeded inputs, at the bars listed in
tests/helpers.py. Sizes span several 2048-element tiles plus ragged tails;
full-size parameter sets are checked in full (GPT-2 124M) or on windows the
oracle recomputes with their global offsets (GPT-2 1.5B, Llama-3-8B).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_bf16_close, assert_bit_equal, assert_f32_close, rel_err, to_np_f32,
                     to_np_u16)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import __graft_entry__
    __graft_entry__.build()  # no-op when the library is up to date
    import mixed_precision_adamw_gb300 as mp
else:  # collected on CPU machines, skipped below
    mp = None

DEV = "cuda"


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def f32(x):
    return float(np.float32(x))


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    return W.bf16_bits(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16))


def dev_u16(a: np.ndarray, pad: int = 0) -> torch.Tensor:
    """Device bf16 tensor holding raw patterns a, optionally starting `pad`
    elements into a larger buffer (pad odd -> only 2-B aligned)."""
    buf = torch.empty(a.size + pad, dtype=torch.int16, device=DEV)
    out = buf[pad:]
    out.copy_(torch.from_numpy(a.view(np.int16)))
    return out.view(torch.bfloat16)


def dev_f32(a: np.ndarray, pad: int = 0) -> torch.Tensor:
    buf = torch.empty(a.size + pad, dtype=torch.float32, device=DEV)
    out = buf[pad:]
    out.copy_(torch.from_numpy(np.ascontiguousarray(a, np.float32)))
    return out


# ---------------------------------------------------------------------------
# rounding randomness and stochastic rounding: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("first,seed,n", [(0, 0, 1 << 20), (123456789, 42, 1000003),
                                          ((1 << 32) - 5000, 7, 10000), ((5 << 32) + 3, 2024, 77777)])
def test_noise_bit_exact(first, seed, n):
    out = torch.empty(n, dtype=torch.int32, device=DEV)
    mp.mp_noise_u32(out, first, seed)
    got = out.cpu().numpy().view(np.uint32)
    assert_bit_equal(got, oracle.noise_fill(first, n, seed), "noise")


def _special_f32(n, rng):
    with np.errstate(over="ignore"):  # magnitudes past the fp32 range become +-Inf on purpose
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-45, 38, n)).astype(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, np.finfo(np.float32).max,
                         -np.finfo(np.float32).max, 1e-45, -1e-45, 1.17549435e-38, 257.0, 1.0 + 2 ** -8],
                        np.float32)
    x[: specials.size] = specials
    # NaNs with low payload bits only, and bf16-representable values
    x[specials.size:specials.size + 4] = np.array([0x7F800001, 0xFF800003, 0x7FC00000, 0x7F80FFFF],
                                                  np.uint32).view(np.float32)
    x[-1000:] = (x[-1000:].view(np.uint32) & 0xFFFF0000).view(np.float32)
    return x


@pytest.mark.parametrize("n,pad_in,pad_out,goff", [
    (2048 * 7 + 5, 0, 0, 0), (2048 * 7 + 5, 1, 0, 17), (2048 * 7 + 5, 0, 1, 1 << 32),
    (1, 0, 0, 5), (2047, 0, 0, 0), (300001, 3, 2, (1 << 32) - 150000),
    # vector path crossing 2^32 inside a 4-element group (offset not a multiple of 4)
    (2048 * 7 + 5, 0, 0, (1 << 32) - 5001), (2048 * 7 + 5, 0, 0, (1 << 32) - 5002),
    (2048 * 7 + 5, 0, 0, (1 << 32) - 5003), (2048 * 7 + 5, 0, 0, (3 << 32) - 1),
    # longer aligned ranges, with a ragged tail, across 2^32, and an 8-B aligned output
    (1_249_283, 0, 0, (1 << 32) - 600_001), ((1 << 22) + 3, 0, 0, 123), ((1 << 22) + 3, 0, 4, 99)])
def test_stochastic_round_bit_exact(n, pad_in, pad_out, goff):
    rng = np.random.default_rng(n + pad_in)
    x = _special_f32(n, rng) if n > 2000 else rng.standard_normal(n).astype(np.float32)
    xin = dev_f32(x, pad_in)
    out = dev_u16(np.zeros(n, np.uint16), pad_out)
    seed = 0xC0FFEE
    mp.mp_stochastic_round(out, xin, seed, global_offset=goff)
    assert_bit_equal(to_np_u16(out), oracle.stochastic_round(x, goff, seed), "sr")


def _long_round_n(tile, tiles_per_sm, extra):
    """A length just past the TMA-staged rounding kernels' minimum (tiles per
    SM of `tile` elements), with a ragged tail."""
    return tiles_per_sm * torch.cuda.get_device_properties(0).multi_processor_count * tile + extra


def _long_f32(n, rng):
    """Weight-like and wide-range values with the special values sprinkled in."""
    x = rng.standard_normal(n, dtype=np.float32)
    x[: n // 2] *= np.float32(0.02)
    with np.errstate(over="ignore"):
        x[n // 2:] *= np.exp2(rng.integers(-140, 127, n - n // 2)).astype(np.float32)
    sp = _special_f32(4096, rng)
    idx = rng.integers(0, n, sp.size)
    x[idx] = sp
    return x


@pytest.mark.parametrize("goff", [0, (1 << 32) - 60_000_001])
def test_stochastic_round_long_range_tma_bit_exact(goff):
    """A range long enough for the TMA-staged bf16 rounding kernel (128 tiles
    of 6,144 elements per SM, plus a ragged tail), across index 2^32 in one
    case: every element bit-exact against the oracle."""
    n = _long_round_n(6144, 128, 12_345)
    rng = np.random.default_rng(77)
    x = _long_f32(n, rng)
    out = torch.empty(n, dtype=torch.int16, device=DEV)
    mp.mp_stochastic_round(out, dev_f32(x), 0xB16, global_offset=goff)
    assert_bit_equal(to_np_u16(out), oracle.stochastic_round(x, goff, 0xB16), "sr long range")


@pytest.mark.parametrize("goff", [0, (1 << 32) - 25_000_003])
def test_accumulate_sr_long_range_tma_bit_exact(goff):
    """A range long enough for the TMA-staged accumulate-and-round kernel (80
    tiles of 4,096 elements per SM, plus a ragged tail), across index 2^32 in
    one case: every accumulator bit-exact against the oracle."""
    n = _long_round_n(4096, 80, 777)
    rng = np.random.default_rng(78)
    acc0 = bf16_from_f32(rng.standard_normal(n, dtype=np.float32) * np.float32(0.02))
    acc0[rng.integers(0, n, 8)] = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x7F7F, 0xFF7F, 0x0001],
                                           np.uint16)
    delta = _long_f32(n, rng)
    acc = dev_u16(acc0)
    mp.mp_accumulate_sr(acc, dev_f32(delta), 0xACC2, global_offset=goff)
    ref = acc0.copy()
    oracle.accumulate_sr(ref, delta, goff, 0xACC2)
    assert_bit_equal(to_np_u16(acc), ref, "accumulate_sr long range")


@pytest.mark.parametrize("n,pad_acc,pad_delta,goff", [
    (2048 * 7 + 5, 0, 0, 0), (2048 * 7 + 5, 1, 0, 17), (2048 * 7 + 5, 0, 1, 1 << 32), (1, 0, 0, 5),
    (2047, 0, 0, 0), (300001, 3, 2, (1 << 32) - 150000), (2048 * 7 + 5, 0, 0, (1 << 32) - 5001),
    (2048 * 7 + 5, 0, 0, (1 << 32) - 5003), ((1 << 22) + 3, 0, 0, 123), (1_249_283, 0, 0, (1 << 32) - 600_001)])
def test_accumulate_sr_bit_exact(n, pad_acc, pad_delta, goff):
    """acc = SR((float)acc + delta): special values on both sides (NaN, Inf,
    signed zeros, subnormals, the largest finite values), vector and scalar
    paths, offsets across 2^32."""
    rng = np.random.default_rng(n + 7 * pad_acc)
    acc0 = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
    acc0[:8] = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x7F7F, 0xFF7F, 0x0001], np.uint16)[: min(8, n)]
    delta = _special_f32(n, rng) if n > 2000 else rng.standard_normal(n).astype(np.float32)
    if n > 2000:
        # ordinary magnitudes too: contributions around the accumulator's own scale
        k = n // 2
        with np.errstate(invalid="ignore", over="ignore"):  # NaN and Inf accumulators give NaN/Inf deltas
            delta[k:] = (oracle.bf16_bits_to_f32(acc0[k:]) * rng.uniform(-1e-2, 1e-2, n - k)).astype(np.float32)
    acc = dev_u16(acc0, pad_acc)
    d = dev_f32(delta, pad_delta)
    seed = 0xACC
    mp.mp_accumulate_sr(acc, d, seed, global_offset=goff)
    ref = acc0.copy()
    oracle.accumulate_sr(ref, delta, goff, seed)
    assert_bit_equal(to_np_u16(acc), ref, "accumulate_sr")


def _fp16_cases(n, rng):
    """fp32 inputs for the fp16 rounding: the specials of the bf16 tests, the
    fp16 boundaries (subnormal/normal at 2^-14, the largest finite 65504, the
    overflow edge 65536, fp16's smallest subnormal 2^-24 and below), values
    just off every fp16 exponent, and magnitudes spread over fp16's range."""
    x = _special_f32(n, rng)
    with np.errstate(over="ignore"):
        x[n // 4: n // 2] = (rng.standard_normal(n // 2 - n // 4) *
                             2.0 ** rng.uniform(-30, 17, n // 2 - n // 4)).astype(np.float32)
    edges = [2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -26, 65504.0, 65519.99, 65520.0, 65535.99, 65536.0,
             65537.0, 1e5, 6.1e-5, 5.96e-8, 3e-8, 1.0, 0.5, 1024.0 + 0.5, 2048.0 + 1.0]
    edges += [2.0 ** e for e in range(-24, 16)]
    e = np.array(edges, np.float32)
    near = np.concatenate([e, np.nextafter(e, np.float32(0)), np.nextafter(e, np.float32(np.inf))])
    near = np.concatenate([near, -near])
    x[16:16 + near.size] = near
    return x


@pytest.mark.parametrize("n,pad_in,pad_out,goff", [
    (2048 * 7 + 5, 0, 0, 0), (2048 * 7 + 5, 1, 0, 17), (2048 * 7 + 5, 0, 1, 1 << 32),
    (1, 0, 0, 5), (2047, 0, 0, 0), (300001, 3, 2, (1 << 32) - 150000),
    (2048 * 7 + 5, 0, 0, (1 << 32) - 5001), (2048 * 7 + 5, 0, 0, (1 << 32) - 5003),
    ((1 << 22) + 3, 0, 0, 123), (1_249_283, 0, 0, (1 << 32) - 600_001)])
def test_stochastic_round_fp16_bit_exact(n, pad_in, pad_out, goff):
    """fp32 -> fp16 stochastic rounding, bit-exact against the oracle: fp16
    subnormals, the subnormal/normal boundary, 65504 .. 65536 and beyond,
    NaN, Inf, signed zeros; vector and scalar paths; offsets across 2^32."""
    rng = np.random.default_rng(3 * n + pad_out)
    x = _fp16_cases(n, rng) if n > 2000 else rng.standard_normal(n).astype(np.float32)
    xin = dev_f32(x, pad_in)
    buf = torch.zeros(n + pad_out, dtype=torch.float16, device=DEV)
    out = buf[pad_out:]
    seed = 0xF16
    mp.mp_stochastic_round_fp16(out, xin, seed, global_offset=goff)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_bit_equal(got, oracle.stochastic_round_fp16(x, goff, seed), "sr fp16")


@pytest.mark.parametrize("n", [2048 * 300 + 777, 2048 * 700 + 777])
@pytest.mark.parametrize("goff", [0, (1 << 32) - 3001])
def test_stochastic_round_fp16_weights_and_scattered_specials(goff, n):
    """Weight-like values (N(0, 0.02), all in fp16's normal range) over many
    tiles and a ragged tail, then the same with one zero, subnormal, NaN or
    overflow scattered into some warps' elements: every warp shape of the
    vector kernel (all normal, some special) is bit-exact against the oracle."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(n) * 0.02).astype(np.float32)
    x = np.where(np.abs(x) < 2.0 ** -13, np.float32(0.5), x).astype(np.float32)
    for special_every in (None, 9973):
        if special_every is not None:
            idx = np.arange(17, n, special_every)
            x[idx] = np.resize(np.array([0.0, -1e-6, np.nan, -7e4, 3e-9, np.inf, 65519.99], np.float32), idx.size)
        out = torch.empty(n, dtype=torch.float16, device=DEV)
        mp.mp_stochastic_round_fp16(out, dev_f32(x), 0x5EED, global_offset=goff)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert_bit_equal(got, oracle.stochastic_round_fp16(x, goff, 0x5EED), f"sr fp16 specials {special_every}")


def test_stochastic_round_fp16_every_pattern_and_unbiased():
    """Every finite fp16 pattern round-trips unchanged; values between two
    fp16 neighbours land on one of them and average to the input over many
    seeds (float64 mean over 4096 draws per value)."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = h.view(np.float16)
    keep = np.isfinite(vals)
    x = vals[keep].astype(np.float32)
    out = torch.empty(x.size, dtype=torch.float16, device=DEV)
    mp.mp_stochastic_round_fp16(out, dev_f32(x), 99)
    assert_bit_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), h[keep], "fp16 round trip")

    rng = np.random.default_rng(5)
    lo = np.concatenate([np.arange(1, 1023, 37), np.arange(0x3C00, 0x3C40), np.arange(0x7B80, 0x7BFF, 7)])
    lo = lo.astype(np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).view(np.float16).astype(np.float64)
    t = rng.uniform(0.05, 0.95, lo.size)
    x = (a + t * (b - a)).astype(np.float32)
    reps = 4096
    xs = torch.from_numpy(np.tile(x, reps)).to(DEV)
    out = torch.empty(xs.numel(), dtype=torch.float16, device=DEV)
    mp.mp_stochastic_round_fp16(out, xs, 1234)
    r = out.view(reps, lo.size)
    bits = r.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all((bits == lo) | (bits == lo + 1))
    mean = r.double().mean(0).cpu().numpy()
    p = (x.astype(np.float64) - a) / (b - a)
    tol = 5.0 * np.sqrt(p * (1 - p) / reps) * (b - a) + 1e-12
    assert np.all(np.abs(mean - x.astype(np.float64)) <= tol)


def test_stochastic_round_full_size_and_drift():
    """SR stress: 64M fp32 weights with |w| log-uniform in [1e-3, 1e1]; a
    constant update of 1e-4 |w| per step for 1000 steps. SR (bit-exact
    against the oracle on the same fp32 inputs) tracks the fp32 trajectory;
    round-to-nearest never moves."""
    n = 64 << 20
    w0 = W.sr_stress_weights(n, device=DEV)
    delta = (w0.abs() * f32(1e-4)).float()
    x = w0.clone()
    out = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    mp.mp_stochastic_round(out, x, W.step_seed(0))
    xs = to_np_f32(x)
    assert_bit_equal(to_np_u16(out), oracle.stochastic_round(xs, 0, W.step_seed(0)), "sr 64M")
    fp32 = w0.clone()
    sr = w0.to(torch.bfloat16)
    acc = w0.to(torch.bfloat16)  # the same trajectory through mp_accumulate_sr (one kernel per step)
    for t in range(1, 1001):
        fp32 += delta
        torch.add(sr.float(), delta, out=x)
        mp.mp_stochastic_round(sr, x, W.step_seed(t))
        mp.mp_accumulate_sr(acc, delta, W.step_seed(t))
        if t in (1, 500):
            idx = slice(12345678, 12345678 + (1 << 20))
            assert_bit_equal(to_np_u16(sr[idx]), oracle.stochastic_round(to_np_f32(x[idx]), 12345678,
                                                                         W.step_seed(t)), f"sr step {t}")
    assert torch.equal(acc.view(torch.int16), sr.view(torch.int16))
    rne = w0.to(torch.bfloat16).float()
    drift_sr = float((sr.float().double() / fp32.double() - 1.0).mean())
    drift_rne = float((rne.double() / fp32.double() - 1.0).mean())
    expect_rne = float(torch.where(w0 > 0, 1 / 1.1 - 1, 1 / 0.9 - 1).double().mean())
    print(f"\nSR stress, 64M weights, 1000 steps: mean relative drift of the bf16 weights from the fp32 "
          f"trajectory: stochastic rounding {drift_sr:+.3e}, round-to-nearest {drift_rne:+.3e}")
    assert abs(drift_rne - expect_rne) < 1e-3
    assert abs(drift_sr) < 1e-4, drift_sr


def test_stochastic_round_fp16_full_size_and_drift():
    """The SR-stress workload rounded to fp16: 64M fp32 weights, |w|
    log-uniform in [1e-3, 10] (all in fp16's normal range), bit-exact against
    the oracle in windows at both ends and in the middle; then a constant
    update of 1e-4 |w| per step (below half an fp16 step) for 1000 steps.
    fp16 stochastic rounding tracks the fp32 trajectory; round-to-nearest
    never moves."""
    n = 64 << 20
    w0 = W.sr_stress_weights(n, device=DEV)
    out = torch.empty(n, dtype=torch.float16, device=DEV)
    mp.mp_stochastic_round_fp16(out, w0, W.step_seed(0))
    got = out.view(torch.int16)
    for a in (0, n // 2 - 777, n - (1 << 20)):
        win = slice(a, a + (1 << 20))
        assert_bit_equal(got[win].cpu().numpy().view(np.uint16),
                         oracle.stochastic_round_fp16(to_np_f32(w0[win]), a, W.step_seed(0)), f"fp16 window {a}")
    delta = (w0.abs() * f32(1e-4)).float()
    fp32 = w0.clone()
    sr = w0.to(torch.float16)
    x = torch.empty_like(w0)
    for t in range(1, 1001):
        fp32 += delta
        torch.add(sr.float(), delta, out=x)
        mp.mp_stochastic_round_fp16(sr, x, W.step_seed(t))
    rne = w0.to(torch.float16).float()
    drift_sr = float((sr.float().double() / fp32.double() - 1.0).mean())
    drift_rne = float((rne.double() / fp32.double() - 1.0).mean())
    print(f"\nfp16 SR stress, 64M weights, 1000 steps: mean relative drift from the fp32 trajectory: "
          f"stochastic rounding {drift_sr:+.3e}, round-to-nearest {drift_rne:+.3e}")
    expect_rne = float(torch.where(w0 > 0, 1 / 1.1 - 1, 1 / 0.9 - 1).double().mean())
    assert abs(drift_rne - expect_rne) < 1e-3
    assert abs(drift_sr) < 1e-4, drift_sr


# ---------------------------------------------------------------------------
# gradient norm
# ---------------------------------------------------------------------------
def _norm_gpu(g: torch.Tensor, clip=1.0):
    n = g.numel()
    ws = torch.empty(max(8, mp.mp_grad_norm_workspace_bytes(n)), dtype=torch.uint8, device=DEV)
    d_norm = torch.empty(1, dtype=torch.float32, device=DEV)
    d_scale = torch.empty(1, dtype=torch.float32, device=DEV)
    d_sumsq = torch.empty(1, dtype=torch.float64, device=DEV)
    mp.mp_grad_norm(g, clip, ws, d_norm, d_scale, d_sumsq)
    return float(d_sumsq.item()), np.float32(d_norm.item()), np.float32(d_scale.item())


# 2,492,429 = 16,384 x 152 + 8 x 257 + 5: on 152 SMs, just past the length from
# which each norm block reads one contiguous run (the last runs empty), with
# a ragged tail; (1 << 24) + 3 with a pad of 3 takes the element-wise path.
@pytest.mark.parametrize("n,pad", [(0, 0), (1, 0), (7, 0), (8, 0), (2047, 1), (2048 * 5 + 3, 0),
                                   (1000003, 0), (1000003, 3), (2492429, 0), (2492429, 3), (1 << 24, 0),
                                   ((1 << 24) + 3, 3)])
def test_grad_norm_parity(n, pad):
    rng = np.random.default_rng(n)
    g = bf16_from_f32(rng.standard_normal(n) * 10.0 ** rng.uniform(-5, 1, n))
    s, nrm, sc = _norm_gpu(dev_u16(g, pad))
    s_o, nrm_o, sc_o = oracle.grad_norm(g, 1.0)
    if n == 0:
        assert s == 0.0 and nrm == 0 and sc == 1.0
        return
    assert rel_err(s, s_o) <= 1e-6
    assert rel_err(float(nrm), math.sqrt(s_o)) <= 1e-6
    assert sc == oracle.clip_scale(float(nrm), 1.0)  # the scale rule is exact given the norm
    # bit-identical on repeated runs
    for _ in range(3):
        assert _norm_gpu(dev_u16(g, pad)) == (s, nrm, sc)


@pytest.mark.parametrize("case", ["tiny", "huge", "mixed", "zeros", "subnormal"])
@pytest.mark.parametrize("n", [3 * 2048 * 152 + 11, 3 * (1 << 20) + 11])  # the interleaved and the staged norm
def test_grad_norm_extreme_ranges(case, n):
    rng = np.random.default_rng(5)
    if case == "tiny":
        x = rng.standard_normal(n) * 1e-30
    elif case == "huge":
        x = rng.standard_normal(n) * 1e25
    elif case == "mixed":
        x = rng.standard_normal(n) * 10.0 ** rng.uniform(-35, 30, n)
    elif case == "zeros":
        x = np.zeros(n)
    else:
        x = rng.standard_normal(n) * 1e-39
    g = bf16_from_f32(x)
    s, nrm, sc = _norm_gpu(dev_u16(g), clip=1.0)
    s_o, nrm_o, sc_o = oracle.grad_norm(g, 1.0)
    assert rel_err(s, s_o) <= 1e-6, (s, s_o)
    assert rel_err(float(nrm), float(nrm_o)) <= 1e-6
    assert sc == oracle.clip_scale(float(nrm), 1.0)


def test_grad_norm_nonfinite():
    g = bf16_from_f32(np.ones(100000))
    for bad in (0x7FC0, 0x7F80, 0xFF80):
        g2 = g.copy()
        g2[77777] = bad
        s, nrm, sc = _norm_gpu(dev_u16(g2))
        assert not math.isfinite(nrm) and math.isnan(sc)


# ---------------------------------------------------------------------------
# the AdamW + SR step
# ---------------------------------------------------------------------------
class State:
    def __init__(self, params, grads, master, m, v):
        self.params, self.grads, self.master, self.m, self.v = params, grads, master, m, v


def _host_state(st):
    return dict(params=W.bf16_bits(st["params"].cpu()).copy(), master=st["master"].cpu().numpy().copy()
                if "master" in st else None, m=st["m"].cpu().numpy().copy(), v=st["v"].cpu().numpy().copy())


def _compare(gpu_st, host, name, exact=True):
    assert_bf16_close(to_np_u16(gpu_st["params"]), host["params"], f"{name} params")
    for k in ("master", "m", "v"):
        if host.get(k) is not None:
            assert_f32_close(to_np_f32(gpu_st[k]), host[k], f"{name} {k}")
    if exact:
        assert_bit_equal(to_np_u16(gpu_st["params"]), host["params"], f"{name} params (bitwise)")
        for k in ("master", "m", "v"):
            if host.get(k) is not None:
                assert_bit_equal(to_np_f32(gpu_st[k]), host[k], f"{name} {k} (bitwise)")


def _run_steps(name, steps, with_master, device_state=None):
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    H = W.HYPER
    st = W.make_state(name, device="cpu", with_master=with_master)
    host = _host_state(st)
    dst = {k: t.to(DEV) for k, t in st.items()}
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])
    for t in range(1, steps + 1):
        g = W.make_grads(name, t)
        gb = W.bf16_bits(g).copy()
        dg = g.to(DEV)
        opt.step(dst["params"], dg, dst.get("master"), dst["m"], dst["v"], t, W.step_seed(t))
        s_o, nrm_o, sc_o = oracle.grad_norm(gb, H["clip"])
        st_o = oracle.adamw_step(host["params"], gb, host["master"], host["m"], host["v"], 0, tab, H["lr"],
                                 H["beta1"], H["beta2"], H["eps"], H["weight_decay"],
                                 float(opt.d_scale.item()), t, W.step_seed(t))
        assert st_o == 0
        opt.check_status()
        assert rel_err(float(opt.d_norm.item()), float(nrm_o)) <= 1e-6
        assert float(opt.d_scale.item()) == oracle.clip_scale(float(opt.d_norm.item()), H["clip"])
        _compare(dst, host, f"{name} step {t}")
    return dst, host


@pytest.mark.parametrize("with_master", [True, False])
def test_tiny_sixteen_steps(with_master):
    _run_steps("tiny", 16, with_master)


@pytest.mark.parametrize("with_master", [True, False])
def test_gpt2_124m_full_parity(with_master):
    _run_steps("gpt2_124m", 2, with_master)


def _random_case(n, seed, tmin=1, tmax=5000):
    gen = torch.Generator().manual_seed(seed)
    tab = W.random_table(n, gen, tmin, tmax)
    rng = np.random.default_rng(seed)
    master = (rng.standard_normal(n) * 0.05).astype(np.float32)
    params = bf16_from_f32(master)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.random(n) * 1e-6).astype(np.float32)
    grads = bf16_from_f32(rng.standard_normal(n) * 1e-2)
    return tab, params, grads, master, m, v


@pytest.mark.parametrize("n,pad,with_master,tmax", [
    (2048 * 9 + 1234, 0, True, 5000), (2048 * 9 + 1234, 0, False, 5000), (2048 * 9 + 1234, 1, True, 5000),
    (5, 0, True, 3), (2048, 0, True, 1), (2048 * 3 + 1, 2, False, 2), (700000, 0, True, 40),
    (1 << 20, 0, True, 1 << 20)])
def test_step_random_tables(n, pad, with_master, tmax):
    tab, params, grads, master, m, v = _random_case(n, n + pad, 1, tmax)
    lr, b1, b2, eps, wd, scale, t, seed = 3e-3, 0.9, 0.95, 1e-8, 0.1, 0.37, 7, 99
    d = dict(params=dev_u16(params, pad), grads=dev_u16(grads, pad), m=dev_f32(m, pad), v=dev_f32(v, pad),
             master=dev_f32(master, pad) if with_master else None)
    d_scale = torch.tensor([scale], dtype=torch.float32, device=DEV)
    mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=lr, beta1=b1,
                     beta2=b2, eps=eps, weight_decay=wd, d_grad_scale=d_scale, t=t, seed=seed)
    host = dict(params=params.copy(), master=master.copy() if with_master else None, m=m.copy(), v=v.copy())
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], 0, tab, lr, b1, b2, eps,
                             wd, f32(scale), t, seed) == 0
    _compare(d, host, f"random n={n}")


@pytest.mark.parametrize("with_master", [True, False])
def test_step_every_line_offset_of_the_vector_path(with_master):
    """Buffers that start 4k elements past a 128-B line (k = 0 .. 15): the
    vector kernel peels the elements before the gradients' next line one per
    thread and tiles the rest; every offset must give the oracle's bits."""
    n = 2048 * 5 + 77
    tab, params, grads, master, m, v = _random_case(n, 4242, 1, 300)
    lr, b1, b2, eps, wd, scale, t, seed = 2e-3, 0.9, 0.95, 1e-8, 0.1, 0.81, 3, 5
    host = dict(params=params.copy(), master=master.copy() if with_master else None, m=m.copy(), v=v.copy())
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], 0, tab, lr, b1, b2, eps,
                             wd, f32(scale), t, seed) == 0
    d_scale = torch.tensor([scale], dtype=torch.float32, device=DEV)
    for k in range(16):
        pad = 4 * k
        d = dict(params=dev_u16(params, pad), grads=dev_u16(grads, pad), m=dev_f32(m, pad), v=dev_f32(v, pad),
                 master=dev_f32(master, pad) if with_master else None)
        mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=lr,
                         beta1=b1, beta2=b2, eps=eps, weight_decay=wd, d_grad_scale=d_scale, t=t, seed=seed)
        _compare(d, host, f"line offset {pad} elements")


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("with_master", [True, False])
@pytest.mark.parametrize("extra,pad,tmax,goff", [(0, 0, 5000, 0), (2047, 4, 1 << 19, 0), (1, 60, 1200, 0),
                                                 (777, 20, 60_000, 0), (1001, 8, 900, (1 << 32) - 700_003)])
def test_step_tma_path(with_master, extra, pad, tmax, goff):
    """Ranges of at least two 2048-element tiles per SM whose tiles start
    16-B aligned in every array run the TMA-staged kernel (whole tiles loaded
    and stored by bulk copies, updated in shared memory). Heads (the elements
    before the gradients' next 128-B line, from the buffer's offset `pad`),
    ragged tails, decay tables of under 32 and of hundreds of segments (the
    two table sizes a launch carries) and a global range across index 2^32
    must give the oracle's bits."""
    n = 2 * _sms() * 2048 + 4096 + extra
    tab, params, grads, master, m, v = _random_case(n, n + pad, 1, tmax)
    if goff:
        tab = [(0, goff, 1)] + [(o + goff, sz, dcy) for o, sz, dcy in tab]
    lr, b1, b2, eps, wd, scale, t, seed = 2e-3, 0.9, 0.95, 1e-8, 0.1, 0.63, 4, 1234
    d = dict(params=dev_u16(params, pad), grads=dev_u16(grads, pad), m=dev_f32(m, pad), v=dev_f32(v, pad),
             master=dev_f32(master, pad) if with_master else None)
    d_scale = torch.tensor([scale], dtype=torch.float32, device=DEV)
    mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=lr, beta1=b1,
                     beta2=b2, eps=eps, weight_decay=wd, d_grad_scale=d_scale, t=t, seed=seed, global_offset=goff,
                     n=n)
    host = dict(params=params.copy(), master=master.copy() if with_master else None, m=m.copy(), v=v.copy())
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], goff, tab, lr, b1, b2,
                             eps, wd, f32(scale), t, seed) == 0
    _compare(d, host, f"TMA path n={n} pad={pad}")


@pytest.mark.parametrize("with_master", [True, False])
def test_step_tma_path_many_steps_and_mixed_alignment(with_master):
    """Eight steps in a row on one state (each step's results feed the next
    through the staged tiles), then the same range with the weights offset
    by 8 B against the gradients, which keeps the register path: both must
    follow the oracle bit for bit."""
    n = 2 * _sms() * 2048 + 3 * 2048 + 513
    tab, params, grads, master, m, v = _random_case(n, 77, 1, 20_000)
    host = dict(params=params.copy(), master=master.copy() if with_master else None, m=m.copy(), v=v.copy())
    d = dict(params=dev_u16(params), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master) if with_master else None)
    d_scale = torch.tensor([0.9], dtype=torch.float32, device=DEV)
    rng = np.random.default_rng(5)
    for t in range(1, 9):
        g = bf16_from_f32(rng.standard_normal(n) * 1e-2)
        mp.mp_adamw_step(d["params"], dev_u16(g), d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=1e-3,
                         beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, d_grad_scale=d_scale, t=t, seed=t)
        assert oracle.adamw_step(host["params"], g, host["master"], host["m"], host["v"], 0, tab, 1e-3, 0.9, 0.95,
                                 1e-8, 0.1, f32(0.9), t, t) == 0
    _compare(d, host, "TMA path, 8 steps")
    # weights 4 elements (8 B) off the gradients' alignment: bulk copies of the
    # weights would start mid-16-B, so this range stays on the register path
    host2 = dict(params=params.copy(), master=master.copy() if with_master else None, m=m.copy(), v=v.copy())
    d2 = dict(params=dev_u16(params, 4), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master) if with_master else None)
    mp.mp_adamw_step(d2["params"], dev_u16(grads), d2["master"], d2["m"], d2["v"], mp.TensorTable(tab), lr=1e-3,
                     beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, d_grad_scale=d_scale, t=1, seed=1)
    assert oracle.adamw_step(host2["params"], grads, host2["master"], host2["m"], host2["v"], 0, tab, 1e-3, 0.9,
                             0.95, 1e-8, 0.1, f32(0.9), 1, 1) == 0
    _compare(d2, host2, "mixed alignment")


@pytest.mark.parametrize("goff", [(1 << 32) - 3001, (1 << 32) - 3002, (1 << 32) - 3003, (1 << 32) - 3004])
def test_step_global_offset_across_2_pow_32(goff):
    """A shard whose global range crosses index 2^32 from an offset that is
    not a multiple of 4: the rounding draws' 2D fold changes inside a group."""
    n = 2048 * 5 + 17
    _, params, grads, master, m, v = _random_case(n, 17)
    tab = [(0, goff - 1000, 1), (goff - 1000, 2500, 0), (goff + 1500, n, 1)]
    d = dict(params=dev_u16(params), grads=dev_u16(grads), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master))
    mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=1e-2,
                     beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.3, d_grad_scale=None, t=2, seed=77,
                     global_offset=goff)
    host = dict(params=params.copy(), master=master.copy(), m=m.copy(), v=v.copy())
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], goff, tab, 1e-2, 0.9,
                             0.95, 1e-8, 0.3, 1.0, 2, 77) == 0
    _compare(d, host, f"offset {goff}")


@pytest.mark.parametrize("nseg", [31, 32, 33, 1023, 1024, 1025])
def test_step_segment_table_size_boundaries(nseg):
    """Tables right at and past the two kernel-parameter table sizes (32 and
    1024 decay segments); 1025 segments split into two launches."""
    seg = 53
    n = nseg * seg
    tab = [(k * seg, seg, k % 2) for k in range(nseg)]
    _, params, grads, master, m, v = _random_case(n, nseg)
    d = dict(params=dev_u16(params), grads=dev_u16(grads), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master))
    mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=1e-2,
                     beta1=0.9, beta2=0.99, eps=1e-8, weight_decay=0.5, d_grad_scale=None, t=4, seed=nseg)
    host = dict(params=params.copy(), master=master.copy(), m=m.copy(), v=v.copy())
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], 0, tab, 1e-2, 0.9, 0.99,
                             1e-8, 0.5, 1.0, 4, nseg) == 0
    _compare(d, host, f"{nseg} segments")


def test_step_many_segments_split_into_launches():
    """A table with 5000 alternating-decay tensors (more segments than one
    launch carries) gives the same result as the oracle."""
    n = 5000 * 37
    tab = [(k * 37, 37, k % 2) for k in range(5000)]
    _, params, grads, master, m, v = _random_case(n, 3)
    d = dict(params=dev_u16(params), grads=dev_u16(grads), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master))
    mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=1e-2,
                     beta1=0.9, beta2=0.99, eps=1e-8, weight_decay=0.5, d_grad_scale=None, t=3, seed=5)
    host = dict(params=params.copy(), master=master.copy(), m=m.copy(), v=v.copy())
    oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], 0, tab, 1e-2, 0.9, 0.99, 1e-8,
                      0.5, 1.0, 3, 5)
    _compare(d, host, "5000 segments")


def test_long_range_split_by_size_and_segments_equals_small_shards():
    """A range longer than one step launch takes (about 201M elements) with
    more than 1024 decay segments: the library cuts it both by size and by
    segment count; the result equals 16 small shard calls (no cuts of
    either kind) bit for bit, and sampled windows equal the oracle."""
    n = (3 << 27) + 777  # 402,654,001: three size cuts, plus segment cuts
    gen = torch.Generator().manual_seed(11)
    tab = W.random_table(n, gen, 1, 200_000)
    assert len(tab) > 3000
    g_dev = torch.randn(n, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    grads = (g_dev * 1e-2).to(torch.bfloat16)
    master = torch.randn(n, generator=torch.Generator(device="cuda").manual_seed(2), device="cuda") * 0.05
    del g_dev
    st = dict(params=master.to(torch.bfloat16), master=master, m=torch.zeros_like(master), v=torch.zeros_like(master))
    kw = dict(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, d_grad_scale=None, t=3, seed=9)
    ttab = mp.TensorTable(tab)
    win = [(0, 4096), (201_000_000, 201_700_000), (n - 5000, n)]
    host = {}
    for a, b in win:
        host[a] = dict(params=W.bf16_bits(st["params"][a:b].cpu()).copy(), master=st["master"][a:b].cpu().numpy(),
                       m=st["m"][a:b].cpu().numpy(), v=st["v"][a:b].cpu().numpy(),
                       grads=W.bf16_bits(grads[a:b].cpu()).copy())
    shards = {k: x.clone() for k, x in st.items()}
    mp.mp_adamw_step(st["params"], grads, st["master"], st["m"], st["v"], ttab, **kw)
    per = (n // 16) // 4 * 4
    for r in range(16):
        a = r * per
        b = n if r == 15 else a + per
        mp.mp_adamw_step(shards["params"][a:b], grads[a:b], shards["master"][a:b], shards["m"][a:b],
                         shards["v"][a:b], ttab, global_offset=a, n=b - a, **kw)
    torch.cuda.synchronize()
    for k in st:
        assert torch.equal(st[k].view(torch.int16) if k == "params" else st[k].view(torch.int32),
                           shards[k].view(torch.int16) if k == "params" else shards[k].view(torch.int32)), k
    del shards
    for a, b in win:
        h = host[a]
        assert oracle.adamw_step(h["params"], h["grads"], h["master"], h["m"], h["v"], a, tab, 1e-2, 0.9, 0.95,
                                 1e-8, 0.1, 1.0, 3, 9) == 0
        _compare({k: st[k][a:b] for k in st}, h, f"window {a}")


def test_shard_launches_equal_whole_buffer_and_oracle_windows():
    """GPT-2 1.5B shapes (1,557,686,400 params): the whole-buffer step and 8
    contiguous shard launches (the ZeRO-1 layout, no communication) are
    bit-identical; windows are checked against the oracle."""
    name = "gpt2_1558m"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    N = W.total(entries)
    H = W.HYPER
    st = W.make_state(name, device=DEV)
    g = W.make_grads(name, 1, device=DEV)
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])
    windows = [(0, 1 << 16), (N // 2 - 4099, 1 << 16), (N - 70001, 70001)]
    for k in range(1, 8):
        windows.append((k * (N // 8) - 3000, 6000))
    before = {k: [(to_np_u16(st["params"][a:a + n]) if k == "params" else to_np_f32(st[k][a:a + n]))
                  for a, n in windows] for k in st}
    gwin = [to_np_u16(g[a:a + n]) for a, n in windows]
    mp.mp_grad_norm(g, H["clip"], opt.workspace, opt.d_norm, opt.d_scale)
    shard = {k: t.clone() for k, t in st.items()}
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"],
              d_grad_scale=opt.d_scale, t=1, seed=W.step_seed(1))
    mp.mp_adamw_step(st["params"], g, st["master"], st["m"], st["v"], opt.table, **kw)
    per = N // 8
    for r in range(8):
        sl = slice(r * per, (r + 1) * per)
        mp.mp_adamw_step(shard["params"][sl], g[sl], shard["master"][sl], shard["m"][sl], shard["v"][sl],
                         opt.table, global_offset=r * per, **kw)
    torch.cuda.synchronize()
    for k in st:
        assert torch.equal(st[k].view(torch.int16) if k == "params" else st[k].view(torch.int32),
                           shard[k].view(torch.int16) if k == "params" else shard[k].view(torch.int32)), k
    scale = float(opt.d_scale.item())
    for i, (a, n) in enumerate(windows):
        host = {k: before[k][i].copy() for k in before}
        assert oracle.adamw_step(host["params"], gwin[i], host["master"], host["m"], host["v"], a, tab, H["lr"],
                                 H["beta1"], H["beta2"], H["eps"], H["weight_decay"], scale, 1, W.step_seed(1)) == 0
        _compare({k: st[k][a:a + n] for k in st}, host, f"1.5B window {a}")


@pytest.mark.slow
def test_llama3_8b_windows():
    """Llama-3-8B shapes (8,030,261,248 params, ~128 GB of state in HBM):
    one full step; windows (including across the 2^32 index boundary) are
    checked against the oracle; the norm against an fp64 sum over all grads."""
    name = "llama3_8b"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    N = W.total(entries)
    H = W.HYPER
    st = W.make_state(name, device=DEV)
    g = W.make_grads(name, 1, device=DEV)
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])
    windows = [(0, 1 << 16), ((1 << 32) - 50000, 100000), (N // 3, 1 << 16), (N - 100003, 100003)]
    before = {k: [(to_np_u16(st["params"][a:a + n]) if k == "params" else to_np_f32(st[k][a:a + n]))
                  for a, n in windows] for k in st}
    gwin = [to_np_u16(g[a:a + n]) for a, n in windows]
    opt.step(st["params"], g, st["master"], st["m"], st["v"], 1, W.step_seed(1))
    torch.cuda.synchronize()
    opt.check_status()
    # norm: fp64 sum over every gradient, streamed in chunks through the oracle
    s_o = 0.0
    chunk = 1 << 28
    for a in range(0, N, chunk):
        s_o += oracle.sumsq(to_np_u16(g[a:min(N, a + chunk)]))
    nrm = float(opt.d_norm.item())
    assert rel_err(nrm, math.sqrt(s_o)) <= 1e-6
    scale = float(opt.d_scale.item())
    assert scale < 1.0
    for i, (a, n) in enumerate(windows):
        host = {k: before[k][i].copy() for k in before}
        assert oracle.adamw_step(host["params"], gwin[i], host["master"], host["m"], host["v"], a, tab, H["lr"],
                                 H["beta1"], H["beta2"], H["eps"], H["weight_decay"], scale, 1, W.step_seed(1)) == 0
        _compare({k: st[k][a:a + n] for k in st}, host, f"8B window {a}")


# ---------------------------------------------------------------------------
# failure handling and memory safety
# ---------------------------------------------------------------------------
def test_nonfinite_norm_refuses_the_step():
    n = 2048 * 4 + 3
    tab, params, grads, master, m, v = _random_case(n, 11)
    grads[1234] = 0x7FC0  # a NaN gradient
    d = dict(params=dev_u16(params), grads=dev_u16(grads), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master))
    opt = mp.Optimizer(tab, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0)
    opt.step(d["params"], d["grads"], d["master"], d["m"], d["v"], 1, 1)
    torch.cuda.synchronize()
    assert math.isnan(float(opt.d_scale.item()))
    with pytest.raises(mp.MpError) as ei:
        opt.check_status()
    assert ei.value.status == mp.MP_ERR_NONFINITE
    assert_bit_equal(to_np_u16(d["params"]), params, "params untouched")
    assert_bit_equal(to_np_f32(d["master"]), master, "master untouched")
    assert_bit_equal(to_np_f32(d["m"]), m, "m untouched")
    assert_bit_equal(to_np_f32(d["v"]), v, "v untouched")


SENT16 = 0x5A5A
SENT32 = 0x7F7FA5A5  # a NaN pattern nothing computes


def _guarded(a: np.ndarray, pad: int, guard: int = 4096):
    """Device copy of a with `guard` sentinel elements on each side; returns
    (whole buffer, view of a)."""
    if a.dtype == np.uint16:
        buf = torch.full((a.size + pad + 2 * guard,), SENT16, dtype=torch.int16, device=DEV)
        v = buf[guard + pad:guard + pad + a.size]
        v.copy_(torch.from_numpy(a.view(np.int16)))
        return buf, v.view(torch.bfloat16)
    buf = torch.full((a.size + pad + 2 * guard,), SENT32, dtype=torch.int32, device=DEV)
    v = buf[guard + pad:guard + pad + a.size]
    v.copy_(torch.from_numpy(a.view(np.int32)))
    return buf, v.view(torch.float32)


def _check_guards(buf, n, pad, guard=4096):
    h = buf.cpu().numpy().astype(np.int64)
    sent = SENT16 if buf.dtype == torch.int16 else SENT32
    assert np.all(h[:guard + pad] == sent) and np.all(h[guard + pad + n:] == sent), "guard band overwritten"


@pytest.mark.parametrize("n,pad", [(1, 0), (2048 * 3 + 7, 0), (2048 * 3 + 7, 1), (4099, 3)])
def test_guard_bands_untouched(n, pad):
    tab, params, grads, master, m, v = _random_case(n, 21)
    bufs = {k: _guarded(a, pad) for k, a in dict(params=params, grads=grads, master=master, m=m, v=v).items()}
    views = {k: b[1] for k, b in bufs.items()}
    opt = mp.Optimizer(tab, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0)
    opt.step(views["params"], views["grads"], views["master"], views["m"], views["v"], 2, 9)
    out_buf, out = _guarded(np.zeros(n, np.uint16), pad)
    mp.mp_stochastic_round(out, views["master"], 4)
    torch.cuda.synchronize()
    for b, _ in list(bufs.values()) + [(out_buf, out)]:
        _check_guards(b, n, pad)


def test_resume_replay_is_bit_identical():
    """llm.c ch. 04 §5.2: restore the fp32 master/m/v, rebuild the bf16
    weights with mp_stochastic_round(master, seed of the last step), and the
    continued run equals the uninterrupted one bit for bit."""
    name = "gpt2_124m"
    n_params = 1 << 22
    from bench import prefix_entries
    entries = prefix_entries(W.layout(W.specs_for(name)), n_params)
    tab = W.table(entries)
    H = W.HYPER
    st0 = W.make_state(name, device=DEV, entries=entries)
    grads = {t: W.make_grads(name, t, device=DEV, entries=entries) for t in range(1, 7)}
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])

    def run(s, t0, t1):
        for t in range(t0, t1):
            opt.step(s["params"], grads[t], s["master"], s["m"], s["v"], t, W.step_seed(t))

    a = {k: x.clone() for k, x in st0.items()}
    run(a, 1, 7)
    b = {k: x.clone() for k, x in st0.items()}
    run(b, 1, 4)
    params_before = b["params"].clone()
    b["params"].fill_(float("nan"))  # the checkpoint holds no bf16 weights
    mp.mp_stochastic_round(b["params"], b["master"], W.step_seed(3))
    assert torch.equal(b["params"].view(torch.int16), params_before.view(torch.int16))
    run(b, 4, 7)
    torch.cuda.synchronize()
    opt.check_status()
    for k in a:
        assert torch.equal(a[k].view(torch.int16) if k == "params" else a[k].view(torch.int32),
                           b[k].view(torch.int16) if k == "params" else b[k].view(torch.int32)), k


@pytest.mark.parametrize("case", ["subnormal_moments", "overflowing_squares", "inf_nan_grads", "subnormal_weights"])
def test_step_extreme_values(case):
    """No flush-to-zero anywhere (subnormal moments and weights), squares that
    overflow to Inf, and Inf/NaN gradients run through with a unit scale: the
    bf16 weights match bit for bit (NaN is canonical there), fp32 state matches
    bit for bit apart from NaN payloads."""
    from helpers import assert_f32_bits_or_both_nan
    rng = np.random.default_rng(31)
    n = 2048 * 6 + 13
    master = (rng.standard_normal(n) * 0.05).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    g = rng.standard_normal(n)
    if case == "subnormal_moments":
        g = g * 1e-22                     # g^2 ~ 1e-44: subnormal second moment
    elif case == "overflowing_squares":
        g = g * 1e20                      # g^2 overflows fp32
    elif case == "inf_nan_grads":
        g = g * 1e-2
        g[::97] = np.inf
        g[5::101] = -np.inf
        g[7::89] = np.nan
    else:
        master = (rng.standard_normal(n) * 1e-39).astype(np.float32)  # subnormal weights, decayed
        g = g * 1e-3
    grads = bf16_from_f32(g)
    params = bf16_from_f32(master)
    tab = [(0, n // 2, 1), (n // 2, n - n // 2, 0)]
    d = dict(params=dev_u16(params), grads=dev_u16(grads), m=dev_f32(m), v=dev_f32(v), master=dev_f32(master))
    mp.mp_adamw_step(d["params"], d["grads"], d["master"], d["m"], d["v"], mp.TensorTable(tab), lr=1e-2,
                     beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, d_grad_scale=None, t=1, seed=3)
    host = dict(params=params.copy(), master=master.copy(), m=m.copy(), v=v.copy())
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], 0, tab, 1e-2, 0.9, 0.95,
                             1e-8, 0.1, 1.0, 1, 3) == 0
    assert_bit_equal(to_np_u16(d["params"]), host["params"], f"{case} params")
    for k in ("master", "m", "v"):
        assert_f32_bits_or_both_nan(to_np_f32(d[k]), host[k], f"{case} {k}")
