"""Property-based pins of the oracle's stochastic rounding, learning-rate
schedules and ZeRO-1 norm (CPU only).

For any fp32 value and any 16-bit draw, the rounding to bf16 and to fp16
(llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §2.3: keep the
value's neighbour toward zero, or move one step away from zero when the
discarded fraction of a step, as 16 bits, exceeds the draw) must:
  - land on one of the value's two neighbours on the target grid, found here
    with torch's bf16 cast and numpy's fp16 cast (round to nearest even,
    library routines that share nothing with the oracle);
  - leave values already on the grid unchanged, whatever the draw;
  - go away from zero exactly when floor(f * 65536) > draw, with f the
    fraction of one step computed here in float64 from those neighbours.
hypothesis draws the values (all fp32 magnitudes, subnormals and the
largest finite values included) and shrinks any counterexample."""
import math

import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402

FINITE_F32 = st.floats(width=32, allow_nan=False, allow_infinity=False)
DRAW = st.integers(min_value=0, max_value=0xFFFF)
SETTINGS = settings(max_examples=3000, deadline=None)
BELOW_65536 = float(np.nextafter(np.float32(65536.0), np.float32(0.0)))  # the largest fp32 below 65536


def _f32_bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def _bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def _bf16_toward_zero(x: float) -> int:
    """Pattern of the bf16 neighbour of x toward zero, from torch's cast."""
    with np.errstate(over="ignore"):
        b = int(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)[0]) & 0xFFFF
    if abs(_bf16_value(b)) > abs(x):  # the cast went away from zero (or to infinity): step back
        b -= 1
    return b


def _fp16_toward_zero(x: float) -> int:
    """Pattern of the fp16 neighbour of x toward zero, from numpy's cast."""
    with np.errstate(over="ignore"):
        h = int(np.array([x], np.float16).view(np.uint16)[0])
    if abs(float(np.array([h], np.uint16).view(np.float16)[0])) > abs(x):
        h -= 1
    return h


def _fp16_value(bits: int) -> float:
    return float(np.array([bits], np.uint16).view(np.float16)[0])


@SETTINGS
@given(x=FINITE_F32, draw=DRAW)
def test_bf16_rounding_lands_on_a_neighbour_by_the_fraction_rule(x, draw):
    x = float(np.float32(x))
    lo = _bf16_toward_zero(x)
    hi = lo + 1  # one step away from zero (sign bit unchanged)
    got = oracle.sr_with_rand(x, draw)
    assert got in (lo, hi), (x, hex(got), hex(lo))
    a = abs(_bf16_value(lo))
    step = abs(_bf16_value(hi)) - a if (hi & 0x7FFF) < 0x7F80 else 2.0 ** ((lo >> 7 & 0xFF) - 127 - 7)
    f = (abs(x) - a) / step
    assert 0.0 <= f < 1.0
    assert (got == hi) == (math.floor(f * 65536) > draw), (x, draw, f)


@SETTINGS
@given(x=FINITE_F32, draw=DRAW)
def test_bf16_rounding_keeps_values_on_the_grid(x, draw):
    b = _f32_bits(float(np.float32(x))) & 0xFFFF0000
    v = float(np.array([b], np.uint32).view(np.float32)[0])
    assert oracle.sr_with_rand(v, draw) == b >> 16


@SETTINGS
@given(x=st.floats(width=32, min_value=-BELOW_65536, max_value=BELOW_65536), draw=DRAW)
def test_fp16_rounding_lands_on_a_neighbour_by_the_fraction_rule(x, draw):
    x = float(np.float32(x))
    lo = _fp16_toward_zero(x)
    hi = lo + 1
    got = oracle.sr_fp16_with_rand(x, draw)
    assert got in (lo, hi), (x, hex(got), hex(lo))
    a = abs(_fp16_value(lo))
    step = 32.0 if (lo & 0x7FFF) == 0x7BFF else abs(_fp16_value(hi)) - a
    f = (abs(x) - a) / step
    assert 0.0 <= f < 1.0
    assert (got == hi) == (math.floor(f * 65536) > draw), (x, draw, f)


@SETTINGS
@given(h=st.integers(min_value=0, max_value=0xFFFF), draw=DRAW)
def test_fp16_rounding_keeps_values_on_the_grid(h, draw):
    v = _fp16_value(h)
    if not math.isfinite(v):
        return
    assert oracle.sr_fp16_with_rand(v, draw) == h


@SETTINGS
@given(x=st.floats(width=32, min_value=65536.0, allow_infinity=True, allow_nan=False),
       neg=st.booleans(), draw=DRAW)
def test_fp16_rounding_past_the_range_is_infinity(x, neg, draw):
    v = -x if neg else x
    assert oracle.sr_fp16_with_rand(v, draw) == (0xFC00 if neg else 0x7C00)


# --------------------------------------------------------------------------
# One AdamW step with drawn hyperparameters against torch.optim.AdamW in
# float64 (llm.c walk-through ch. 04 §2.2: m and v as lerps, bias-corrected
# moments, decoupled decay on decay-flagged tensors, the clip scale on the
# gradient). The bound is fp32 rounding of each operation of the step, taken
# from the float64 reference values, with a factor 4 of slack. The betas are
# 0 or at least 1e-4: torch forms m as m0 + (1 - beta1)(g - m0), and below
# 2^-53 the float64 1 - beta1 is exactly 1, dropping beta1 * m0 from its
# reference.
# --------------------------------------------------------------------------
U = 2.0 ** -24


def _log_uniform(lo, hi):
    return st.floats(min_value=math.log10(lo), max_value=math.log10(hi)).map(lambda e: 10.0 ** e)


def _f32(x):
    return float(np.float32(x))


@settings(max_examples=300, deadline=None)
@given(b1=st.one_of(st.just(0.0), st.floats(1e-4, 0.999)), b2=st.one_of(st.just(0.0), st.floats(1e-4, 0.9999)),
       lr=_log_uniform(1e-6, 1.0),
       eps=_log_uniform(1e-10, 1e-2), wd=st.floats(0.0, 1.0), t=st.integers(1, 100000),
       scale=st.floats(0.01, 1.0), decay=st.booleans(), master=st.booleans(), seed=st.integers(0, 2 ** 32 - 1))
def test_one_step_tracks_torch_adamw_fp64(b1, b2, lr, eps, wd, t, scale, decay, master, seed):
    b1, b2, lr, eps, wd, scale = (_f32(x) for x in (b1, b2, lr, eps, wd, scale))
    rng = np.random.default_rng(seed)
    n = 256
    sign = lambda: rng.choice([-1.0, 1.0], n)  # noqa: E731
    g32 = (sign() * 10.0 ** rng.uniform(-6, 2, n)).astype(np.float32)
    g32[:8] = 0.0
    gbits = W_bf16(g32)
    g = (gbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    old32 = (sign() * 10.0 ** rng.uniform(-3, 3, n)).astype(np.float32)
    pbits = W_bf16(old32)
    if not master:
        old32 = (pbits.astype(np.uint32) << 16).view(np.float32)
    m0 = (sign() * 10.0 ** rng.uniform(-6, 2, n)).astype(np.float32)
    v0 = (10.0 ** rng.uniform(-12, 4, n)).astype(np.float32)
    ms, m, v, params = old32.copy(), m0.copy(), v0.copy(), pbits.copy()
    assert oracle.adamw_step(params, gbits.copy(), ms if master else None, m, v, 0, [(0, n, int(decay))],
                             lr, b1, b2, eps, wd, scale, t, 11) == 0

    wd_e = wd if decay else 0.0
    p = torch.nn.Parameter(torch.from_numpy(old32.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd_e, foreach=False)
    opt.state[p] = {"step": torch.tensor(float(t - 1)), "exp_avg": torch.from_numpy(m0.astype(np.float64)),
                    "exp_avg_sq": torch.from_numpy(v0.astype(np.float64))}
    p.grad = torch.from_numpy(g * scale)
    opt.step()
    p_ref = p.detach().numpy()
    m_ref = opt.state[p]["exp_avg"].numpy()
    v_ref = opt.state[p]["exp_avg_sq"].numpy()

    old = old32.astype(np.float64)
    gs = np.abs(g * scale)
    DN = 2.0 ** -149  # fp32 subnormal spacing: the absolute error floor of each operation
    dm = 2 * U * (b1 * np.abs(m0) + (1 - b1) * gs) + U * (1 - b1) * gs + 2 * DN
    dv = 5 * U * (b2 * v0 + (1 - b2) * gs * gs) + 2 * DN
    bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
    m_hat, v_hat = m_ref / bc1, v_ref / bc2
    dmh = dm / bc1 + 2 * U * np.abs(m_hat) + DN
    dvh = dv / bc2 + 2 * U * v_hat + DN
    sq = np.sqrt(v_hat)
    with np.errstate(divide="ignore"):
        dsq = np.minimum(np.sqrt(dvh), np.where(sq > 0, dvh / (2 * sq), np.inf)) + U * sq
    d = sq + eps
    dd = dsq + U * d
    u = m_hat / d
    du = dmh / d + np.abs(u) * dd / d + U * np.abs(u) + DN
    term = u + wd_e * old
    dterm = du + U * wd_e * np.abs(old) + U * np.abs(term) + DN
    dp = U * np.abs(p_ref) + lr * dterm + U * lr * np.abs(term) + U * np.abs(old) + DN

    def worst(err, bound):
        return float((err / bound).max())

    assert (np.abs(m - m_ref) <= 4 * dm).all(), worst(np.abs(m - m_ref), dm)
    assert (np.abs(v - v_ref) <= 4 * dv).all(), worst(np.abs(v - v_ref), dv)
    if master:
        err = np.abs(ms.astype(np.float64) - p_ref)
        assert (err <= 4 * dp).all(), worst(err, dp)
    # the bf16 weight is within one bf16 step of the fp32 result
    pf = (params.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(p_ref), 1e-30))) - 7)
    assert (np.abs(pf - p_ref) <= ulp * (1 + 1e-6) + 4 * dp).all()


def W_bf16(x32: np.ndarray) -> np.ndarray:
    """bf16 patterns of fp32 values by torch's round-to-nearest cast."""
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# Learning-rate schedules and the ZeRO-1 norm (llm.c ch. 04 §4): properties
# over drawn arguments.
# --------------------------------------------------------------------------
# lr_min = frac * lr_max with frac 0 or at least 1e-6: the schedules' double
# arithmetic (lr_max - (lr_max - lr_min) * p) returns lr_min at the end only
# while lr_min is not far below lr_max's rounding error.
SCHED = st.tuples(st.integers(0, 3), st.integers(0, 400), st.integers(1, 20_000),
                  st.floats(1e-6, 1.0), st.one_of(st.just(0.0), st.floats(1e-6, 1.0)), st.floats(0.01, 1.0))


@settings(max_examples=300, deadline=None)
@given(SCHED)
def test_lr_schedule_stays_between_its_bounds_and_moves_one_way(args):
    kind, warmup, span, hi, frac_lo, f = args
    lo = float(np.float32(hi * frac_lo))
    hi32 = float(np.float32(hi))
    total = warmup + span
    ulp = 2.0 ** -23
    prev = None
    ts = sorted(set([1, warmup, warmup + 1, total, total + 5] + list(range(1, total + 2, max(1, total // 60)))))
    for t in [t for t in ts if t >= 1]:
        x = float(oracle.lr(kind, warmup, total, hi, lo, f, t))
        if t <= warmup:
            assert 0.0 < x <= hi32 * (1 + ulp)
            if prev is not None and prev[0] <= warmup:
                assert x >= prev[1] * (1 - ulp)  # the warm-up rises
        else:
            assert lo * (1 - ulp) <= x <= hi32 * (1 + ulp)
            if prev is not None and prev[0] > warmup:
                assert x <= prev[1] * (1 + ulp)  # after it, nothing rises
            if kind == 0:
                assert x == hi32
            if t >= total and kind != 0:
                assert x == np.float32(lo)
        prev = (t, x)


@settings(max_examples=500, deadline=None)
@given(st.lists(st.floats(0.0, 1e30), min_size=1, max_size=64), st.floats(1e-3, 1e3))
def test_zero1_norm_is_the_rank_sum_within_rounding(parts, clip):
    s, nrm, sc = oracle.norm_from_parts(parts, clip)
    exact = math.fsum(parts)
    assert abs(s - exact) <= len(parts) * 2.0 ** -53 * exact
    # the norm is the float rounding of the sum's square root (below fp32's
    # range that is a subnormal or zero: half its spacing, 2^-150, at most)
    r = math.sqrt(s)
    assert abs(float(nrm) - r) <= max(2.0 ** -24 * r, 2.0 ** -150)
    # and the clip scale follows the rule min(1, clip / norm) in fp32
    if float(nrm) == 0.0:
        assert sc == 1.0
    else:
        with np.errstate(over="ignore"):  # a subnormal norm overflows clip / norm to +Inf, as in fp32
            q = np.float32(np.float32(clip) / nrm)
        assert sc == min(np.float32(1.0), q)
