"""Pins of the CPU oracle to facts the pages and mathematics fix (no GPU).

Each test checks the oracle against something other than itself: numbers the
pages print (tests/golden/), closed forms of the first Adam step, invariants
(no decay on 1D tensors, shard invariance), exhaustive enumeration of the
rounding rule, a statistical check of unbiasedness, and library routines
(torch.optim.AdamW in fp64, math.fsum, torch's bf16 cast).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

F32 = np.float32


def f32(x):
    return float(np.float32(x))


def bf16_value(bits):
    return float(oracle.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0])


# --------------------------------------------------------------------------
# Bias correction — CMU 11-667 lecture 13 notes §1.7 and §7.3 exercise 1.
# --------------------------------------------------------------------------
def test_bias_correction_multipliers_match_printed_values(golden):
    rows = golden("bias_correction_multipliers.txt")
    assert len(rows) == 11
    for b1, b2, t, printed in rows:
        bc1, bc2 = oracle.bias_corrections(float(b1), float(b2), int(t))
        mult = float(bc1) / math.sqrt(float(bc2))
        # printed to 3 significant figures: within half a unit of the last digit
        digits = len(printed.split(".")[1])
        assert abs(mult - float(printed)) <= 0.5 * 10 ** -digits + 1e-9, (b1, b2, t, mult, printed)


def test_bias_correction_is_one_minus_beta_to_the_t():
    # t = 1: bc = 1 - beta exactly as rounded once to float
    bc1, bc2 = oracle.bias_corrections(0.9, 0.95, 1)
    assert bc1 == F32(1.0 - float(F32(0.9))) and bc2 == F32(1.0 - float(F32(0.95)))
    # large t: corrections tend to 1
    bc1, bc2 = oracle.bias_corrections(0.9, 0.95, 10000)
    assert bc1 == F32(1.0) and bc2 == F32(1.0)


# --------------------------------------------------------------------------
# First Adam step in closed form — llm.c ch. 04 §2.2 with m = v = 0, t = 1:
# m = (1-b1) g, v = (1-b2) g^2, so m_hat = g, v_hat = g^2 and
# p = old - lr * (g / (|g| + eps) + wd * old).
# --------------------------------------------------------------------------
def _one_tensor_step(g_vals, old, lr, b1, b2, eps, wd, decay=1, scale=1.0, t=1, master=True):
    n = len(g_vals)
    gbits = W.bf16_bits(torch.tensor(g_vals, dtype=torch.float32).to(torch.bfloat16))
    g = oracle.bf16_bits_to_f32(gbits).astype(np.float64)
    old = np.asarray(old, dtype=np.float32)
    ms = old.copy()
    params = W.bf16_bits(torch.from_numpy(old.copy()).to(torch.bfloat16)).copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    st = oracle.adamw_step(params, gbits.copy(), ms if master else None, m, v, 0, [(0, n, decay)],
                           lr, b1, b2, eps, wd, scale, t, 7)
    assert st == 0
    return g, old.astype(np.float64), ms, m, v, params


@pytest.mark.parametrize("lr,wd,eps", [(1e-3, 0.1, 1e-8), (0.1, 0.5, 1e-8), (0.05, 0.0, 1e-3)])
def test_first_step_closed_form(lr, wd, eps):
    rng = np.random.default_rng(0)
    n = 4096
    g_vals = rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 1, n)
    old = (rng.standard_normal(n) * 0.05).astype(np.float32)
    b1, b2 = 0.9, 0.95
    g, old64, p, m, v, _ = _one_tensor_step(g_vals, old, lr, b1, b2, eps, wd)
    B1, B2, LR, WD, EPS = (f32(x) for x in (b1, b2, lr, wd, eps))
    # moments
    np.testing.assert_allclose(m, (1.0 - B1) * g, rtol=2 ** -22, atol=0)
    np.testing.assert_allclose(v, (1.0 - B2) * g * g, rtol=2 ** -21, atol=0)
    # update: bias correction cancels (1 - beta) exactly up to rounding
    expect = old64 - LR * (g / (np.abs(g) + EPS) + WD * old64)
    err = np.abs(p.astype(np.float64) - expect)
    bound = 2 ** -22 * (np.abs(old64) + LR * (1.0 + WD * np.abs(old64))) + 2 ** -24 * np.abs(expect)
    assert (err <= bound).all(), float((err / bound).max())


def test_first_step_moves_each_weight_by_lr_sign_g_when_eps_is_tiny():
    rng = np.random.default_rng(1)
    n = 2048
    g_vals = rng.standard_normal(n) * 10.0 ** rng.uniform(-8, 2, n)
    old = (rng.standard_normal(n) * 0.02).astype(np.float32)
    lr = 1e-3
    g, old64, p, _, _, _ = _one_tensor_step(g_vals, old, lr, 0.9, 0.999, 1e-30, 0.0)
    step = p.astype(np.float64) - old64
    np.testing.assert_allclose(step, -f32(lr) * np.sign(g), rtol=1e-5, atol=2 ** -24 * 0.1)


def test_no_master_variant_reads_old_weight_from_bf16():
    rng = np.random.default_rng(2)
    n = 512
    g_vals = rng.standard_normal(n) * 1e-3
    old = W.bf16_bits(torch.from_numpy((rng.standard_normal(n) * 0.05).astype(np.float32)).to(torch.bfloat16))
    old_f = oracle.bf16_bits_to_f32(old)
    g, old64, _, _, _, params = _one_tensor_step(g_vals, old_f, 0.01, 0.9, 0.95, 1e-8, 0.1, master=False)
    expect = old64 - f32(0.01) * (g / (np.abs(g) + f32(1e-8)) + f32(0.1) * old64)
    got = oracle.bf16_bits_to_f32(params).astype(np.float64)
    # the bf16 result is one of the two bf16 neighbours of the fp32 update,
    # which itself carries fp32 rounding of order 2^-23 (|old| + lr)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(expect))) - 7)
    fp32_err = 2 ** -22 * (np.abs(old64) + f32(0.01) * (1 + f32(0.1) * np.abs(old64)))
    assert (np.abs(got - expect) <= ulp * 1.0001 + fp32_err).all()


def test_nonfinite_scale_writes_nothing():
    n = 64
    params = np.arange(n, dtype=np.uint16)
    grads = np.full(n, 0x3F80, dtype=np.uint16)
    master = np.ones(n, np.float32)
    m = np.ones(n, np.float32)
    v = np.ones(n, np.float32)
    for bad in (float("nan"), float("inf"), float("-inf")):
        before = [a.copy() for a in (params, master, m, v)]
        st = oracle.adamw_step(params, grads, master, m, v, 0, [(0, n, 1)],
                               1e-3, 0.9, 0.95, 1e-8, 0.1, bad, 1, 3)
        assert st == 5
        for a, b in zip((params, master, m, v), before):
            assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# Decay only on 2D tensors — llm.c ch. 04 §2.2.
# --------------------------------------------------------------------------
def test_zero_gradient_leaves_1d_tensors_unchanged_and_decays_2d():
    entries = W.layout(W.specs_for("tiny"))
    tab = W.table(entries)
    st = W.make_state("tiny")
    master = st["master"].numpy().copy()
    params = W.bf16_bits(st["params"]).copy()
    N = master.size
    m = np.zeros(N, np.float32)
    v = np.zeros(N, np.float32)
    grads = np.zeros(N, np.uint16)
    lr, wd = 1e-3, 0.1
    master0, params0 = master.copy(), params.copy()
    assert oracle.adamw_step(params, grads, master, m, v, 0, tab, lr, 0.9, 0.95, 1e-8, wd, 1.0, 1, 11) == 0
    LR, WD = F32(lr), F32(wd)
    for e in entries:
        sl = slice(e.offset, e.offset + e.size)
        if e.spec.decay:
            expect = master0[sl] - LR * (WD * master0[sl])  # fp32 ops, same rounding
            assert np.array_equal(master[sl], expect), e.spec.name
        else:
            assert np.array_equal(master[sl], master0[sl]), e.spec.name
            assert np.array_equal(params[sl], params0[sl]), e.spec.name  # 1 and 0 are exact in bf16
    assert np.all(m == 0) and np.all(v == 0)


# --------------------------------------------------------------------------
# 16 steps against torch.optim.AdamW (fp64) on the 28,672-param model —
# CMU 11-667 lecture 13 notes §1.6 check their optimizers against torch.optim
# over 16 steps; llm.c's update is the same mathematics (decoupled decay).
# --------------------------------------------------------------------------
def test_sixteen_steps_track_torch_adamw_fp64():
    name = "tiny"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    st = W.make_state(name)
    master = st["master"].numpy().copy()
    params = W.bf16_bits(st["params"]).copy()
    N = master.size
    m = np.zeros(N, np.float32)
    v = np.zeros(N, np.float32)
    H = {k: f32(x) for k, x in W.HYPER.items()}

    ref = [torch.nn.Parameter(st["master"][e.offset:e.offset + e.size].double().clone()) for e in entries]
    groups = [dict(params=[p for p, e in zip(ref, entries) if e.spec.decay], weight_decay=H["weight_decay"]),
              dict(params=[p for p, e in zip(ref, entries) if not e.spec.decay], weight_decay=0.0)]
    opt = torch.optim.AdamW(groups, lr=H["lr"], betas=(H["beta1"], H["beta2"]), eps=H["eps"], foreach=False)

    scales = []
    gmax = np.zeros(N)
    for t in range(1, 17):
        g = W.make_grads(name, t)
        gbits = W.bf16_bits(g).copy()
        _, norm, scale = oracle.grad_norm(gbits, H["clip"])
        scales.append(float(scale))
        assert oracle.adamw_step(params, gbits, master, m, v, 0, tab, H["lr"], H["beta1"], H["beta2"],
                                 H["eps"], H["weight_decay"], float(scale), t, W.step_seed(t)) == 0
        gd = g.double() * float(scale)
        gmax = np.maximum(gmax, np.abs(gd.numpy()))
        for p, e in zip(ref, entries):
            p.grad = gd[e.offset:e.offset + e.size].clone()
        opt.step()
    assert max(scales) < 1.0  # clipping was active on every step
    refp = torch.cat([p.detach() for p in ref]).numpy()
    st_m = torch.cat([opt.state[p]["exp_avg"] for p in ref]).numpy()
    st_v = torch.cat([opt.state[p]["exp_avg_sq"] for p in ref]).numpy()
    # fp32 rounding: about one ulp per step of the largest magnitude the weight
    # passed through, |p| <= |p0| + 16 lr (1 + wd |p|), over 16 steps
    err = np.abs(master.astype(np.float64) - refp)
    p0 = np.abs(st["master"].numpy().astype(np.float64))
    bound = 16 * 2 ** -23 * (np.maximum(p0, np.abs(refp)) + 16 * H["lr"] * 1.2)
    assert (err <= bound).all(), float((err / bound).max())
    assert float(err.mean()) < 1e-8
    # m is a signed average: its rounding error scales with the gradients it
    # averaged, not with |m| (which may cross zero)
    assert (np.abs(m - st_m) <= 16 * 2 ** -23 * (np.abs(st_m) + gmax)).all()
    np.testing.assert_allclose(v, st_v, rtol=2e-6, atol=1e-16)
    # the bf16 weights are a stochastic rounding of the fp32 master
    pf = oracle.bf16_bits_to_f32(params).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(master.astype(np.float64)), 1e-30))) - 7)
    assert (np.abs(pf - master) <= ulp).all()


# --------------------------------------------------------------------------
# Stochastic rounding — llm.c ch. 04 §2.3.
# --------------------------------------------------------------------------
SR_VALUES = [1.0 + 2 ** -9, -(1.0 + 3 * 2 ** -10), 257.0, 0.1, -3.3e-5, 1e-40, -2.5e-39, 3.0e38]


def _bits(x):
    return int(np.array([x], np.float32).view(np.uint32)[0])


@pytest.mark.parametrize("x", SR_VALUES)
def test_sr_exhaustive_over_all_draws(x):
    b = _bits(x)
    lo, trunc = b & 0xFFFF, b >> 16
    ups = 0
    for r in range(65536):
        out = oracle.sr_with_rand(x, r)
        assert out in (trunc, trunc + 1)
        ups += out == trunc + 1
    assert ups == lo  # P(away from zero) = lo16 / 65536 exactly
    down = bf16_value(trunc)
    up = bf16_value(trunc + 1)
    xf = float(np.float32(x))
    # truncation moves toward zero, the increment away from zero
    assert abs(down) <= abs(xf) < abs(up) and math.copysign(1, down) == math.copysign(1, xf)
    # {down, up} are x's two bf16 neighbours: torch's round-to-nearest cast picks one of them
    assert torch.tensor(xf, dtype=torch.float64).to(torch.bfloat16).item() in (down, up)


def test_sr_leaves_bf16_representable_values_unchanged():
    rng = np.random.default_rng(3)
    pats = rng.integers(0, 0x7F80, 4000).astype(np.uint32)
    pats |= (rng.integers(0, 2, 4000).astype(np.uint32) << 15)
    xs = (pats << 16).view(np.float32)
    for x, p in zip(xs[:400], pats[:400]):
        for r in (0, 1, 0x7FFF, 0xFFFF):
            assert oracle.sr_with_rand(float(x), r) == p
    out = oracle.stochastic_round(xs, 12345, 99)
    assert np.array_equal(out, pats.astype(np.uint16))


def test_sr_special_values():
    assert oracle.sr_with_rand(float("inf"), 0) == 0x7F80
    assert oracle.sr_with_rand(float("-inf"), 0) == 0xFF80
    assert oracle.sr_with_rand(0.0, 0) == 0x0000
    assert oracle.sr_with_rand(-0.0, 0) == 0x8000
    assert oracle.sr_with_rand(float("nan"), 0xFFFF) == 0x7FC0
    # NaNs whose payload lies only in the low 16 bits would truncate to an
    # infinity; pass their raw patterns through the array entry point (a
    # Python float would quiet them and set a high payload bit)
    nans = np.array([0x7F800001, 0xFF800003, 0x7F80FFFF, 0xFF80FFFF, 0x7FC00000, 0x7FFFFFFF],
                    np.uint32).view(np.float32)
    for seed in range(4):
        assert np.all(oracle.stochastic_round(nans, 1000 * seed, seed) == 0x7FC0)
    # the largest finite fp32 rounds to bf16 max or to +Inf (carry into the exponent)
    big = float(np.finfo(np.float32).max)
    assert oracle.sr_with_rand(big, 0xFFFF) == 0x7F7F
    assert oracle.sr_with_rand(big, 0) == 0x7F80
    # smallest subnormal: up w.p. 1/65536 ... to the smallest bf16 subnormal
    tiny = float(np.array([1], np.uint32).view(np.float32)[0])
    assert oracle.sr_with_rand(tiny, 0) == 0x0001
    assert oracle.sr_with_rand(tiny, 1) == 0x0000


@pytest.mark.parametrize("x", [1.0 + 2 ** -9, -0.3, 7.77e-3, 1.0 + 2 ** -8])
def test_sr_is_unbiased_over_1e5_seeds(x):
    """The mean over 10^5 seeds lies within 4 sigma of x (llm.c ch. 04 §2.3:
    the rounding equals the true value in expectation)."""
    L = oracle.lib()
    n = 100_000
    k = 987654321
    outs = np.fromiter((L.oracle_sr(x, k, s) for s in range(n)), dtype=np.uint16, count=n)
    vals = oracle.bf16_bits_to_f32(outs).astype(np.float64)
    b = _bits(x)
    f = (b & 0xFFFF) / 65536.0
    ulp = abs(bf16_value((b >> 16) + 1) - bf16_value(b >> 16))
    sigma = ulp * math.sqrt(f * (1 - f)) / math.sqrt(n)
    xf = float(np.float32(x))
    assert abs(vals.mean() - xf) <= 4 * sigma, (vals.mean() - xf, sigma)


def test_sr_halfway_values_from_bf16_facts(golden):
    """257 and 1 + 2^-8 sit exactly half-way between two bf16 values (CMU
    11-667 lecture 13 notes §7.3 exercise 5); SR sends exactly half of all
    draws each way, where round-to-nearest-even always picks the even one."""
    for x, lo_val, hi_val in ((257.0, 256.0, 258.0), (1.0 + 2 ** -8, 1.0, 1.0078125)):
        outs = [bf16_value(oracle.sr_with_rand(x, r)) for r in range(65536)]
        assert outs.count(hi_val) == 32768 and outs.count(lo_val) == 32768


def test_bf16_facts_of_the_input_cast(golden):
    for fmt, x, expect in golden("bf16_facts.txt"):
        dt = torch.bfloat16 if fmt == "bf16" else torch.float16
        got = torch.tensor(float(x), dtype=torch.float64).to(dt).double().item()
        assert got == float(expect), (fmt, x, got)


# --------------------------------------------------------------------------
# Rounding randomness: uniform low 16 bits (what makes SR unbiased).
# Its exact values follow the published SquirrelNoise5 definition; the pages
# print no test vector for it.
# --------------------------------------------------------------------------
def _chi2_uniform16(vals):
    counts = np.bincount(vals.astype(np.int64), minlength=65536)
    e = vals.size / 65536.0
    return float(((counts - e) ** 2 / e).sum())


@pytest.mark.parametrize("first,seed", [(0, 0), (123456789, 42), ((1 << 32) - 100000, 7), (5 << 32, 2024)])
def test_noise_low16_uniform_chi2(first, seed):
    r = oracle.noise_fill(first, 1 << 22, seed)
    chi2 = _chi2_uniform16(r & 0xFFFF)
    dof = 65535
    assert abs(chi2 - dof) < 6 * math.sqrt(2 * dof), chi2
    chi2_hi = _chi2_uniform16(r >> 16)
    assert abs(chi2_hi - dof) < 6 * math.sqrt(2 * dof), chi2_hi


def test_noise_over_seeds_uniform_and_uncorrelated():
    L = oracle.lib()
    n = 1 << 20
    r = np.fromiter((L.oracle_noise_u32(77, s) for s in range(n)), dtype=np.uint32, count=n)
    chi2 = _chi2_uniform16(r & 0xFFFF)
    assert abs(chi2 - 65535) < 6 * math.sqrt(2 * 65535)
    a = oracle.noise_fill(1000, n + 1, 5).astype(np.float64)
    for x, y in ((a[:-1], a[1:]), (r[:-1].astype(np.float64), r[1:].astype(np.float64))):
        c = np.corrcoef(x, y)[0, 1]
        assert abs(c) < 5 / math.sqrt(n), c
    b = oracle.noise_fill(1000, n, 6).astype(np.float64)
    assert abs(np.corrcoef(a[:-1], b)[0, 1]) < 5 / math.sqrt(n)


def test_noise_depends_on_the_high_index_word():
    lo = oracle.noise_fill(0, 4096, 9)
    hi = oracle.noise_fill(1 << 32, 4096, 9)
    assert np.mean(lo == hi) < 0.01


def test_noise_avalanche():
    """Strict avalanche: flipping any one bit of the element index (its low
    44 bits) or of the seed flips each of the 32 output bits with probability
    1/2. A hash that mixes fully has this; dropping one of its multiply or
    xor-shift rounds breaks it for some input bit. 4000 random (index, seed)
    pairs per input bit; every estimate within 0.05 of 1/2 (about 6 standard
    deviations)."""
    L = oracle.lib()
    rng = np.random.default_rng(11)
    n = 4000
    idx = rng.integers(0, 1 << 44, n, dtype=np.uint64)
    seeds = rng.integers(0, 1 << 32, n, dtype=np.uint64)
    f = L.oracle_noise_u32
    base = np.array([f(int(i), int(s)) for i, s in zip(idx, seeds)], dtype=np.uint64)
    shifts = np.arange(32, dtype=np.uint64)
    for b in range(44 + 32):
        if b < 44:
            out = [f(int(i) ^ (1 << b), int(s)) for i, s in zip(idx, seeds)]
        else:
            out = [f(int(i), int(s) ^ (1 << (b - 44))) for i, s in zip(idx, seeds)]
        flips = ((base ^ np.array(out, dtype=np.uint64))[:, None] >> shifts) & 1
        worst = float(np.abs(flips.mean(axis=0) - 0.5).max())
        assert worst < 0.05, (b, worst)


# --------------------------------------------------------------------------
# Gradient norm and clip scale — llm.c ch. 04 §4.
# --------------------------------------------------------------------------
def test_norm_of_all_ones_is_sqrt_n():
    for n in (1, 7, 28672, 1 << 20):
        s, nrm, sc = oracle.grad_norm(np.full(n, 0x3F80, np.uint16), 1.0)
        assert s == float(n)
        assert nrm == F32(math.sqrt(n))
        assert sc == (F32(1.0) / F32(math.sqrt(n)) if n > 1 else F32(1.0))


def test_norm_of_power_of_two_pattern_is_exact():
    n = 100003
    k = np.arange(n) % 9 - 4
    vals = np.ldexp(1.0, k) * np.where(np.arange(n) % 2 == 0, 1.0, -1.0)
    bits = W.bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))
    s = oracle.sumsq(bits)
    assert s == float(sum(4.0 ** int(e) for e in k))  # every partial sum is exact


def test_norm_matches_math_fsum():
    rng = np.random.default_rng(4)
    for n, scale in ((1000, 1e-3), (200003, 1.0), (50000, 1e20), (5000, 1e-25)):
        vals = rng.standard_normal(n) * scale
        bits = W.bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))
        g = oracle.bf16_bits_to_f32(bits).astype(np.float64)
        exact = math.fsum(g * g)  # squares of bf16 values are exact in fp64
        s = oracle.sumsq(bits)
        assert abs(s - exact) <= n * 2 ** -53 * exact


def test_clip_scale_rule():
    cs = oracle.clip_scale
    assert cs(2.0, 1.0) == F32(0.5)
    assert cs(0.5, 1.0) == F32(1.0)
    assert cs(1.0, 1.0) == F32(1.0)
    assert cs(0.0, 1.0) == F32(1.0)
    assert cs(3.0, 1.0) == F32(1.0) / F32(3.0)
    assert cs(10.0, 2.5) == F32(0.25)
    for bad in (float("nan"), float("inf")):
        assert math.isnan(cs(bad, 1.0))


def test_norm_with_nonfinite_grads_gives_nan_scale():
    g = np.full(100, 0x3F80, np.uint16)
    g[37] = 0x7FC0
    _, nrm, sc = oracle.grad_norm(g, 1.0)
    assert math.isnan(nrm) and math.isnan(sc)
    g[37] = 0xFF80  # -inf
    _, nrm, sc = oracle.grad_norm(g, 1.0)
    assert math.isinf(nrm) and math.isnan(sc)


# --------------------------------------------------------------------------
# ZeRO-1 shards — CMU 11-667 lecture 13 notes §5.2 (max difference 0 versus
# data parallelism); llm.c ch. 04 §3.2 (contiguous num_params / world slices).
# --------------------------------------------------------------------------
def test_shard_bytes_of_the_tiny_model(golden):
    kv = {k: int(v) for k, v in golden("zero1_state_bytes.txt")}
    N = W.total(W.layout(W.specs_for("tiny")))
    assert N == kv["params"]
    assert 8 * N == kv["adam_state_bytes_full"]
    assert 8 * N // kv["cards"] == kv["adam_state_bytes_per_card"]


@pytest.mark.parametrize("with_master", [True, False])
def test_sharded_steps_equal_whole_buffer_steps(with_master):
    name = "tiny"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    st = W.make_state(name)
    N = W.total(entries)
    whole = dict(params=W.bf16_bits(st["params"]).copy(), master=st["master"].numpy().copy(),
                 m=np.zeros(N, np.float32), v=np.zeros(N, np.float32))
    shard = {k: a.copy() for k, a in whole.items()}
    H = W.HYPER
    world = 4
    for t in range(1, 41):
        g = W.bf16_bits(W.make_grads(name, t)).copy()
        _, _, scale = oracle.grad_norm(g, H["clip"])
        args = (H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], float(scale), t, W.step_seed(t))
        oracle.adamw_step(whole["params"], g, whole["master"] if with_master else None, whole["m"], whole["v"],
                          0, tab, *args)
        per = N // world
        for r in range(world):
            sl = slice(r * per, (r + 1) * per)
            views = {k: shard[k][sl] for k in shard}
            assert oracle.adamw_step(views["params"], g[sl].copy(), views["master"] if with_master else None,
                                     views["m"], views["v"], r * per, tab, *args) == 0
    for k in whole:
        if k == "master" and not with_master:
            continue
        assert np.array_equal(whole[k], shard[k]), k


# --------------------------------------------------------------------------
# Why stochastic rounding: small updates survive (llm.c ch. 04 §2.3; CMU
# 11-667 lecture 13 notes §2.3). Constant update 1e-4 |w0| for 1000 steps.
# --------------------------------------------------------------------------
def test_sr_tracks_small_updates_where_round_to_nearest_stalls():
    n = 1 << 14
    w0 = W.sr_stress_weights(n).numpy()
    delta = (np.float32(1e-4) * np.abs(w0)).astype(np.float32)
    fp32 = w0.copy()
    sr_bits = W.bf16_bits(torch.from_numpy(w0).to(torch.bfloat16)).copy()
    rne = torch.from_numpy(w0).to(torch.bfloat16)
    for t in range(1, 1001):
        fp32 = (fp32 + delta).astype(np.float32)
        x = (oracle.bf16_bits_to_f32(sr_bits) + delta).astype(np.float32)
        sr_bits = oracle.stochastic_round(x, 0, W.step_seed(t))
        rne = (rne.float() + torch.from_numpy(delta)).to(torch.bfloat16)
    rel_rne = float(np.mean(rne.float().numpy().astype(np.float64) / fp32 - 1.0))
    rel_sr = float(np.mean(oracle.bf16_bits_to_f32(sr_bits).astype(np.float64) / fp32 - 1.0))
    # round-to-nearest never moves (the update is below half a bf16 step):
    assert np.array_equal(rne.float().numpy(), torch.from_numpy(w0).to(torch.bfloat16).float().numpy())
    # so its relative drift is w0 / (w0 + 1000 * 1e-4 |w0|) - 1 = -1/11 for w0 > 0 and +1/9 for w0 < 0
    expect = float(np.mean(np.where(w0 > 0, 1 / 1.1 - 1, 1 / 0.9 - 1)))
    assert abs(rel_rne - expect) < 2e-3
    assert abs(rel_sr) < 2e-3  # SR follows the fp32 trajectory in expectation


# --------------------------------------------------------------------------
# Stochastic rounding to fp16 — the rule of llm.c ch. 04 §2.3 on fp16's grid
# (§6: unfinished upstream). The fp16 grid comes from numpy's float16.
# --------------------------------------------------------------------------
def _fp16_neighbours(x):
    """The fp16 values toward zero (a) and away from zero (b) of fp32 x, from
    numpy's float16 grid."""
    ax = abs(float(x))
    with np.errstate(over="ignore"):  # past the largest finite fp16 the neighbour is infinity
        h = np.float16(ax)  # round to nearest
        if float(h) > ax:
            h = np.nextafter(h, np.float16(0))
        b = np.nextafter(h, np.float16(np.inf))
    return float(h), float(b)


def test_sr_fp16_keeps_every_fp16_value():
    h = np.arange(0, 0x7C00, dtype=np.uint16)           # every finite non-negative fp16
    vals = np.concatenate([h.view(np.float16), -h.view(np.float16)]).astype(np.float32)
    for r in (0, 1, 12345, 65535):
        got = np.array([oracle.sr_fp16_with_rand(float(v), r) for v in vals[::97]], np.uint16)
        assert np.array_equal(got.view(np.float16).astype(np.float32), vals[::97])


@pytest.mark.parametrize("x", [1.0 + 2 ** -12, 3.14159, -0.1, 1000.3, 65504.5, 65535.9, -65520.0,
                               1e-5, 3e-8, -1.5e-7, 6.1e-5])
def test_sr_fp16_exhaustive_over_draws(x):
    """Over all 65,536 draws the result is one of numpy's two fp16 neighbours
    and rounds away from zero exactly floor(f * 65536) times."""
    x = float(np.float32(x))
    a, b = _fp16_neighbours(x)
    f = (abs(x) - a) / (b - a) if math.isfinite(b) else (abs(x) - a) / 32.0
    outs = np.array([oracle.sr_fp16_with_rand(x, r) for r in range(65536)], np.uint16)
    vals = np.abs(outs.view(np.float16).astype(np.float64))
    assert set(np.unique(vals).tolist()) <= {a, b}
    assert int((vals == b).sum()) == math.floor(f * 65536)
    assert np.all((outs & 0x8000) == (0x8000 if x < 0 else 0))
    # round-to-nearest (numpy) is one of the two outcomes
    with np.errstate(over="ignore"):
        assert abs(float(np.float16(x))) in (a, b)


def test_sr_fp16_halfway_value_from_the_pages(golden):
    """2049 is exactly half-way between the fp16 values 2048 and 2050 ([CMU13]
    §7.3 ex. 5: 2049 rounds to 2048 in fp16): half of the draws go up."""
    rows = [r for r in golden("bf16_facts.txt") if r[0] == "fp16" and r[1] == "2049"]
    assert rows and float(rows[0][2]) == 2048.0
    outs = [oracle.sr_fp16_with_rand(2049.0, r) for r in range(65536)]
    assert outs.count(0x6801) == 32768 and outs.count(0x6800) == 32768  # 2050 and 2048


def test_sr_fp16_special_values_and_unbiasedness():
    assert oracle.sr_fp16_with_rand(float("nan"), 3) == 0x7E00
    assert oracle.sr_fp16_with_rand(float("inf"), 3) == 0x7C00
    assert oracle.sr_fp16_with_rand(float("-inf"), 3) == 0xFC00
    assert oracle.sr_fp16_with_rand(0.0, 3) == 0x0000 and oracle.sr_fp16_with_rand(-0.0, 3) == 0x8000
    for big in (65536.0, 1e6, 3e38):
        assert oracle.sr_fp16_with_rand(big, 0) == 0x7C00 and oracle.sr_fp16_with_rand(-big, 65535) == 0xFC00
    # unbiased over 10^5 seeds: 1 + 0.3 fp16 steps
    x = float(np.float32(1.0 + 0.3 * 2 ** -10))
    xs = np.full(100_000, x, np.float32)
    res = np.array([oracle.stochastic_round_fp16(xs[:1], 0, s)[0] for s in range(100_000)], np.uint16)
    v = res.view(np.float16).astype(np.float64)
    p = (x - 1.0) / 2 ** -10
    sigma = 2 ** -10 * math.sqrt(p * (1 - p) / v.size)
    assert abs(float(v.mean()) - x) < 4 * sigma


# --------------------------------------------------------------------------
# Accumulating into bf16 with stochastic rounding — llm.c ch. 04 §2.3: the
# same rounding writes the encoder's embedding gradients (a bf16 gradient
# plus an fp32 contribution, rounded back to bf16).
# --------------------------------------------------------------------------
def _bf16(vals):
    return W.bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)).copy()


def test_accumulate_sr_adding_zero_changes_nothing():
    rng = np.random.default_rng(5)
    acc = rng.integers(0, 1 << 16, 100_000, dtype=np.uint32).astype(np.uint16)
    keep = (acc & 0x7F80) != 0x7F80  # drop NaN and Inf patterns
    keep &= (acc & 0x7FFF) != 0      # and signed zeros (IEEE: -0 + +0 = +0)
    acc = acc[keep]
    out = acc.copy()
    oracle.accumulate_sr(out, np.zeros(acc.size, np.float32), 123, 9)
    assert np.array_equal(out, acc)
    z = np.array([0x8000, 0x0000], np.uint16)  # -0 + 0 = +0, +0 + 0 = +0 (round to nearest)
    oracle.accumulate_sr(z, np.zeros(2, np.float32), 0, 1)
    assert z.tolist() == [0x0000, 0x0000]


def test_accumulate_sr_exact_when_the_sum_is_representable():
    # integers up to 256 are exact in bf16 ([CMU13] §7.3 ex. 5: 257 is not)
    a = np.arange(0, 129, dtype=np.float32)
    d = np.arange(0, 129, dtype=np.float32)[::-1].copy()  # a + d = 128
    acc = _bf16(a)
    oracle.accumulate_sr(acc, d, 0, 77)
    assert np.array_equal(oracle.bf16_bits_to_f32(acc), np.full(a.size, 128.0, np.float32))
    acc = _bf16([1.0, -2.0, 0.5])
    # one bf16 step at each magnitude: 2^-7 at 1, 2^-6 at 2, 2^-8 at 0.5
    oracle.accumulate_sr(acc, np.array([2.0 ** -7, -2.0 ** -6, 2.0 ** -8], np.float32), 0, 3)
    assert np.array_equal(oracle.bf16_bits_to_f32(acc), np.array([1 + 2.0 ** -7, -2 - 2.0 ** -6, 0.5 + 2.0 ** -8],
                                                                   np.float32))


def test_accumulate_sr_is_unbiased_over_seeds():
    """1 + 0.3 ulp: over 10^5 seeds the mean result is 1 + 0.3 ulp within 4σ."""
    ulp = 2.0 ** -7
    seeds = 100_000
    res = np.empty(seeds, np.float32)
    for s in range(seeds):
        acc = np.array([0x3F80], np.uint16)
        oracle.accumulate_sr(acc, np.array([0.3 * ulp], np.float32), 42, s)
        res[s] = oracle.bf16_bits_to_f32(acc)[0]
    x = float(np.float32(1.0) + np.float32(0.3 * ulp))
    p = (x - 1.0) / ulp
    assert set(np.unique(res).tolist()) <= {1.0, 1.0 + ulp}
    sigma = ulp * math.sqrt(p * (1 - p) / seeds)
    assert abs(float(res.astype(np.float64).mean()) - x) < 4 * sigma


def test_accumulate_sr_keeps_small_contributions_and_shards():
    """1000 contributions of 1e-4·|a0| each (below half a bf16 step): the
    rounded accumulator follows the fp32 sum where round-to-nearest stalls;
    accumulating the buffer as two shards at their global offsets gives the
    same bits as the whole buffer."""
    n = 1 << 14
    a0 = W.sr_stress_weights(n, seed=7).numpy()
    delta = (np.float32(1e-4) * np.abs(a0)).astype(np.float32)
    fp32 = a0.copy()
    acc = W.bf16_bits(torch.from_numpy(a0).to(torch.bfloat16)).copy()
    halves = acc.copy()
    for t in range(1, 1001):
        fp32 = (fp32 + delta).astype(np.float32)
        oracle.accumulate_sr(acc, delta, 0, W.step_seed(t))
        h0, h1 = halves[: n // 2].copy(), halves[n // 2:].copy()
        oracle.accumulate_sr(h0, delta[: n // 2].copy(), 0, W.step_seed(t))
        oracle.accumulate_sr(h1, delta[n // 2:].copy(), n // 2, W.step_seed(t))
        halves = np.concatenate([h0, h1])
    assert np.array_equal(acc, halves)
    rel = float(np.mean(oracle.bf16_bits_to_f32(acc).astype(np.float64) / fp32 - 1.0))
    assert abs(rel) < 2e-3
    rne = torch.from_numpy(a0).to(torch.bfloat16)
    assert torch.equal((rne.float() + torch.from_numpy(delta)).to(torch.bfloat16), rne)  # RNE never moves


# --------------------------------------------------------------------------
# Bit-perfect resume — llm.c ch. 04 §5.2: bf16 weights are not checkpointed;
# they are rebuilt from the fp32 master with the saved rounding randomness.
# With draws keyed on the global index, the rebuild is SR(master, seed_t).
# --------------------------------------------------------------------------
def test_resume_rebuilds_bf16_bit_identically():
    name = "tiny"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    H = W.HYPER
    st = W.make_state(name)
    N = W.total(entries)

    def fresh():
        return dict(params=W.bf16_bits(st["params"]).copy(), master=st["master"].numpy().copy(),
                    m=np.zeros(N, np.float32), v=np.zeros(N, np.float32))

    def run(s, t0, t1):
        for t in range(t0, t1):
            g = W.bf16_bits(W.make_grads(name, t)).copy()
            _, _, scale = oracle.grad_norm(g, H["clip"])
            assert oracle.adamw_step(s["params"], g, s["master"], s["m"], s["v"], 0, tab, H["lr"], H["beta1"],
                                     H["beta2"], H["eps"], H["weight_decay"], float(scale), t, W.step_seed(t)) == 0

    a = fresh()
    run(a, 1, 7)
    b = fresh()
    run(b, 1, 4)
    ckpt = {k: b[k].copy() for k in ("master", "m", "v")}  # no bf16 weights saved
    b = dict(ckpt, params=oracle.stochastic_round(ckpt["master"], 0, W.step_seed(3)))
    run(b, 4, 7)
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


# --------------------------------------------------------------------------
# Outlier skip — llm.c ch. 04 §4: a window of 128 past grad norms, z-score of
# the new norm, skip the update when z is above a threshold.
# --------------------------------------------------------------------------
def test_outlier_zscore_matches_statistics_pstdev():
    import statistics
    rng = np.random.default_rng(7)
    o = oracle.OutlierCheck()
    hist = []
    for i in range(400):
        x = float(np.float32(1.0 + 0.1 * rng.standard_normal() + (5.0 if i % 97 == 96 else 0.0)))
        st, z, sc = o.check(x, 0.0, 0.5)
        assert st == 0 and sc == np.float32(0.5)  # threshold 0 never skips
        if len(hist) < 128:
            assert math.isnan(z)
        else:
            w = hist[-128:]
            ref = (x - statistics.fmean(w)) / statistics.pstdev(w)
            assert abs(z - ref) <= 1e-9 * max(1.0, abs(ref))
        hist.append(x)


def test_outlier_closed_form_and_skip():
    o = oracle.OutlierCheck()
    m, d = 2.0, 0.25  # window: 64 x (m - d) and 64 x (m + d): mean m, population std d
    for i in range(128):
        o.check(m - d if i % 2 else m + d, 3.0, 1.0)
    st, z, sc = o.check(m + 3 * d, 2.5, 0.75)
    assert z == 3.0 and st == 8 and math.isnan(sc)  # z > 2.5: skipped, scale poisoned
    o2 = oracle.OutlierCheck()
    for i in range(128):
        o2.check(m - d if i % 2 else m + d, 3.0, 1.0)
    st, z, sc = o2.check(m + 3 * d, 3.0, 0.75)
    assert z == 3.0 and st == 0 and sc == np.float32(0.75)  # not above the threshold: kept


def test_outlier_window_ignores_nonfinite_norms_and_slides():
    o = oracle.OutlierCheck()
    for i in range(127):
        o.check(1.0, 3.0, 1.0)
    for bad in (float("nan"), float("inf")):
        st, z, _ = o.check(bad, 3.0, 1.0)
        assert math.isnan(z) and o.state.count == 127
    o.check(1.0, 3.0, 1.0)
    assert o.state.count == 128
    st, z, _ = o.check(1.0, 3.0, 1.0)
    assert math.isnan(z)  # zero spread: 0 / 0
    st, z, _ = o.check(2.0, 3.0, 1.0)
    assert z == math.inf and st == 8
    # the window now holds 127 ones and one 2.0 (the oldest slot was replaced)
    assert sorted(o.state.window)[-1] == 2.0 and sum(o.state.window) == 129.0


# --------------------------------------------------------------------------
# The norm in pieces — llm.c ch. 04 §4: the global norm covers every gradient;
# under ZeRO-1 (§3.2, §4) each rank sums its own shard and the per-rank sums
# are combined; CMU 11-667 lecture 13 notes §5.2: ZeRO-1 matches data
# parallelism (max difference 0 on their example).
# --------------------------------------------------------------------------
def test_sumsq_continued_in_pieces_equals_one_pass():
    rng = np.random.default_rng(5)
    g = _bf16(rng.standard_normal(100_003) * 10.0 ** rng.uniform(-6, 3, 100_003))
    whole = oracle.sumsq(g)
    for cuts in ([0], [1], [50_000], [7, 64, 99_999], list(range(0, 100_003, 9_973))):
        s, a = 0.0, 0
        for c in cuts + [g.size]:
            s = oracle.sumsq_from(s, g[a:c])
            a = c
        assert s == whole, cuts  # bit for bit: the same additions in the same order
    # the running total is where the sum starts: 7 + 1000 * 1^2
    ones = np.full(1000, 0x3F80, np.uint16)
    assert oracle.sumsq_from(7.0, ones) == 1007.0
    assert oracle.sumsq_from(2.5, ones[:0]) == 2.5


def test_norm_from_parts_equals_whole_buffer_norm_on_exact_sums():
    # +-2^k gradients: every sum of squares is exact in fp64, so 8 shard sums
    # added in rank order give exactly the whole-buffer sum, norm and scale
    rng = np.random.default_rng(9)
    k = rng.integers(-8, 10, 8 * 4096)  # squares 2^-16 .. 2^18: 34 bits of range, 15 of count
    g = _bf16(np.where(rng.random(k.size) < 0.5, -1.0, 1.0) * np.exp2(k.astype(np.float64)))
    per = g.size // 8
    parts = [oracle.sumsq(g[r * per:(r + 1) * per]) for r in range(8)]
    s_w, n_w, sc_w = oracle.grad_norm(g, 1.0)
    s_p, n_p, sc_p = oracle.norm_from_parts(parts, 1.0)
    assert s_p == s_w == math.fsum(float(x) ** 2 for x in oracle.bf16_bits_to_f32(g).astype(np.float64))
    assert n_p == n_w and sc_p == sc_w
    # one part is oracle_grad_norm itself
    assert oracle.norm_from_parts([s_w], 1.0) == (s_w, n_w, sc_w)


def test_norm_from_parts_adds_in_rank_order_in_fp64():
    # left to right: (2^53 + 1) rounds back to 2^53 (ties to even), and again
    # for the next 1; another order would keep the two ones
    s, nrm, sc = oracle.norm_from_parts([2.0 ** 53, 1.0, 1.0], 1.0)
    assert s == 2.0 ** 53
    s, _, _ = oracle.norm_from_parts([1.0, 1.0, 2.0 ** 53], 1.0)
    assert s == 2.0 ** 53 + 2.0
    # closed cases of the clip rule: sum 4 -> norm 2 -> scale 1/2; sum 0.25 -> 1
    assert oracle.norm_from_parts([1.0, 3.0], 1.0)[1:] == (F32(2.0), F32(0.5))
    assert oracle.norm_from_parts([0.25, 0.0], 1.0)[1:] == (F32(0.5), F32(1.0))
    # a non-finite part refuses the step (NaN scale), like a non-finite norm
    assert math.isnan(oracle.norm_from_parts([1.0, math.inf], 1.0)[2])
    assert math.isnan(oracle.norm_from_parts([math.nan], 1.0)[2])


def test_norm_from_parts_within_rounding_of_the_exact_sum():
    rng = np.random.default_rng(12)
    g = _bf16(rng.standard_normal(80_000) * 1e-3)
    exact = math.fsum(float(x) ** 2 for x in oracle.bf16_bits_to_f32(g).astype(np.float64))
    for world in (2, 4, 8):
        per = g.size // world
        parts = [oracle.sumsq(g[r * per:(r + 1) * per]) for r in range(world)]
        s, _, _ = oracle.norm_from_parts(parts, 1.0)
        assert abs(s - exact) <= g.size * 2.0 ** -53 * exact


# --------------------------------------------------------------------------
# Learning-rate schedules — llm.c ch. 04 §4 names four (cosine, linear,
# constant, WSD) without formulas; the reading is in the oracle's comment.
# Pinned by closed forms at chosen steps and by the shapes' invariants.
# --------------------------------------------------------------------------
def _ulp_close(a, b, ulps=1):
    a, b = F32(a), F32(b)
    return abs(int(a.view(np.int32)) - int(b.view(np.int32))) <= ulps


LR = dict(warmup=10, total=110, lr_max=6e-4, lr_min=6e-5)


def _lr(kind, t, **kw):
    a = {**LR, **kw}
    return oracle.lr(kind, a["warmup"], a["total"], a["lr_max"], a["lr_min"], a.get("decay_frac", 0.2), t)


@pytest.mark.parametrize("kind", [oracle.LR_CONSTANT, oracle.LR_COSINE, oracle.LR_LINEAR, oracle.LR_WSD])
def test_lr_warmup_is_linear_and_reaches_the_peak(kind):
    hi = F32(LR["lr_max"])
    assert _lr(kind, 10) == hi  # the last warm-up step reaches lr_max exactly
    assert _lr(kind, 5) == F32(float(hi) / 2)  # half way: exactly half (a power-of-two ratio)
    assert _ulp_close(_lr(kind, 1), float(hi) / 10)
    ramp = [float(_lr(kind, t)) for t in range(1, 11)]
    assert all(b > a for a, b in zip(ramp, ramp[1:]))
    # no warm-up: the first step is already past it
    assert _lr(kind, 1, warmup=0) <= hi


def test_lr_constant_after_warmup():
    for t in (11, 50, 110, 10_000):
        assert _lr(oracle.LR_CONSTANT, t) == F32(LR["lr_max"])


def test_lr_cosine_closed_forms():
    hi, lo = float(F32(LR["lr_max"])), float(F32(LR["lr_min"]))
    assert _ulp_close(_lr(oracle.LR_COSINE, 60), (hi + lo) / 2)  # p = 1/2: cos = 0
    assert _ulp_close(_lr(oracle.LR_COSINE, 35), lo + (hi - lo) * (1 + math.sqrt(0.5)) / 2)  # p = 1/4
    assert _ulp_close(_lr(oracle.LR_COSINE, 85), lo + (hi - lo) * (1 - math.sqrt(0.5)) / 2)  # p = 3/4
    assert _lr(oracle.LR_COSINE, 110) == F32(lo)  # p = 1: cos = -1
    assert _lr(oracle.LR_COSINE, 500) == F32(lo)  # past the end: stays at lr_min
    # symmetric about the middle: lr(mid - d) + lr(mid + d) = hi + lo
    for d in (1, 7, 33, 49):
        s = float(_lr(oracle.LR_COSINE, 60 - d)) + float(_lr(oracle.LR_COSINE, 60 + d))
        assert abs(s - (hi + lo)) <= 2 * 2.0 ** -24 * hi
    tail = [float(_lr(oracle.LR_COSINE, t)) for t in range(10, 111)]
    assert all(b <= a for a, b in zip(tail, tail[1:]))


def test_lr_linear_closed_forms():
    hi, lo = float(F32(LR["lr_max"])), float(F32(LR["lr_min"]))
    assert _ulp_close(_lr(oracle.LR_LINEAR, 35), hi - (hi - lo) / 4)
    assert _ulp_close(_lr(oracle.LR_LINEAR, 60), (hi + lo) / 2)
    assert _lr(oracle.LR_LINEAR, 110) == F32(lo)
    assert _lr(oracle.LR_LINEAR, 111) == F32(lo)
    # equal steps down: constant differences
    d = [float(_lr(oracle.LR_LINEAR, t)) - float(_lr(oracle.LR_LINEAR, t + 1)) for t in range(11, 109)]
    assert max(d) - min(d) <= 4 * 2.0 ** -24 * hi


def test_lr_wsd_closed_forms():
    hi, lo = float(F32(LR["lr_max"])), float(F32(LR["lr_min"]))
    # stable at lr_max for the first 80 % of the post-warm-up steps
    for t in range(11, 91):
        assert _lr(oracle.LR_WSD, t) == F32(hi), t
    assert _ulp_close(_lr(oracle.LR_WSD, 100), (hi + lo) / 2)  # half way through the decay
    assert _ulp_close(_lr(oracle.LR_WSD, 95), hi - (hi - lo) / 4)
    assert _lr(oracle.LR_WSD, 110) == F32(lo)
    # decay over the whole run (f = 1) is the linear schedule
    for t in range(11, 111):
        assert _ulp_close(_lr(oracle.LR_WSD, t, decay_frac=1.0), _lr(oracle.LR_LINEAR, t)), t


def test_lr_rejects_invalid_arguments():
    assert math.isnan(_lr(oracle.LR_COSINE, 0))
    assert math.isnan(_lr(oracle.LR_COSINE, 5, total=10))  # total <= warmup for a decaying kind
    assert math.isnan(_lr(oracle.LR_WSD, 20, decay_frac=0.0))
    assert math.isnan(_lr(oracle.LR_WSD, 20, decay_frac=1.5))
    assert math.isnan(oracle.lr(4, 0, 10, 1e-3, 0.0, 0.5, 3))
    assert math.isnan(oracle.lr(oracle.LR_LINEAR, -1, 10, 1e-3, 0.0, 0.5, 3))
    assert _lr(oracle.LR_CONSTANT, 5, total=0) == F32(LR["lr_max"] / 2)  # constant ignores total
