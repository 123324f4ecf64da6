"""A seeded random sweep of the CUDA paths against the oracle, bit for bit:
the update over a range (random sizes, global offsets up to 5·2^32, tables
of 1 to 2^20-element tensors, unaligned buffers and vector-aligned buffers
that start mid-line, both variants, betas, eps, lr, decay and step counts),
the whole-step call (cluster kernel below 32,768 params, the general path
above), the standalone rounding to bf16 and to fp16, the
accumulate-and-round, on values from 1e-40 to 1e38; the ZeRO-1 norm over
random shard counts; and host-to-device copies by the SMs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp

CASES = 280


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _bf16(x):
    return W.bf16_bits(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)).copy()


def _dev16(a, pad):
    b = torch.empty(a.size + pad, dtype=torch.int16, device="cuda")
    out = b[pad:]
    out.copy_(torch.from_numpy(a.view(np.int16)))
    return out.view(torch.bfloat16)


def _dev32(a, pad):
    b = torch.empty(a.size + pad, dtype=torch.float32, device="cuda")
    out = b[pad:]
    out.copy_(torch.from_numpy(a))
    return out


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _bits(t):
    return t.contiguous().cpu().numpy().view(np.uint32)


def _update_case(rng, whole):
    n = int(rng.choice([1, 3, 8, 2047, 2048, 2049, 4100, 30000, 32768, 32769, 70001, 300007]))
    goff = 0 if whole else int(rng.choice([0, 4, 17, (1 << 32) - int(rng.integers(1, 3000)), 5 << 32]))
    pad = int(rng.choice([0, 0, 0, 1, 2, 4, 12, 28]))  # 4, 12, 28: vector path, tiles after a peeled head
    seed = int(rng.integers(0, 1 << 32))
    gen = torch.Generator().manual_seed(int(rng.integers(0, 1 << 30)))
    tmax = int(rng.choice([1, 7, 100, 5000, 1 << 20]))
    tail = W.random_table(n, gen, 1, tmax)
    tab = ([(0, goff, int(rng.integers(0, 2)))] if goff else []) + [(o + goff, s, d) for o, s, d in tail]
    master = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 1)).astype(np.float32)
    params, grads = _bf16(master), _bf16(rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 0))
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.random(n) * 1e-5).astype(np.float32)
    with_master = bool(rng.integers(0, 2))
    hp = dict(lr=float(10.0 ** rng.uniform(-5, -1)), beta1=float(rng.choice([0.0, 0.9, 0.95])),
              beta2=float(rng.choice([0.95, 0.999, 0.5])), eps=float(10.0 ** rng.uniform(-10, -3)),
              weight_decay=float(rng.choice([0.0, 0.1, 0.5])))
    t = int(rng.integers(1, 5000))
    host = dict(params=params.copy(), master=master.copy() if with_master else None, m=m.copy(), v=v.copy())
    d = dict(params=_dev16(params, pad), m=_dev32(m, pad), v=_dev32(v, pad),
             master=_dev32(master, pad) if with_master else None)
    dg = _dev16(grads, pad)
    what = f"n={n} goff={goff} pad={pad} master={with_master} tensors={len(tab)} t={t}"
    if whole:
        opt = mp.Optimizer(tab, clip=1.0, **hp)
        opt.step(d["params"], dg, d["master"], d["m"], d["v"], t, seed)
        torch.cuda.synchronize()
        scale = float(opt.d_scale.item())
        _, nrm, _ = oracle.grad_norm(grads, 1.0)
        assert abs(float(opt.d_norm.item()) - float(nrm)) <= 1e-6 * float(nrm), what
        assert scale == oracle.clip_scale(float(opt.d_norm.item()), 1.0), what
    else:
        scale = float(np.float32(rng.uniform(0.01, 1.0)))
        mp.mp_adamw_step(d["params"], dg, d["master"], d["m"], d["v"], mp.TensorTable(tab), **hp,
                         d_grad_scale=torch.tensor([scale], device="cuda"), t=t, seed=seed, global_offset=goff, n=n)
    assert oracle.adamw_step(host["params"], grads, host["master"], host["m"], host["v"], goff, tab, hp["lr"],
                             hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], scale, t, seed) == 0
    assert np.array_equal(_u16(d["params"]), host["params"]), what
    for k in ("m", "v") + (("master",) if with_master else ()):
        assert np.array_equal(_bits(d[k]), host[k].view(np.uint32)), (k, what)


def _zero1_norm_case(rng):
    """Per-shard sums of squares (mp_grad_sumsq) combined in rank order
    (mp_clip_scale_from_sumsq): the same bits as the oracle's ZeRO-1 norm of
    those sums, and each sum within 1e-6 of the oracle's own."""
    world = int(rng.choice([1, 2, 3, 8, 16]))
    per = int(rng.choice([1, 5, 2048, 4099, 100_003]))
    pad = int(rng.choice([0, 1, 4]))
    g = _bf16(rng.standard_normal(world * per) * 10.0 ** rng.uniform(-5, 1))
    dg = _dev16(g, pad)
    ws = torch.empty(max(8, mp.mp_grad_norm_workspace_bytes(per)), dtype=torch.uint8, device="cuda")
    parts = torch.empty(world, dtype=torch.float64, device="cuda")
    for r in range(world):
        mp.mp_grad_sumsq(dg[r * per:(r + 1) * per], ws, parts[r:r + 1])
    clip = float(rng.choice([0.5, 1.0, 100.0]))
    d_norm, d_scale = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    total = torch.empty(1, dtype=torch.float64, device="cuda")
    mp.mp_clip_scale_from_sumsq(parts, clip, d_norm, d_scale, total)
    torch.cuda.synchronize()
    gp = parts.cpu().numpy()
    s, nrm, sc = oracle.norm_from_parts(gp, clip)
    assert total.item() == s and np.float32(d_norm.item()) == nrm and np.float32(d_scale.item()) == sc, (world, per)
    for r in range(world):
        ref = oracle.sumsq(g[r * per:(r + 1) * per])
        assert abs(gp[r] - ref) <= 1e-6 * ref, (world, per, r)


def _copy_case(rng):
    nbytes = int(rng.choice([1, 15, 16, 17, 4096, 100_003, 1 << 22]))
    so, do = int(rng.choice([0, 1, 8, 16])), int(rng.choice([0, 3, 16]))
    host = torch.empty(nbytes + so, dtype=torch.uint8, pin_memory=True)
    host.copy_(torch.from_numpy(rng.integers(0, 256, nbytes + so, dtype=np.uint8)))
    dev = torch.zeros(nbytes + do, dtype=torch.uint8, device="cuda")
    mp.mp_copy_from_host(dev[do:], host[so:], nbytes, blocks_per_sm=int(rng.choice([1, 2, 4])))
    torch.cuda.synchronize()
    assert torch.equal(dev[do:].cpu(), host[so:]), (nbytes, so, do)


def test_random_sweep_against_the_oracle():
    rng = np.random.default_rng(20261202)
    counts = dict(step=0, whole=0, sr=0, acc=0, sr16=0, zero1=0, copy=0)
    for _ in range(CASES):
        kind = str(rng.choice(list(counts)))
        counts[kind] += 1
        if kind in ("step", "whole"):
            _update_case(rng, kind == "whole")
            continue
        if kind == "zero1":
            _zero1_norm_case(rng)
            continue
        if kind == "copy":
            _copy_case(rng)
            continue
        n = int(rng.choice([1, 7, 2049, 30001, 300007]))
        goff = int(rng.choice([0, 17, (1 << 32) - int(rng.integers(1, 3000))]))
        pad, pad_in, seed = int(rng.choice([0, 1])), int(rng.choice([0, 1])), int(rng.integers(0, 1 << 32))
        with np.errstate(over="ignore"):
            x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-40, 38, n)).astype(np.float32)
        if kind == "sr":
            out = _dev16(np.zeros(n, np.uint16), pad)
            mp.mp_stochastic_round(out, _dev32(x, pad_in), seed, global_offset=goff)
            assert np.array_equal(_u16(out), oracle.stochastic_round(x, goff, seed)), (n, goff, pad)
        elif kind == "sr16":
            out = _dev16(np.zeros(n, np.uint16), pad)
            mp.mp_stochastic_round_fp16(out.view(torch.float16), _dev32(x, pad_in), seed, global_offset=goff)
            assert np.array_equal(_u16(out), oracle.stochastic_round_fp16(x, goff, seed)), (n, goff, pad)
        else:
            acc0 = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
            acc = _dev16(acc0, pad)
            mp.mp_accumulate_sr(acc, _dev32(x, pad_in), seed, global_offset=goff)
            ref = acc0.copy()
            oracle.accumulate_sr(ref, x, goff, seed)
            assert np.array_equal(_u16(acc), ref), (n, goff, pad)
    assert min(counts.values()) >= 15, counts
