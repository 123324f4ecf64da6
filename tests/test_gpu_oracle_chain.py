"""The oracle's own chain against the GPU, at the bars the method sets.

In these tests the oracle computes every step from its own results: its fp64
norm over all gradients, its clip scale, its bias corrections and learning
rate, its update of its own state. Nothing it uses comes from the GPU except
the seeded inputs both sides start from. Each step the GPU state is compared
with the oracle's at the bars of tests/helpers.py: fp32 master, m and v
within 1e-6 relative; at most 1e-6 of the bf16 weights different, by one bf16
step at most; the norm within 1e-6 of the oracle's fp64 value. Whether the two
clip scales came out bit-equal is recorded; while they are, the states must
also be bit-identical (the kernels follow the oracle's operation order).

Parameter sets and step counts: GPT-2 124M, 10 steps, with and without fp32
master weights; Llama-3-8B, 5 steps, on windows (the oracle's norm still
covers all 8.03B gradients); the tiny set, 16 steps under each learning-rate
schedule; the ZeRO-1 norm over 8 shards and a ZeRO-1 step over one NCCL rank.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bf16_close, assert_bit_equal, assert_f32_close, rel_err, to_np_f32, to_np_u16

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp
else:
    mp = None

DEV = "cuda"
H = W.HYPER


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _host(st):
    return dict(params=to_np_u16(st["params"]).copy(), m=to_np_f32(st["m"]).copy(), v=to_np_f32(st["v"]).copy(),
                master=to_np_f32(st["master"]).copy() if "master" in st else None)


def _compare(gpu, host, name, exact):
    assert_bf16_close(to_np_u16(gpu["params"]), host["params"], f"{name} params")
    for k in ("master", "m", "v"):
        if host.get(k) is not None:
            assert_f32_close(to_np_f32(gpu[k]), host[k], f"{name} {k}")
    if exact:
        assert_bit_equal(to_np_u16(gpu["params"]), host["params"], f"{name} params (bitwise)")
        for k in ("master", "m", "v"):
            if host.get(k) is not None:
                assert_bit_equal(to_np_f32(gpu[k]), host[k], f"{name} {k} (bitwise)")


def _oracle_norm_chunked(g_dev, chunk=1 << 27):
    """The oracle's norm over a device buffer: one fp64 sum in index order,
    continued across host-sized pieces (bit-identical to one pass)."""
    s = 0.0
    n = g_dev.numel()
    for a in range(0, n, chunk):
        s = oracle.sumsq_from(s, to_np_u16(g_dev[a:min(n, a + chunk)]))
    return oracle.norm_from_parts([s], H["clip"])


@pytest.mark.parametrize("with_master", [True, False])
def test_gpt2_124m_ten_steps_oracle_chain(with_master, record_property):
    name = "gpt2_124m"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    st = W.make_state(name, device=DEV, with_master=with_master)
    host = _host(st)
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])
    scales_equal = []
    for t in range(1, 11):
        g = W.make_grads(name, t, device=DEV)
        opt.step(st["params"], g, st.get("master"), st["m"], st["v"], t, W.step_seed(t))
        gb = to_np_u16(g)
        s_o, nrm_o, sc_o = oracle.grad_norm(gb, H["clip"])
        assert oracle.adamw_step(host["params"], gb, host["master"], host["m"], host["v"], 0, tab, H["lr"],
                                 H["beta1"], H["beta2"], H["eps"], H["weight_decay"], float(sc_o), t,
                                 W.step_seed(t)) == 0
        opt.check_status()
        assert rel_err(float(opt.d_norm.item()), float(nrm_o)) <= 1e-6
        scales_equal.append(float(opt.d_scale.item()) == float(sc_o))
        _compare(st, host, f"124M step {t}", exact=all(scales_equal))
    record_property("clip_scales_bit_equal", f"{sum(scales_equal)}/{len(scales_equal)}")
    print(f"\nGPT-2 124M, 10 steps (master={with_master}): GPU and oracle clip scales bit-equal on "
          f"{sum(scales_equal)} of {len(scales_equal)} steps")


@pytest.mark.slow
def test_llama3_8b_five_steps_oracle_chain(record_property):
    name = "llama3_8b"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    N = W.total(entries)
    st = W.make_state(name, device=DEV)
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])
    windows = [(0, 1 << 16), ((1 << 32) - 50000, 100000), (N // 3, 1 << 16), (N - 100003, 100003)]
    host = [{k: (to_np_u16(st[k][a:a + n]) if k == "params" else to_np_f32(st[k][a:a + n])).copy() for k in st}
            for a, n in windows]
    g = torch.empty(N, dtype=torch.bfloat16, device=DEV)
    scales_equal = []
    for t in range(1, 6):
        W.make_grads(name, t, device=DEV, out=g)
        opt.step(st["params"], g, st["master"], st["m"], st["v"], t, W.step_seed(t))
        _, nrm_o, sc_o = _oracle_norm_chunked(g)
        opt.check_status()
        assert rel_err(float(opt.d_norm.item()), float(nrm_o)) <= 1e-6
        assert float(sc_o) < 1.0  # clipping fires on this set
        scales_equal.append(float(opt.d_scale.item()) == float(sc_o))
        for (a, n), hw in zip(windows, host):
            assert oracle.adamw_step(hw["params"], to_np_u16(g[a:a + n]), hw["master"], hw["m"], hw["v"], a, tab,
                                     H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], float(sc_o), t,
                                     W.step_seed(t)) == 0
            _compare({k: st[k][a:a + n] for k in st}, hw, f"8B step {t} window {a}", exact=all(scales_equal))
    record_property("clip_scales_bit_equal", f"{sum(scales_equal)}/{len(scales_equal)}")
    print(f"\nLlama-3-8B, 5 steps: GPU and oracle clip scales bit-equal on {sum(scales_equal)} of 5 steps")


@pytest.mark.parametrize("kind", ["constant", "cosine", "linear", "wsd"])
def test_tiny_sixteen_steps_under_each_lr_schedule(kind):
    """16 steps of the tiny set; the library's schedule sets each step's
    learning rate, the oracle computes its own from the same definition."""
    name = "tiny"
    tab = W.table(W.layout(W.specs_for(name)))
    sched = dict(lr_max=2e-3, lr_min=2e-4, warmup=4, total=14, decay_frac=0.5)
    schedule = mp.LRSchedule(kind, **sched)
    st = W.make_state(name, device=DEV)
    host = _host(st)
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"], schedule=schedule)
    lrs, scales_equal = [], []
    for t in range(1, 17):
        g = W.make_grads(name, t, device=DEV)
        opt.step(st["params"], g, st["master"], st["m"], st["v"], t, W.step_seed(t))
        lr_o = oracle.lr(mp.LR_KINDS[kind], sched["warmup"], sched["total"], sched["lr_max"], sched["lr_min"],
                         sched["decay_frac"], t)
        assert schedule.lr(t) == float(lr_o), t
        lrs.append(float(lr_o))
        gb = to_np_u16(g)
        _, _, sc_o = oracle.grad_norm(gb, H["clip"])
        assert oracle.adamw_step(host["params"], gb, host["master"], host["m"], host["v"], 0, tab, float(lr_o),
                                 H["beta1"], H["beta2"], H["eps"], H["weight_decay"], float(sc_o), t,
                                 W.step_seed(t)) == 0
        scales_equal.append(float(opt.d_scale.item()) == float(sc_o))
        _compare(st, host, f"tiny {kind} step {t}", exact=all(scales_equal))
    assert lrs[3] == np.float32(2e-3)  # warm-up ends at the peak
    if kind != "constant":
        assert lrs[-1] == np.float32(2e-4)  # past the end: the floor


def test_split_norm_equals_whole_norm_and_oracle_parts():
    """mp_grad_sumsq gives mp_grad_norm's sum bit for bit; the scale from one
    sum is mp_grad_norm's; from 8 per-shard sums it is the oracle's ZeRO-1
    norm of those same sums (the same left-to-right fp64 additions)."""
    n = 8_000_000
    gen = torch.Generator(device=DEV).manual_seed(3)
    g = (torch.randn(n, generator=gen, device=DEV) * 1e-2).to(torch.bfloat16)
    ws = torch.empty(max(8, mp.mp_grad_norm_workspace_bytes(n)), dtype=torch.uint8, device=DEV)
    f = lambda: torch.full((1,), -1.0, dtype=torch.float32, device=DEV)  # noqa: E731
    d_norm, d_scale, d_sumsq = f(), f(), torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
    mp.mp_grad_norm(g, 1.0, ws, d_norm, d_scale, d_sumsq)
    s1 = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
    mp.mp_grad_sumsq(g, ws, s1)
    n1, sc1, tot1 = f(), f(), torch.empty(1, dtype=torch.float64, device=DEV)
    mp.mp_clip_scale_from_sumsq(s1, 1.0, n1, sc1, tot1)
    torch.cuda.synchronize()
    assert s1.item() == d_sumsq.item() == tot1.item()
    assert (n1.item(), sc1.item()) == (d_norm.item(), d_scale.item())
    # 8 shards (ragged alignment: every shard starts 8-element aligned here)
    per = n // 8
    parts = torch.empty(8, dtype=torch.float64, device=DEV)
    for r in range(8):
        mp.mp_grad_sumsq(g[r * per:(r + 1) * per], ws, parts[r:r + 1])
    n8, sc8, tot8 = f(), f(), torch.empty(1, dtype=torch.float64, device=DEV)
    mp.mp_clip_scale_from_sumsq(parts, 1.0, n8, sc8, tot8)
    torch.cuda.synchronize()
    gpu_parts = parts.cpu().numpy()
    s_o, nrm_o, sc_o = oracle.norm_from_parts(gpu_parts, 1.0)
    assert tot8.item() == s_o and np.float32(n8.item()) == nrm_o and np.float32(sc8.item()) == sc_o
    # and each GPU part meets the norm's bar against the oracle's own sums
    gb = to_np_u16(g)
    for r in range(8):
        ref = oracle.sumsq(gb[r * per:(r + 1) * per])
        assert abs(gpu_parts[r] - ref) <= 1e-6 * ref


def test_zero1_emulated_eight_ranks_oracle_chain(record_property):
    """GPT-2 124M as 8 ZeRO-1 shards on one GPU, 3 steps: each virtual rank's
    sum of squares of its shard, the scale from the 8 sums in rank order,
    then the 8 shard updates. The oracle does the same from its own sums.
    (On one GPU every rank's averaged gradients are the step's gradients.)"""
    name = "gpt2_124m"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    N = W.total(entries)
    world = 8
    per = N // world
    st = W.make_state(name, device=DEV)
    host = _host(st)
    table = mp.TensorTable(tab)
    ws = torch.empty(max(8, mp.mp_grad_norm_workspace_bytes(per)), dtype=torch.uint8, device=DEV)
    parts = torch.empty(world, dtype=torch.float64, device=DEV)
    d_norm = torch.empty(1, dtype=torch.float32, device=DEV)
    d_scale = torch.empty(1, dtype=torch.float32, device=DEV)
    d_status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    scales_equal = []
    for t in range(1, 4):
        g = W.make_grads(name, t, device=DEV)
        for r in range(world):
            mp.mp_grad_sumsq(g[r * per:(r + 1) * per], ws, parts[r:r + 1])
        mp.mp_clip_scale_from_sumsq(parts, H["clip"], d_norm, d_scale)
        for r in range(world):
            sl = slice(r * per, (r + 1) * per)
            mp.mp_adamw_step(st["params"][sl], g[sl], st["master"][sl], st["m"][sl], st["v"][sl], table,
                             d_grad_scale=d_scale, t=t, seed=W.step_seed(t), global_offset=r * per, n=per,
                             d_status=d_status, **kw)
        gb = to_np_u16(g)
        o_parts = [oracle.sumsq(gb[r * per:(r + 1) * per]) for r in range(world)]
        _, nrm_o, sc_o = oracle.norm_from_parts(o_parts, H["clip"])
        for r in range(world):
            sl = slice(r * per, (r + 1) * per)
            assert oracle.adamw_step(host["params"][sl], gb[sl], host["master"][sl], host["m"][sl], host["v"][sl],
                                     r * per, tab, H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"],
                                     float(sc_o), t, W.step_seed(t)) == 0
        assert int(d_status.item()) == 0
        gpu_parts = parts.cpu().numpy()
        assert all(abs(a - b) <= 1e-6 * b for a, b in zip(gpu_parts, o_parts))
        assert rel_err(float(d_norm.item()), float(nrm_o)) <= 1e-6
        scales_equal.append(float(d_scale.item()) == float(sc_o))
        _compare(st, host, f"ZeRO-1 x8 step {t}", exact=all(scales_equal))
    record_property("clip_scales_bit_equal", f"{sum(scales_equal)}/3")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_zero1_one_nccl_rank_equals_single_gpu_step():
    """The ZeRO-1 driver with real NCCL collectives on a one-rank group: the
    reduce-scatter and all-gathers are copies, and 3 steps must equal the
    single-GPU whole-step call bit for bit (GPT-2 124M)."""
    import torch.distributed as dist
    from mixed_precision_adamw_gb300.zero1 import Zero1Optimizer
    if not dist.is_nccl_available():
        pytest.skip("torch built without NCCL")
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        name = "gpt2_124m"
        tab = W.table(W.layout(W.specs_for(name)))
        ref = W.make_state(name, device=DEV)
        z_params = ref["params"].clone()
        zopt = Zero1Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                              weight_decay=H["weight_decay"], clip=H["clip"], device=DEV)
        zst = zopt.make_shard_state(ref["master"])
        opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                           weight_decay=H["weight_decay"], clip=H["clip"])
        for t in range(1, 4):
            g = W.make_grads(name, t, device=DEV)
            zopt.step(z_params, g, zst["master"], zst["m"], zst["v"], t, W.step_seed(t))
            opt.step(ref["params"], g, ref["master"], ref["m"], ref["v"], t, W.step_seed(t))
            torch.cuda.synchronize()
            assert zopt.take_status() == 0
            assert torch.equal(zopt.d_scale, opt.d_scale) and torch.equal(zopt.d_norm, opt.d_norm)
            assert torch.equal(z_params.view(torch.int16), ref["params"].view(torch.int16))
            for k in ("master", "m", "v"):
                assert torch.equal(zst[k].view(torch.int32), ref[k].view(torch.int32)), k
    finally:
        dist.destroy_process_group()


def test_degenerate_norm_halves_and_empty_update():
    """Empty and degenerate inputs of the ZeRO-1 norm's halves and the update:
    an empty shard sums to 0; all-zero sums give norm 0 and scale 1; a
    non-finite sum gives a NaN scale; an empty update writes nothing. The
    oracle's ZeRO-1 norm agrees on each."""
    ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    g = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    parts = torch.full((3,), -1.0, dtype=torch.float64, device=DEV)
    mp.mp_grad_sumsq(g, ws, parts[0:1], n=0)
    parts[1:] = 0.0
    d_norm, d_scale = torch.full((1,), -1.0, device=DEV), torch.full((1,), -1.0, device=DEV)
    mp.mp_clip_scale_from_sumsq(parts, 1.0, d_norm, d_scale)
    torch.cuda.synchronize()
    assert parts[0].item() == 0.0
    _, nrm, sc = oracle.norm_from_parts([0.0, 0.0, 0.0], 1.0)
    assert (np.float32(d_norm.item()), np.float32(d_scale.item())) == (nrm, sc) == (0.0, 1.0)
    for bad in (float("inf"), float("nan")):
        parts[2] = bad
        mp.mp_clip_scale_from_sumsq(parts, 1.0, d_norm, d_scale)
        torch.cuda.synchronize()
        assert np.isnan(d_scale.item()) and np.isnan(oracle.norm_from_parts(parts.cpu().numpy(), 1.0)[2])
    # an empty update over a non-empty table: nothing written, no device error
    st = {k: torch.full((8,), 3.0, dtype=torch.float32, device=DEV) for k in ("master", "m", "v")}
    params = torch.full((8,), 3.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    mp.mp_adamw_step(params, params.clone(), st["master"], st["m"], st["v"], mp.TensorTable([(0, 8, 1)]), lr=1e-3,
                     beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, d_grad_scale=None, t=1, seed=1,
                     global_offset=3, n=0, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bool((params.float() == 3.0).all())
    assert all(bool((x == 3.0).all()) for x in st.values())
