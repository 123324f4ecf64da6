"""Replayable steps: mp_optimizer_step_graph keeps the step count, rounding
seed and learning rate in device memory, so one captured CUDA graph of the
call serves every later step.

A run of graph replays must equal, bit for bit, the same run of ordinary
mp_optimizer_step calls with t = 1, 2, ... and seed = seed_base + t (the
train loop of llm.c ch. 04 §4), and on the tiny set also the oracle step by
step. The device refuses a step whose t it cannot look up (negative count,
or t beyond a bias table that has not reached (1, 1))."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bit_equal, rel_err, to_np_f32, to_np_u16

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp

H = W.HYPER


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _opt(tab, outlier_z=None, **over):
    h = dict(H)
    h.update(over)
    return mp.Optimizer(tab, lr=h["lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["eps"],
                        weight_decay=h["weight_decay"], clip=h["clip"], outlier_z=outlier_z)


def _clone(st, pad=0):
    """Copies of the state, each starting `pad` elements into its buffer
    (pad 1: not vector-aligned, so the scalar kernels run)."""
    out = {}
    for k, x in st.items():
        if x is None:
            out[k] = None
            continue
        buf = torch.empty(x.numel() + pad, dtype=x.dtype, device=x.device)
        out[k] = buf[pad:]
        out[k].copy_(x)
    return out


def _assert_same(a, b, what):
    for k in a:
        if a[k] is None:
            continue
        if a[k].dtype == torch.bfloat16:
            assert_bit_equal(to_np_u16(a[k]), to_np_u16(b[k]), f"{what} {k}")
        else:
            assert_bit_equal(to_np_f32(a[k]), to_np_f32(b[k]), f"{what} {k}")


def _random_state(n, seed, with_master, pad=0, tmax=5000):
    gen = torch.Generator().manual_seed(seed)
    tab = W.random_table(n, gen, 1, tmax)
    master = torch.randn(n, generator=gen) * 0.05

    def dev(x, dtype):
        buf = torch.empty(n + pad, dtype=dtype, device="cuda")
        out = buf[pad:]
        out.copy_(x.to(dtype))
        return out
    st = dict(params=dev(master, torch.bfloat16), master=dev(master, torch.float32) if with_master else None,
              m=dev(torch.zeros(n), torch.float32), v=dev(torch.zeros(n), torch.float32))
    grads = [(torch.randn(n, generator=gen) * 1e-2 * (1 + k % 3)).to(torch.bfloat16) for k in range(6)]
    return tab, st, grads


def _eager(tab, st, grads_seq, seed_base, t0=0, outlier_z=None, lr_at=None):
    """Ordinary steps t0+1, t0+2, ...; returns the norm of each step."""
    opt = _opt(tab, outlier_z)
    dg = torch.empty(st["m"].numel(), dtype=torch.bfloat16, device="cuda")
    norms, statuses = [], []
    for k, g in enumerate(grads_seq):
        t = t0 + k + 1
        dg.copy_(g)
        if lr_at is not None:
            opt.hyper_struct.lr = lr_at(t)
        opt.step(st["params"], dg, st["master"], st["m"], st["v"], t, (seed_base + t) & 0xFFFFFFFF)
        norms.append(opt.d_norm.clone())
        statuses.append(opt.take_status())
    return [float(x.item()) for x in norms], statuses


def _graph_run(tab, st, grads_seq, seed_base, t0=0, outlier_z=None, lr_at=None):
    """The same steps: the first one as a plain call (it also warms the
    library up), the rest as replays of one captured graph."""
    opt = _opt(tab, outlier_z)
    opt.init_device_clock(t=t0, seed_base=seed_base, lr=lr_at(t0 + 1) if lr_at else None)
    dg = torch.empty(st["m"].numel(), dtype=torch.bfloat16, device="cuda")
    norms, statuses = [], []

    def after(t):
        norms.append(opt.d_norm.clone())
        statuses.append(opt.take_status())
        if lr_at is not None:
            opt.set_lr(lr_at(t + 1))

    dg.copy_(grads_seq[0])
    opt.step_graph(st["params"], dg, st["master"], st["m"], st["v"])
    after(t0 + 1)
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        opt.step_graph(st["params"], dg, st["master"], st["m"], st["v"])
    for k, g in enumerate(grads_seq[1:], start=2):
        dg.copy_(g)
        graph.replay()
        after(t0 + k)
    torch.cuda.synchronize()
    return [float(x.item()) for x in norms], statuses, opt


@pytest.mark.parametrize("n,with_master,pad,tmax", [
    (3_000_017, True, 0, 200_000), (3_000_017, False, 0, 200_000), (1_234_567, True, 1, 5_000),
    (2_500_003, True, 0, 600)])  # the last: > 1024 decay segments, several launches per step
def test_graph_replays_equal_ordinary_steps(n, with_master, pad, tmax):
    tab, st, grads = _random_state(n, n + pad, with_master, pad, tmax)
    seed_base = 4321
    a, b = _clone(st, pad), _clone(st, pad)
    norms_e, stat_e = _eager(tab, a, grads, seed_base)
    norms_g, stat_g, opt = _graph_run(tab, b, grads, seed_base)
    assert norms_e == norms_g and stat_e == stat_g == [0] * len(grads)
    _assert_same(a, b, f"graph n={n}")
    clock = opt.device_clock()
    T = len(grads)
    assert clock["t"] == T and clock["seed"] == seed_base + T
    bc1, bc2 = oracle.bias_corrections(H["beta1"], H["beta2"], T)
    assert clock["bc1"] == float(bc1) and clock["bc2"] == float(bc2)


def test_graph_tiny_sixteen_steps_against_the_oracle():
    name = "tiny"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    st = W.make_state(name)
    host = dict(params=W.bf16_bits(st["params"]).copy(), master=st["master"].numpy().copy(),
                m=st["m"].numpy().copy(), v=st["v"].numpy().copy())
    dst = {k: x.cuda() for k, x in st.items()}
    grads = [W.make_grads(name, t) for t in range(1, 17)]
    norms, statuses, _ = _graph_run(tab, dst, grads, W.BASE_SEED)
    # oracle afterwards, step by step, then the final states must agree bitwise
    for t, g in enumerate(grads, start=1):
        gb = W.bf16_bits(g).copy()
        _, nrm, sc = oracle.grad_norm(gb, H["clip"])
        assert rel_err(norms[t - 1], float(nrm)) <= 1e-6
        scale = oracle.clip_scale(norms[t - 1], H["clip"])
        assert oracle.adamw_step(host["params"], gb, host["master"], host["m"], host["v"], 0, tab, H["lr"],
                                 H["beta1"], H["beta2"], H["eps"], H["weight_decay"], scale, t,
                                 W.step_seed(t)) == 0
    assert statuses == [0] * 16
    assert_bit_equal(to_np_u16(dst["params"]), host["params"], "tiny params")
    for k in ("master", "m", "v"):
        assert_bit_equal(to_np_f32(dst[k]), host[k], f"tiny {k}")


def test_graph_resume_and_learning_rate_schedule():
    tab, st, grads = _random_state(777_777, 5, True)
    lr_at = lambda t: 1e-3 * (0.5 ** (t // 2))  # noqa: E731  (a step schedule)
    a, b = _clone(st), _clone(st)
    norms_e, _ = _eager(tab, a, grads, 99, t0=41, lr_at=lr_at)
    norms_g, _, opt = _graph_run(tab, b, grads, 99, t0=41, lr_at=lr_at)
    assert norms_e == norms_g
    _assert_same(a, b, "resume at t=42 with an lr schedule")
    assert opt.device_clock()["t"] == 41 + len(grads)


def test_graph_with_outlier_check_skips_like_ordinary_steps():
    name = "tiny"
    tab = W.table(W.layout(W.specs_for(name)))
    st = {k: x.cuda() for k, x in W.make_state(name).items()}
    grads = [W.make_grads(name, t) for t in range(1, 134)]
    grads[130] = (grads[130].float() * 100.0).to(torch.bfloat16)  # step 131: a norm spike
    a, b = _clone(st), _clone(st)
    _, stat_e = _eager(tab, a, grads, W.BASE_SEED, outlier_z=5.0)
    _, stat_g, opt = _graph_run(tab, b, grads, W.BASE_SEED, outlier_z=5.0)
    assert stat_e == stat_g and stat_g[130] == mp.MP_SKIPPED_OUTLIER and stat_g.count(0) == 132
    _assert_same(a, b, "outlier run")
    assert opt.device_clock()["t"] == 133  # the skipped step still counts


def test_graph_host_gradients():
    tab, st, grads = _random_state(1_000_003, 11, True)
    n = st["m"].numel()
    a, b = _clone(st), _clone(st)
    norms_e, _ = _eager(tab, a, grads, 7)
    opt = _opt(tab)
    opt.init_device_clock(t=0, seed_base=7)
    host_g = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    host_norm = torch.empty(1, dtype=torch.float32, pin_memory=True)
    dg = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    host_g.copy_(grads[0])
    opt.step_graph(b["params"], dg, b["master"], b["m"], b["v"], host_grads=host_g, host_norm=host_norm)
    torch.cuda.synchronize()
    norms = [float(host_norm.item())]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        opt.step_graph(b["params"], dg, b["master"], b["m"], b["v"], host_grads=host_g, host_norm=host_norm)
    for g in grads[1:]:
        host_g.copy_(g)  # the previous replay has finished: synchronised below
        graph.replay()
        torch.cuda.synchronize()
        norms.append(float(host_norm.item()))
    assert norms == norms_e
    _assert_same(a, b, "graph with host gradients")
    assert torch.equal(dg.view(torch.int16), grads[-1].cuda().view(torch.int16))


def test_device_refuses_steps_it_cannot_count():
    tab, st, grads = _random_state(50_000, 3, True)
    opt = _opt(tab)
    dg = grads[0].cuda()
    before = _clone(st)
    # a table of 3 entries that has not reached (1, 1): steps 1..3 are fine, step 4 is refused
    opt.init_device_clock(t=3, seed_base=1)
    opt.d_bias = mp.mp_bias_table(H["beta1"], H["beta2"], 3).cuda()
    opt.step_graph(st["params"], dg, st["master"], st["m"], st["v"])
    assert opt.take_status() == mp.MP_ERR_RANGE
    assert opt.device_clock()["t"] == 3
    _assert_same(before, st, "refused step")
    # a negative count is refused too, and so is a count that cannot advance
    for t0 in (-5, (1 << 31) - 1):
        opt.init_device_clock(t=t0, seed_base=1)
        opt.step_graph(st["params"], dg, st["master"], st["m"], st["v"])
        assert opt.take_status() == mp.MP_ERR_RANGE
        assert opt.device_clock()["t"] == t0
        _assert_same(before, st, f"refused step (t = {t0})")
    # a short table that ends at (1, 1) serves every later step: betas 0 give bc = 1 from t = 1
    opt0 = _opt(tab, beta1=0.0, beta2=0.0)
    opt0.init_device_clock(t=1000, seed_base=1)
    assert opt0.d_bias.numel() == 2
    opt0.step_graph(st["params"], dg, st["master"], st["m"], st["v"])
    assert opt0.take_status() == 0 and opt0.device_clock()["t"] == 1001
    ref = _clone(before)
    opt_e = _opt(tab, beta1=0.0, beta2=0.0)
    opt_e.step(ref["params"], dg, ref["master"], ref["m"], ref["v"], 1001, 1 + 1001)
    _assert_same(ref, st, "betas 0, t = 1001")


def test_empty_step_still_counts():
    """n = 0: nothing to update, but the step count advances (the train loop's
    step moves on) and the norm of nothing is 0 with scale 1."""
    import ctypes
    tab = mp.TensorTable([])
    opt = _opt([(0, 8, 1)])
    opt.init_device_clock(t=4, seed_base=10)
    hyper = mp.MpHyper(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0)
    st = mp.lib().mp_optimizer_step_graph(None, None, None, None, None, None, 0, tab.ctypes_array, 0,
                                          ctypes.byref(hyper), opt.d_state.data_ptr(), opt.d_bias.data_ptr(),
                                          opt.d_bias.numel() // 2, opt.workspace.data_ptr(),
                                          opt.workspace.numel(), None, 0.0, None, opt.d_norm.data_ptr(),
                                          opt.d_scale.data_ptr(), opt.d_status.data_ptr(), None, None)
    assert st == mp.MP_OK
    torch.cuda.synchronize()
    clock = opt.device_clock()
    assert clock["t"] == 5 and clock["seed"] == 15
    assert float(opt.d_norm.item()) == 0.0 and float(opt.d_scale.item()) == 1.0
    assert opt.take_status() == 0


def test_graph_soak_two_thousand_steps_equal_ordinary_steps():
    """2001 steps on a 4M-element buffer whose table has more than 1024 decay
    segments (several launches per step), with the outlier check on: one
    plain call, then a graph of two captured steps (alternating gradient
    buffers) replayed 1000 times, against 2001 ordinary calls. Every state
    bit, the last norm, the status and the device step count agree at the
    end: no replay reorders, drops or repeats work."""
    n = 4_000_037
    tab, st, grads = _random_state(n, 99, True, 0, 5000)
    g0, g1 = grads[0].cuda(), grads[1].cuda()
    seed_base, steps = 777, 2001
    a, b = _clone(st), _clone(st)

    opt_e = _opt(tab, outlier_z=3.0)
    for t in range(1, steps + 1):
        opt_e.step(a["params"], g0 if t % 2 else g1, a["master"], a["m"], a["v"], t, (seed_base + t) & 0xFFFFFFFF)
    torch.cuda.synchronize()

    opt_g = _opt(tab, outlier_z=3.0)
    opt_g.init_device_clock(t=0, seed_base=seed_base)
    opt_g.step_graph(b["params"], g0, b["master"], b["m"], b["v"])  # step 1, outside the capture
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        opt_g.step_graph(b["params"], g1, b["master"], b["m"], b["v"])  # even steps
        opt_g.step_graph(b["params"], g0, b["master"], b["m"], b["v"])  # odd steps
    for _ in range((steps - 1) // 2):
        graph.replay()
    torch.cuda.synchronize()

    _assert_same(a, b, "soak")
    assert float(opt_e.d_norm.item()) == float(opt_g.d_norm.item())
    assert opt_e.take_status() == opt_g.take_status()
    clock = opt_g.device_clock()
    assert clock["t"] == steps and clock["seed"] == seed_base + steps
