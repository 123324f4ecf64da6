"""The one-launch step for small parameter sets (a cluster of 16 CTAs doing
norm, clip scale, outlier check and update): bit-identical to the general
path's separate kernels for every size up to its limit, and across it.

Which path ran is visible from outside: the general path writes its norm
partials into the caller's workspace, the cluster kernel keeps them in
shared memory and leaves the workspace untouched."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp

H = W.HYPER
KW = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
SMALL_MAX = 32768


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _same(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def _case(n, seed, with_master, nseg_max=24):
    gen = torch.Generator().manual_seed(seed)
    lo = max(1, n // nseg_max)
    tab = W.random_table(n, gen, lo, max(lo, 3 * lo))
    master = torch.randn(n, generator=gen) * 0.05
    st = dict(params=master.to(torch.bfloat16).cuda(), master=master.cuda() if with_master else None,
              m=(torch.randn(n, generator=gen) * 1e-3).cuda(), v=(torch.rand(n, generator=gen) * 1e-6).cuda())
    grads = [(torch.randn(n, generator=gen) * 0.02 * (1 + k)).to(torch.bfloat16).cuda() for k in range(3)]
    return tab, st, grads


def _clone(st):
    return {k: (x.clone() if x is not None else None) for k, x in st.items()}


def _nseg(tab):
    """Decay segments of a table: maximal runs of equal flags."""
    flags = [d for _, size, d in tab if size > 0]
    return sum(1 for i, d in enumerate(flags) if i == 0 or d != flags[i - 1])


def _sentinel(ws):
    ws.fill_(0xA5)
    return ws.clone()


@pytest.mark.parametrize("n", [1, 7, 8, 9, 2047, 2048, 2049, 10_000, 28_672, 30_721, 32_767, 32_768,
                               32_769, 32_776, 65_536])
@pytest.mark.parametrize("with_master", [True, False])
def test_whole_step_equals_separate_kernels(n, with_master):
    tab, st, grads = _case(n, n, with_master)
    a, b = _clone(st), _clone(st)
    opt = mp.Optimizer(tab, clip=H["clip"], **KW)
    ref = mp.Optimizer(tab, clip=H["clip"], **KW)
    for t, g in enumerate(grads, start=1):
        before = _sentinel(opt.workspace)
        opt.step(a["params"], g, a["master"], a["m"], a["v"], t, W.step_seed(t))
        mp.mp_grad_norm(g, H["clip"], ref.workspace, ref.d_norm, ref.d_scale)
        mp.mp_adamw_step(b["params"], g, b["master"], b["m"], b["v"], ref.table, d_grad_scale=ref.d_scale, t=t,
                         seed=W.step_seed(t), d_status=ref.d_status, **KW)
        torch.cuda.synchronize()
        small = torch.equal(opt.workspace, before)
        # small sets with at most 32 decay segments take the cluster kernel
        assert small == (n <= SMALL_MAX and _nseg(tab) <= 32), (n, _nseg(tab))
        assert _same(opt.d_norm, ref.d_norm) and _same(opt.d_scale, ref.d_scale), t
        assert opt.take_status() == 0 and ref.take_status() == 0
    for k in a:
        if a[k] is not None:
            assert _same(a[k], b[k]), k


@pytest.mark.parametrize("n,nseg_max", [(20_000, 200), (32_768, 300)])
def test_many_segments_take_the_general_path(n, nseg_max):
    """More than 32 decay segments do not fit the cluster kernel's table: the
    whole-step call then runs the general path, with the same results."""
    tab, st, grads = _case(n, 7 * n, True, nseg_max=nseg_max)
    assert _nseg(tab) > 32
    a, b = _clone(st), _clone(st)
    opt = mp.Optimizer(tab, clip=H["clip"], **KW)
    ref = mp.Optimizer(tab, clip=H["clip"], **KW)
    before = _sentinel(opt.workspace)
    opt.step(a["params"], grads[0], a["master"], a["m"], a["v"], 1, 3)
    mp.mp_grad_norm(grads[0], H["clip"], ref.workspace, ref.d_norm, ref.d_scale)
    mp.mp_adamw_step(b["params"], grads[0], b["master"], b["m"], b["v"], ref.table, d_grad_scale=ref.d_scale,
                     t=1, seed=3, **KW)
    torch.cuda.synchronize()
    assert not torch.equal(opt.workspace, before)
    for k in a:
        assert _same(a[k], b[k]), k


def test_small_step_graph_with_host_gradients():
    """The tiny set as a captured graph reading pinned host gradients: the
    cluster kernel in a graph, against ordinary whole-step calls."""
    name = "tiny"
    tab = W.table(W.layout(W.specs_for(name)))
    st = {k: x.cuda() for k, x in W.make_state(name).items()}
    n = st["m"].numel()
    a, b = _clone(st), _clone(st)
    grads = [W.make_grads(name, t) for t in range(1, 9)]
    ref = mp.Optimizer(tab, clip=H["clip"], **KW)
    for t, g in enumerate(grads, start=1):
        ref.step(a["params"], g.cuda(), a["master"], a["m"], a["v"], t, 50 + t)
    opt = mp.Optimizer(tab, clip=H["clip"], **KW)
    opt.init_device_clock(t=0, seed_base=50)
    host_g = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    dev_g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    host_g.copy_(grads[0])
    opt.step_graph(b["params"], dev_g, b["master"], b["m"], b["v"], host_grads=host_g)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        opt.step_graph(b["params"], dev_g, b["master"], b["m"], b["v"], host_grads=host_g)
    for g in grads[1:]:
        host_g.copy_(g)
        graph.replay()
        torch.cuda.synchronize()
    assert opt.take_status() == 0 and opt.device_clock()["t"] == len(grads)
    for k in a:
        assert _same(a[k], b[k]), k


def test_tiny_set_takes_the_cluster_kernel():
    tab = W.table(W.layout(W.specs_for("tiny")))
    st = {k: x.cuda() for k, x in W.make_state("tiny").items()}
    opt = mp.Optimizer(tab, clip=H["clip"], **KW)
    before = _sentinel(opt.workspace)
    opt.step(st["params"], W.make_grads("tiny", 1).cuda(), st["master"], st["m"], st["v"], 1, W.step_seed(1))
    torch.cuda.synchronize()
    assert torch.equal(opt.workspace, before)


@pytest.mark.parametrize("n,host_off", [(28_672, 0), (32_768, 0), (4099, 0), (4099, 1), (20_000, 3),
                                        (20_000, 4)])
def test_small_step_with_host_gradients(n, host_off):
    """host_off elements into a pinned buffer: 1 and 3 leave the host
    gradients 2-B aligned only (the general path then runs), 4 is 8-B aligned.
    The reference reads device gradients at the same offset, so that both
    norms take the same vector or element-wise path (the two differ in the
    rounding of the fp32 squares' pairwise sums)."""
    tab, st, grads = _case(n, 3 * n, True)
    a, b = _clone(st), _clone(st)
    opt = mp.Optimizer(tab, clip=H["clip"], **KW)
    ref = mp.Optimizer(tab, clip=H["clip"], **KW)
    host_g = torch.empty(n + host_off, dtype=torch.bfloat16, pin_memory=True)[host_off:]
    host_norm = torch.empty(1, dtype=torch.float32, pin_memory=True)
    dev_copy = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    g_ref = torch.empty(n + host_off, dtype=torch.bfloat16, device="cuda")[host_off:]
    for t, g in enumerate(grads, start=1):
        host_g.copy_(g.cpu())
        g_ref.copy_(g)
        opt.step(a["params"], dev_copy, a["master"], a["m"], a["v"], t, W.step_seed(t), host_grads=host_g,
                 host_norm=host_norm)
        mp.mp_grad_norm(g_ref, H["clip"], ref.workspace, ref.d_norm, ref.d_scale)
        mp.mp_adamw_step(b["params"], g_ref, b["master"], b["m"], b["v"], ref.table, d_grad_scale=ref.d_scale,
                         t=t, seed=W.step_seed(t), **KW)
        torch.cuda.synchronize()
        assert _same(dev_copy, g)
        assert float(host_norm.item()) == float(ref.d_norm.item())
    for k in a:
        assert _same(a[k], b[k]), k


def test_small_step_refuses_a_nonfinite_norm_and_writes_nothing():
    tab, st, grads = _case(30_000, 5, True)
    g = grads[0].clone()
    g[12345] = float("inf")
    before = _clone(st)
    opt = mp.Optimizer(tab, clip=H["clip"], **KW)
    opt.step(st["params"], g, st["master"], st["m"], st["v"], 1, 1)
    assert opt.take_status() == mp.MP_ERR_NONFINITE
    assert torch.isinf(opt.d_norm).all() and torch.isnan(opt.d_scale).all()
    for k in st:
        assert _same(st[k], before[k]), k


def test_small_step_outlier_and_device_clock_match_general_path():
    """Outlier window, skip and the device step counter through the cluster
    kernel (n = 30,000, replayable steps) against the same run through the
    general path's separate kernels (norm, outlier check, update)."""
    n_small = 30_000
    gen = torch.Generator().manual_seed(9)
    tab_small = [(0, 10_000, 1), (10_000, 5_000, 0), (15_000, 15_000, 1)]
    master = torch.randn(n_small, generator=gen) * 0.05
    grads = [(torch.randn(n_small, generator=gen) * 0.01).to(torch.bfloat16) for _ in range(140)]
    grads[133][:n_small] = (grads[133][:n_small].float() * 300.0).to(torch.bfloat16)  # a norm spike
    small = dict(params=master[:n_small].to(torch.bfloat16).cuda(), master=master[:n_small].cuda(),
                 m=torch.zeros(n_small, device="cuda"), v=torch.zeros(n_small, device="cuda"))
    ref = _clone(small)
    o_small = mp.Optimizer(tab_small, clip=H["clip"], outlier_z=4.0, **KW)
    o_ref = mp.Optimizer(tab_small, clip=H["clip"], outlier_z=4.0, **KW)
    o_small.init_device_clock(t=0, seed_base=77)
    statuses = []
    for t, g in enumerate(grads, start=1):
        gs = g[:n_small].cuda()
        o_small.step_graph(small["params"], gs, small["master"], small["m"], small["v"])
        # the general path: the separate kernels, outlier check in between
        mp.mp_grad_norm(gs, H["clip"], o_ref.workspace, o_ref.d_norm, o_ref.d_scale)
        o_ref.outlier.check(o_ref.d_norm, o_ref.d_scale, o_ref.d_status)
        mp.mp_adamw_step(ref["params"], gs, ref["master"], ref["m"], ref["v"], o_ref.table,
                         d_grad_scale=o_ref.d_scale, t=t, seed=77 + t, d_status=o_ref.d_status, **KW)
        st_s, st_r = o_small.take_status(), o_ref.take_status()
        assert st_s == st_r, t
        assert _same(o_small.d_norm, o_ref.d_norm) and _same(o_small.outlier.d_z, o_ref.outlier.d_z), t
        statuses.append(st_s)
    assert statuses.count(mp.MP_SKIPPED_OUTLIER) >= 1 and statuses[133] == mp.MP_SKIPPED_OUTLIER
    assert o_small.device_clock()["t"] == len(grads)
    assert _same(o_small.outlier.state, o_ref.outlier.state)
    for k in small:
        assert _same(small[k], ref[k]), k
