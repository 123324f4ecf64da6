"""mp_optimizer_step: the whole step in one native call, against the same
kernels called one by one, and with the gradients read from page-locked
host memory by the norm kernel."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _setup(n_params=(1 << 22) + 12345):
    from bench import prefix_entries
    name = "gpt2_124m"
    entries = prefix_entries(W.layout(W.specs_for(name)), n_params)
    st = W.make_state(name, device="cuda", entries=entries)
    g = W.make_grads(name, 1, device="cuda", entries=entries)
    return W.table(entries), st, g


def _same(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def test_one_call_equals_the_separate_calls():
    tab, st, g = _setup()
    H = W.HYPER
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    a = {k: x.clone() for k, x in st.items()}
    b = {k: x.clone() for k, x in st.items()}
    opt = mp.Optimizer(tab, clip=H["clip"], **kw)
    for t in (1, 2, 3):
        opt.step(a["params"], g, a["master"], a["m"], a["v"], t, W.step_seed(t))
        norm_a = opt.d_norm.clone()
        mp.mp_grad_norm(g, H["clip"], opt.workspace, opt.d_norm, opt.d_scale)
        mp.mp_adamw_step(b["params"], g, b["master"], b["m"], b["v"], opt.table, d_grad_scale=opt.d_scale, t=t,
                         seed=W.step_seed(t), **kw)
        assert _same(norm_a, opt.d_norm)
    torch.cuda.synchronize()
    for k in a:
        assert _same(a[k], b[k]), k


def test_host_gradients_read_by_the_norm_kernel():
    tab, st, g = _setup()
    H = W.HYPER
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    host_g = torch.empty(g.numel(), dtype=torch.bfloat16, pin_memory=True)
    host_g.copy_(g.cpu())
    host_norm = torch.full((1,), -1.0, dtype=torch.float32, pin_memory=True)
    landing = torch.zeros_like(g)
    a = {k: x.clone() for k, x in st.items()}
    b = {k: x.clone() for k, x in st.items()}
    opt_a = mp.Optimizer(tab, clip=H["clip"], **kw)
    opt_b = mp.Optimizer(tab, clip=H["clip"], **kw)
    opt_a.step(a["params"], g, a["master"], a["m"], a["v"], 1, 11)
    opt_b.step(b["params"], landing, b["master"], b["m"], b["v"], 1, 11, host_grads=host_g, host_norm=host_norm)
    torch.cuda.synchronize()
    assert _same(landing, g)  # the device copy of the host gradients
    assert host_norm.item() == opt_b.d_norm.item() == opt_a.d_norm.item()
    for k in a:
        assert _same(a[k], b[k]), k


def test_pageable_host_gradients_are_refused():
    tab, st, g = _setup(1 << 16)
    H = W.HYPER
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"])
    pageable = g.cpu()  # not page-locked
    before = {k: x.clone() for k, x in st.items()}
    with pytest.raises(mp.MpError) as ei:
        opt.step(st["params"], torch.empty_like(g), st["master"], st["m"], st["v"], 1, 1, host_grads=pageable)
    assert ei.value.status == mp.MP_ERR_ACCESS
    torch.cuda.synchronize()
    for k in st:
        assert _same(st[k], before[k]), k


@pytest.mark.parametrize("host_off,dev_off,n", [(1, 1, 2048 * 5 + 7), (1, 0, 100003), (0, 3, 4099), (0, 0, 7)])
def test_host_gradients_unaligned_and_ragged(host_off, dev_off, n):
    """Unaligned host or device buffers take the element-wise copy path; the
    result must equal the same step on device gradients bit for bit, and the
    landing buffer must not be written outside its n elements. The reference
    gradients are 16-B aligned exactly when both copy buffers are, so both
    norms take the same vector or element-wise path (the two paths differ in
    the rounding of the fp32 squares' pairwise sums, within the norm's
    tolerance but not bit for bit)."""
    gen = torch.Generator().manual_seed(n + host_off)
    tab = W.random_table(n, gen, 1, 3000)
    g_cpu = (torch.randn(n, generator=gen) * 1e-2).to(torch.bfloat16)
    master = (torch.randn(n, generator=gen) * 0.05).cuda()
    st = dict(params=master.to(torch.bfloat16), master=master, m=torch.zeros_like(master), v=torch.zeros_like(master))
    host = torch.empty(n + host_off, dtype=torch.bfloat16, pin_memory=True)
    host[host_off:].copy_(g_cpu)
    guard = 4096
    land_buf = torch.full((n + dev_off + 2 * guard,), 0x5A5A, dtype=torch.int16, device="cuda")
    landing = land_buf[guard + dev_off:guard + dev_off + n].view(torch.bfloat16)
    H = W.HYPER
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    a = {k: x.clone() for k, x in st.items()}
    b = {k: x.clone() for k, x in st.items()}
    opt_a = mp.Optimizer(tab, clip=H["clip"], **kw)
    opt_b = mp.Optimizer(tab, clip=H["clip"], **kw)
    ref_off = 0 if host_off % 8 == 0 and dev_off % 8 == 0 else 1
    g_ref = torch.empty(n + ref_off, dtype=torch.bfloat16, device="cuda")[ref_off:]
    g_ref.copy_(g_cpu)
    opt_a.step(a["params"], g_ref, a["master"], a["m"], a["v"], 3, 5)
    opt_b.step(b["params"], landing, b["master"], b["m"], b["v"], 3, 5, host_grads=host[host_off:])
    torch.cuda.synchronize()
    assert _same(landing, g_cpu.cuda())
    h = land_buf.cpu()
    assert torch.all(h[:guard + dev_off] == 0x5A5A) and torch.all(h[guard + dev_off + n:] == 0x5A5A)
    assert opt_a.d_norm.item() == opt_b.d_norm.item()
    for k in a:
        assert _same(a[k], b[k]), k


def _staged_norm_threshold():
    """Elements from which aligned device gradients take the TMA-staged norm
    kernel: two 4 KB pieces (256 vectors of 8) per norm block, 4 blocks per SM."""
    return 2 * 4 * torch.cuda.get_device_properties(0).multi_processor_count * 256 * 8


@pytest.mark.parametrize("extra", [-8, 0, 8 * 257 + 5, 2_509_635, 37_509_633])
def test_staged_norm_partials_equal_the_register_norm_bit_for_bit(extra):
    """Device gradients past the threshold go through the TMA-staged norm
    kernel; pinned host gradients always through the register kernel, which
    reads them over the link. Both add every square in the same order, so
    every per-block partial left in the workspace must be the same fp64 bits,
    and so must the norm and the updated state."""
    n = _staged_norm_threshold() + extra
    gen = torch.Generator().manual_seed(n)
    g_cpu = (torch.randn(n, generator=gen) * 1e-2).to(torch.bfloat16)
    host = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    host.copy_(g_cpu)
    master = (torch.randn(n, generator=gen) * 0.05).cuda()
    st = dict(params=master.to(torch.bfloat16), master=master, m=torch.zeros_like(master), v=torch.zeros_like(master))
    tab = [(0, n // 3, 1), (n // 3, n - n // 3, 0)]
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0)
    a = {k: x.clone() for k, x in st.items()}
    b = {k: x.clone() for k, x in st.items()}
    opt_a, opt_b = mp.Optimizer(tab, **kw), mp.Optimizer(tab, **kw)
    opt_a.workspace.zero_()
    opt_b.workspace.fill_(0x5A)
    opt_a.step(a["params"], g_cpu.cuda(), a["master"], a["m"], a["v"], 2, 9)
    landing = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    opt_b.step(b["params"], landing, b["master"], b["m"], b["v"], 2, 9, host_grads=host)
    torch.cuda.synchronize()
    nb = 4 * torch.cuda.get_device_properties(0).multi_processor_count
    wa = opt_a.workspace[: nb * 8].view(torch.int64)
    wb = opt_b.workspace[: nb * 8].view(torch.int64)
    assert torch.equal(wa, wb)
    assert opt_a.d_norm.item() == opt_b.d_norm.item()
    for k in a:
        assert _same(a[k], b[k]), k


@pytest.mark.parametrize("scale", [1e-30, 1e25])
@pytest.mark.parametrize("n", [3 * 2048 * 152 + 11, 3 * (1 << 20) + 11])
def test_host_gradients_extreme_values_take_the_fp64_path(scale, n):
    """Blocks whose fp32 squares underflow or overflow recompute in fp64 from
    the device copy; the norm must match the device-gradient path (which,
    at the larger size, is the TMA-staged norm kernel)."""
    g_cpu = (torch.randn(n, generator=torch.Generator().manual_seed(1)) * scale).to(torch.bfloat16)
    host = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    host.copy_(g_cpu)
    master = torch.zeros(n, device="cuda")
    st = dict(params=master.to(torch.bfloat16), master=master, m=torch.zeros_like(master), v=torch.zeros_like(master))
    opt_a = mp.Optimizer([(0, n, 1)], lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0)
    opt_b = mp.Optimizer([(0, n, 1)], lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0)
    landing = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    a = {k: x.clone() for k, x in st.items()}
    b = {k: x.clone() for k, x in st.items()}
    opt_a.step(a["params"], g_cpu.cuda(), a["master"], a["m"], a["v"], 1, 2)
    opt_b.step(b["params"], landing, b["master"], b["m"], b["v"], 1, 2, host_grads=host)
    torch.cuda.synchronize()
    assert opt_a.d_norm.item() == opt_b.d_norm.item() and np.isfinite(opt_a.d_norm.item())
    for k in a:
        assert _same(a[k], b[k]), k


@pytest.mark.parametrize("nbytes,src_off,dst_off", [(0, 0, 0), (1, 0, 0), (15, 0, 0), (16, 0, 0),
                                                     ((1 << 24) + 9, 0, 0), ((1 << 20) + 3, 3, 0),
                                                     ((1 << 20) + 5, 0, 5), (1 << 22, 16, 32)])
def test_copy_from_host_is_exact(nbytes, src_off, dst_off):
    """mp_copy_from_host: every byte arrives, aligned (vectors plus a tail) or
    not (byte by byte), and nothing outside the destination range changes."""
    g = torch.Generator().manual_seed(nbytes)
    host = torch.empty(nbytes + src_off, dtype=torch.uint8, pin_memory=True)
    host.copy_(torch.randint(0, 256, (nbytes + src_off,), generator=g, dtype=torch.uint8))
    dev = torch.full((nbytes + dst_off + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    mp.mp_copy_from_host(dev[dst_off:dst_off + max(nbytes, 1)], host[src_off:src_off + max(nbytes, 1)], nbytes)
    torch.cuda.synchronize()
    got = dev.cpu()
    assert torch.equal(got[dst_off:dst_off + nbytes], host[src_off:src_off + nbytes])
    assert bool((got[:dst_off] == 0xA5).all()) and bool((got[dst_off + nbytes:] == 0xA5).all())


def test_copy_from_host_refuses_pageable_memory():
    dev = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(mp.MpError) as e:
        mp.mp_copy_from_host(dev, torch.zeros(64, dtype=torch.uint8))  # not page-locked
    assert e.value.status == mp.MP_ERR_ACCESS


@pytest.mark.parametrize("transfer,n_params", [("kernel", (1 << 22) + 12345), ("engine", (1 << 22) + 12345),
                                               ("kernel", 100_003)])
def test_host_gradient_pipeline_equals_device_gradient_steps(transfer, n_params):
    """HostGradPipeline: each step's gradients copied from page-locked host
    memory on a copy stream, overlapped with the previous step's update; 6
    steps with different gradients must equal the same steps on device
    gradients bit for bit, and the host norms must be each step's norm."""
    tab, st, _ = _setup(n_params)
    H = W.HYPER
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    n = st["m"].numel()
    entries_n = n
    a = {k: x.clone() for k, x in st.items()}
    b = {k: x.clone() for k, x in st.items()}
    grads = [(torch.randn(entries_n, device="cuda", generator=torch.Generator(device="cuda").manual_seed(s))
              * 1e-2 * (1 + s)).to(torch.bfloat16) for s in range(6)]
    host = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(6)]
    for h, g in zip(host, grads):
        h.copy_(g)
    norms = [torch.empty(1, dtype=torch.float32, pin_memory=True) for _ in range(6)]
    opt_a = mp.Optimizer(tab, clip=H["clip"], **kw)
    pipe = mp.HostGradPipeline(opt_a, transfer=transfer)
    for t in range(1, 7):
        pipe.step(a["params"], host[t - 1], a["master"], a["m"], a["v"], t, W.step_seed(t), host_norm=norms[t - 1])
    opt_b = mp.Optimizer(tab, clip=H["clip"], **kw)
    ref_norms = []
    for t in range(1, 7):
        opt_b.step(b["params"], grads[t - 1], b["master"], b["m"], b["v"], t, W.step_seed(t))
        ref_norms.append(opt_b.d_norm.clone())
    torch.cuda.synchronize()
    for k in a:
        assert _same(a[k], b[k]), k
    for got, ref in zip(norms, ref_norms):
        assert float(got.item()) == float(ref.item())
    # one host buffer reused for every step, rewritten after each copy has run
    c = {k: x.clone() for k, x in a.items()}
    d = {k: x.clone() for k, x in a.items()}
    opt_c = mp.Optimizer(tab, clip=H["clip"], **kw)
    opt_d = mp.Optimizer(tab, clip=H["clip"], **kw)
    pipe_c = mp.HostGradPipeline(opt_c, transfer=transfer)
    one = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    for t in range(7, 10):
        pipe_c.last_copy().synchronize()
        one.copy_(grads[t - 7])
        pipe_c.step(c["params"], one, c["master"], c["m"], c["v"], t, W.step_seed(t))
        opt_d.step(d["params"], grads[t - 7], d["master"], d["m"], d["v"], t, W.step_seed(t))
    torch.cuda.synchronize()
    for k in c:
        assert _same(c[k], d[k]), k
    with pytest.raises(ValueError):
        pipe.step(a["params"], grads[0], a["master"], a["m"], a["v"], 7, 7)  # device tensor, not pinned host
    with pytest.raises(ValueError):  # one gradient short of the parameter set
        pipe.step(a["params"], host[0][:-1], a["master"], a["m"], a["v"], 7, 7)
    with pytest.raises(ValueError):  # fp32 values, not bf16 patterns
        pipe.step(a["params"], torch.zeros(n, dtype=torch.float32, pin_memory=True), a["master"], a["m"], a["v"],
                  7, 7)
