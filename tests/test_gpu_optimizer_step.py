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
