"""The device-side grad-norm outlier check against the oracle, and its effect
on the step (llm.c ch. 04 §4: skip the update when the norm's z-score over a
window of 128 past norms is above a threshold)."""
import math
import struct

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


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _bits(x: float) -> int:
    return struct.unpack("<Q", struct.pack("<d", x))[0]


def test_outlier_check_bit_exact_against_oracle():
    rng = np.random.default_rng(3)
    norms = (1.0 + 0.05 * rng.standard_normal(400)).astype(np.float32)
    norms[150] = 9.0    # spike: skipped
    norms[151] = np.nan  # non-finite: never joins the window
    norms[200] = np.inf
    norms[260] = 1.3    # mild: kept at threshold 6
    det = mp.OutlierDetector(6.0)
    ref = oracle.OutlierCheck()
    d_norm = torch.empty(1, dtype=torch.float32, device="cuda")
    d_scale = torch.empty(1, dtype=torch.float32, device="cuda")
    d_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    skips = 0
    for i, x in enumerate(norms):
        d_norm.fill_(float(x))
        d_scale.fill_(0.5)
        d_status.zero_()
        det.check(d_norm, d_scale, d_status)
        st_o, z_o, sc_o = ref.check(float(x), 6.0, 0.5)
        z = det.d_z.item()
        assert (math.isnan(z) and math.isnan(z_o)) or _bits(z) == _bits(z_o), (i, z, z_o)
        assert int(d_status.item()) == st_o, i
        sc = d_scale.item()
        assert (math.isnan(sc) and math.isnan(sc_o)) or sc == sc_o, i
        skips += st_o == 8
    assert skips >= 1 and ref.state.count == 398


def test_outlier_skip_leaves_the_state_untouched_and_later_steps_proceed():
    name = "tiny"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    H = W.HYPER
    st = {k: t.cuda() for k, t in W.make_state(name).items()}
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"], outlier_z=5.0)
    t = 0
    for t in range(1, 131):
        opt.step(st["params"], W.make_grads(name, t).cuda(), st["master"], st["m"], st["v"], t, W.step_seed(t))
    assert opt.take_status() == 0
    before = {k: x.clone() for k, x in st.items()}
    spike = (W.make_grads(name, 131).float() * 100.0).to(torch.bfloat16).cuda()
    opt.step(st["params"], spike, st["master"], st["m"], st["v"], 131, W.step_seed(131))
    torch.cuda.synchronize()
    assert opt.take_status() == mp.MP_SKIPPED_OUTLIER
    assert opt.outlier.d_z.item() > 5.0
    for k in st:
        assert torch.equal(st[k].view(torch.int16) if k == "params" else st[k].view(torch.int32),
                           before[k].view(torch.int16) if k == "params" else before[k].view(torch.int32)), k
    # the next ordinary step runs normally
    opt.step(st["params"], W.make_grads(name, 132).cuda(), st["master"], st["m"], st["v"], 132, W.step_seed(132))
    torch.cuda.synchronize()
    assert opt.take_status() == 0
    assert not torch.equal(st["master"], before["master"])
