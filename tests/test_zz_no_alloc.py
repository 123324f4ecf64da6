"""mp_grad_norm_noalloc: the gradient norm for callers that cannot allocate
device memory (a framework that owns all of it and hands over only tensors,
or a loop that cannot take cudaMalloc's device-wide synchronisation).

It must give what mp_grad_norm gives on the same inputs, call after call,
although its partial sums live in a scratch array shared by every call. This
file is collected last, so a run that stops at its first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp
    return mp


def _grads(n, seed, scale):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(n, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _with_workspace(mp, g):
    n = g.numel()
    ws = torch.empty(max(8, mp.mp_grad_norm_workspace_bytes(n)), dtype=torch.uint8, device="cuda")
    out = (torch.empty(1, dtype=torch.float32, device="cuda"), torch.empty(1, dtype=torch.float32, device="cuda"),
           torch.empty(1, dtype=torch.float64, device="cuda"))
    mp.mp_grad_norm(g, 1.0, ws, out[0], out[1], out[2])
    return out


def _without_workspace(mp, g):
    """Straight through the C ABI with raw device pointers."""
    out = (torch.full((1,), -1.0, dtype=torch.float32, device="cuda"),
           torch.full((1,), -1.0, dtype=torch.float32, device="cuda"),
           torch.full((1,), -1.0, dtype=torch.float64, device="cuda"))
    st = mp.lib().mp_grad_norm_noalloc(
        ctypes.c_void_p(g.data_ptr()), g.numel(), ctypes.c_float(1.0), ctypes.c_void_p(out[0].data_ptr()),
        ctypes.c_void_p(out[1].data_ptr()), ctypes.c_void_p(out[2].data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mp.MP_OK, mp.status_string(st)
    return out


def test_noalloc_norm_matches_workspace_norm_on_two_calls_in_a_row(mp):
    # two different inputs back to back: a large one (many blocks, every
    # scratch slot in use) then a smaller one that reuses fewer slots
    for n, seed, scale in ((50_000_003, 1, 1e-3), (3 * 2048 + 5, 2, 7.0)):
        g = _grads(n, seed, scale)
        ref = _with_workspace(mp, g)
        got = _without_workspace(mp, g)
        torch.cuda.synchronize()
        norm_r, scale_r, sumsq_r = (x.item() for x in ref)
        norm_g, scale_g, sumsq_g = (x.item() for x in got)
        # the bar the norm tests use: relative error <= 1e-6 (here the same
        # kernels run, so the results are expected to be identical)
        assert abs(sumsq_g - sumsq_r) <= 1e-6 * abs(sumsq_r)
        assert abs(norm_g - norm_r) <= 1e-6 * abs(norm_r)
        assert np.float32(scale_g) == np.float32(scale_r)
        assert (norm_g, scale_g, sumsq_g) == (norm_r, scale_r, sumsq_r)
