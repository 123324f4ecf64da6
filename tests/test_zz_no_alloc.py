"""mp_grad_norm_noalloc: the gradient norm for callers that cannot allocate
device memory (a framework that owns all of it and hands over only tensors,
or a loop that cannot take cudaMalloc's device-wide synchronisation).

It must give what mp_grad_norm gives on the same inputs, call after call,
although its partial sums live in a scratch array shared by every call, and
its sum of squares must meet the norm's bar against the oracle's fp64 sum.
This file is collected last, so a run that stops at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

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


def _fresh_outputs():
    return (torch.full((1,), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((1,), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((1,), -1.0, dtype=torch.float64, device="cuda"))


def _without_workspace(mp, g):
    """Straight through the C ABI with raw device pointers."""
    out = _fresh_outputs()
    st = mp.lib().mp_grad_norm_noalloc(
        ctypes.c_void_p(g.data_ptr()), g.numel(), ctypes.c_float(1.0), ctypes.c_void_p(out[0].data_ptr()),
        ctypes.c_void_p(out[1].data_ptr()), ctypes.c_void_p(out[2].data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mp.MP_OK, mp.status_string(st)
    return out


def _through_binding(mp, g):
    """The Python wrapper of the same entry point."""
    out = _fresh_outputs()
    mp.mp_grad_norm_noalloc(g, 1.0, out[0], out[1], out[2])
    return out


def _host_bits(g):
    return g.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("call", [_without_workspace, _through_binding])
def test_noalloc_norm_matches_workspace_norm_on_two_calls_in_a_row(mp, call):
    # Back to back: a large input (every scratch slot this device's grid
    # uses), a small one that reuses fewer slots, and a 2-byte-aligned view
    # (the element-by-element path, whose grid and mapping differ).
    big = _grads(50_000_003, 1, 1e-3)
    cases = [big, _grads(3 * 2048 + 5, 2, 7.0), big[1:1_000_001]]
    for g in cases:
        ref = _with_workspace(mp, g)
        got = call(mp, g)
        torch.cuda.synchronize()
        norm_r, scale_r, sumsq_r = (x.item() for x in ref)
        norm_g, scale_g, sumsq_g = (x.item() for x in got)
        # the bar the norm tests use: relative error <= 1e-6 against the
        # oracle's fp64 sum of squares in index order
        sumsq_o = oracle.sumsq(_host_bits(g))
        assert abs(sumsq_g - sumsq_o) <= 1e-6 * abs(sumsq_o)
        assert abs(norm_g - np.sqrt(sumsq_o)) <= 1e-6 * np.sqrt(sumsq_o)
        # the same kernels as mp_grad_norm: identical results expected
        assert abs(sumsq_g - sumsq_r) <= 1e-6 * abs(sumsq_r)
        assert np.float32(scale_g) == np.float32(scale_r)
        assert (norm_g, scale_g, sumsq_g) == (norm_r, scale_r, sumsq_r)
