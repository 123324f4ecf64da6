"""Independent optimizer steps issued from two host threads onto two CUDA
streams give exactly the results of running them one after the other: the
library keeps no per-call host state between calls (its only host caches —
device attributes and occupancy — hold the same values for every caller),
and each call's kernels touch only that call's buffers."""
import threading

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


def _case(n, seed, max_size):
    gen = torch.Generator().manual_seed(seed)
    tab = W.random_table(n, gen, 1, max_size)
    master = (torch.randn(n, generator=gen) * 0.05).cuda()
    grads = [(torch.randn(n, generator=gen) * 1e-2).to(torch.bfloat16).cuda() for _ in range(3)]
    st = dict(params=master.to(torch.bfloat16), master=master, m=torch.zeros_like(master),
              v=torch.zeros_like(master))
    return tab, st, grads


def _run(tab, st, grads, stream, with_master):
    H = W.HYPER
    with torch.cuda.stream(stream):  # the optimizer's buffers are initialised on this stream too
        opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                           weight_decay=H["weight_decay"], clip=H["clip"])
        for t, g in enumerate(grads, start=1):
            opt.step(st["params"], g, st["master"] if with_master else None, st["m"], st["v"], t, 100 + t,
                     stream=stream)
    return opt


def _clone(st):
    return {k: x.clone() for k, x in st.items()}


def _same(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def test_two_threads_two_streams_match_sequential_runs():
    cases = [_case(3_000_017, 1, 200_000), _case(1_234_567, 2, 5_000)]
    masters = [True, False]
    torch.cuda.synchronize()

    seq = []
    for (tab, st, grads), wm in zip(cases, masters):
        s = _clone(st)
        torch.cuda.synchronize()
        _run(tab, s, grads, torch.cuda.current_stream(), wm)
        torch.cuda.synchronize()
        seq.append(s)

    conc = [_clone(st) for _, st, _ in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            tab, _, grads = cases[i]
            _run(tab, conc[i], grads, streams[i], masters[i])
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(2):
        for k in seq[i]:
            assert _same(seq[i][k], conc[i][k]), (i, k)
