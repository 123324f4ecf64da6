"""The C ABI library builds, loads and exports every declared symbol, and its
host-side argument checks reject bad input before any device work (no GPU
needed: every call here fails validation before it would touch CUDA)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mp():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_adamw_gb300 as mp
    return mp


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(mp_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mp_grad_norm", "mp_adamw_step", "mp_stochastic_round", "mp_grad_norm_workspace_bytes",
                     "mp_status_string", "mp_last_cuda_error", "mp_noise_u32", "mp_abi_version"):
        assert required in names


def test_library_exports_every_declared_symbol(mp):
    lib = ctypes.CDLL(mp.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(mp):
    assert mp.abi_version() == 1
    for s in range(8):
        assert mp.status_string(s).startswith("MP_")
    assert "unknown" in mp.status_string(99)


FAKE = 0x100000  # never dereferenced: each call below fails validation first


def _step(mp, **kw):
    args = dict(params=FAKE, grads=FAKE, master=FAKE, m=FAKE, v=FAKE, goff=0, n=100,
                table=[(0, 100, 1)], lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, scale=FAKE, t=1, seed=1,
                status=None)
    args.update(kw)
    tab = mp.TensorTable(args["table"]) if args["table"] is not None else None
    return mp.lib().mp_adamw_step(args["params"], args["grads"], args["master"], args["m"], args["v"],
                                  args["goff"], args["n"], tab.ctypes_array if tab else None,
                                  tab.n_tensors if tab else 0, args["lr"], args["b1"], args["b2"], args["eps"],
                                  args["wd"], args["scale"], args["t"], args["seed"], args["status"], None)


def test_step_argument_checks(mp):
    assert _step(mp, n=0) == mp.MP_OK
    assert _step(mp, params=None) == mp.MP_ERR_NULL
    assert _step(mp, m=None) == mp.MP_ERR_NULL
    assert _step(mp, table=None) == mp.MP_ERR_NULL
    assert _step(mp, params=FAKE + 1) == mp.MP_ERR_ALIGN
    assert _step(mp, master=FAKE + 2) == mp.MP_ERR_ALIGN
    assert _step(mp, scale=FAKE + 2) == mp.MP_ERR_ALIGN
    assert _step(mp, t=0) == mp.MP_ERR_RANGE
    assert _step(mp, b1=1.0) == mp.MP_ERR_RANGE
    assert _step(mp, b2=-0.1) == mp.MP_ERR_RANGE
    assert _step(mp, lr=float("nan")) == mp.MP_ERR_RANGE
    assert _step(mp, eps=float("inf")) == mp.MP_ERR_RANGE
    assert _step(mp, goff=(1 << 62), n=10) == mp.MP_ERR_RANGE
    # table: gap, overlap, not from 0, bad flag, too short for the range
    assert _step(mp, table=[(0, 50, 1), (51, 49, 0)]) == mp.MP_ERR_TABLE
    assert _step(mp, table=[(0, 50, 1), (49, 51, 0)]) == mp.MP_ERR_TABLE
    assert _step(mp, table=[(1, 100, 1)]) == mp.MP_ERR_TABLE
    assert _step(mp, table=[(0, 100, 2)]) == mp.MP_ERR_TABLE
    assert _step(mp, table=[(0, 99, 1)]) == mp.MP_ERR_TABLE
    assert _step(mp, goff=50, n=51, table=[(0, 100, 1)]) == mp.MP_ERR_TABLE
    assert _step(mp, table=[]) == mp.MP_ERR_NULL or _step(mp, table=[]) == mp.MP_ERR_TABLE


def test_norm_and_sr_argument_checks(mp):
    L = mp.lib()
    assert L.mp_grad_norm(None, 10, 1.0, FAKE, 4096, FAKE, FAKE, None, None) == mp.MP_ERR_NULL
    assert L.mp_grad_norm(FAKE, 10, 1.0, None, 4096, FAKE, FAKE, None, None) == mp.MP_ERR_WORKSPACE
    assert L.mp_grad_norm(FAKE, 10, 1.0, FAKE, 4096, None, FAKE, None, None) == mp.MP_ERR_NULL
    assert L.mp_grad_norm(FAKE + 1, 10, 1.0, FAKE, 4096, FAKE, FAKE, None, None) == mp.MP_ERR_ALIGN
    assert L.mp_grad_norm(FAKE, 10, 1.0, FAKE + 4, 4096, FAKE, FAKE, None, None) == mp.MP_ERR_ALIGN
    assert L.mp_grad_norm(FAKE, 10, 0.0, FAKE, 4096, FAKE, FAKE, None, None) == mp.MP_ERR_RANGE
    assert L.mp_grad_norm(FAKE, 10, float("inf"), FAKE, 4096, FAKE, FAKE, None, None) == mp.MP_ERR_RANGE
    assert L.mp_stochastic_round(None, FAKE, 0, 10, 1, None) == mp.MP_ERR_NULL
    assert L.mp_stochastic_round(FAKE + 1, FAKE, 0, 10, 1, None) == mp.MP_ERR_ALIGN
    assert L.mp_stochastic_round(FAKE, FAKE + 2, 0, 10, 1, None) == mp.MP_ERR_ALIGN
    assert L.mp_stochastic_round(FAKE, FAKE, (1 << 62), 10, 1, None) == mp.MP_ERR_RANGE
    assert L.mp_stochastic_round(FAKE, FAKE, 0, 0, 1, None) == mp.MP_OK
    assert L.mp_stochastic_round_fp16(None, FAKE, 0, 10, 1, None) == mp.MP_ERR_NULL
    assert L.mp_stochastic_round_fp16(FAKE, None, 0, 10, 1, None) == mp.MP_ERR_NULL
    assert L.mp_stochastic_round_fp16(FAKE + 1, FAKE, 0, 10, 1, None) == mp.MP_ERR_ALIGN
    assert L.mp_stochastic_round_fp16(FAKE, FAKE + 2, 0, 10, 1, None) == mp.MP_ERR_ALIGN
    assert L.mp_stochastic_round_fp16(FAKE, FAKE, (1 << 62), 10, 1, None) == mp.MP_ERR_RANGE
    assert L.mp_stochastic_round_fp16(FAKE, FAKE, 0, 0, 1, None) == mp.MP_OK
    assert L.mp_accumulate_sr(None, FAKE, 0, 10, 1, None) == mp.MP_ERR_NULL
    assert L.mp_accumulate_sr(FAKE, None, 0, 10, 1, None) == mp.MP_ERR_NULL
    assert L.mp_accumulate_sr(FAKE + 1, FAKE, 0, 10, 1, None) == mp.MP_ERR_ALIGN
    assert L.mp_accumulate_sr(FAKE, FAKE + 2, 0, 10, 1, None) == mp.MP_ERR_ALIGN
    assert L.mp_accumulate_sr(FAKE, FAKE, (1 << 62), 10, 1, None) == mp.MP_ERR_RANGE
    assert L.mp_accumulate_sr(FAKE, FAKE, 0, 0, 1, None) == mp.MP_OK
    assert L.mp_noise_u32(None, 0, 10, 1, None) == mp.MP_ERR_NULL
    assert L.mp_noise_u32(FAKE + 2, 0, 10, 1, None) == mp.MP_ERR_ALIGN


def test_product_never_touches_the_oracle():
    """The CUDA path and the oracle share no code: the package neither
    imports, links nor names the oracle."""
    pkg = os.path.join(ROOT, "mixed_precision_adamw_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read().lower()
                assert "oracle" not in text, f"{fn} mentions the oracle"
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".c", ".h", ".py")):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "mixed_precision_adamw_gb300" not in text and "mp_adamw.h" not in text


def test_optimizer_step_argument_checks(mp):
    L = mp.lib()
    tab = mp.TensorTable([(0, 100, 1)])
    hyper = mp.MpHyper(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0)
    bad_clip = mp.MpHyper(1e-3, 0.9, 0.95, 1e-8, 0.1, 0.0)
    bad_beta = mp.MpHyper(1e-3, 1.0, 0.95, 1e-8, 0.1, 1.0)

    def call(**kw):
        a = dict(params=FAKE, grads=FAKE, host=None, master=FAKE, m=FAKE, v=FAKE, n=100, hyper=hyper, t=1,
                 ws=FAKE, wsb=4096, ost=None, z=0.0, dz=None, norm=FAKE, scale=FAKE, status=None, hnorm=None)
        a.update(kw)
        return L.mp_optimizer_step(a["params"], a["grads"], a["host"], a["master"], a["m"], a["v"], a["n"],
                                   tab.ctypes_array, tab.n_tensors,
                                   ctypes.byref(a["hyper"]) if a["hyper"] is not None else None, a["t"], 3,
                                   a["ws"], a["wsb"], a["ost"], a["z"], a["dz"], a["norm"], a["scale"],
                                   a["status"], a["hnorm"], None)
    assert call(hyper=None) == mp.MP_ERR_NULL
    assert call(norm=None) == mp.MP_ERR_NULL
    assert call(ws=None) == mp.MP_ERR_WORKSPACE
    assert call(hyper=bad_clip) == mp.MP_ERR_RANGE
    assert call(hyper=bad_beta) == mp.MP_ERR_RANGE
    assert call(t=0) == mp.MP_ERR_RANGE
    assert call(params=None) == mp.MP_ERR_NULL
    assert call(ost=FAKE + 4) == mp.MP_ERR_ALIGN
    assert call(dz=FAKE + 4) == mp.MP_ERR_ALIGN
    assert call(host=FAKE + 1) == mp.MP_ERR_ALIGN
    assert call(n=101) == mp.MP_ERR_TABLE
    assert mp.status_string(mp.MP_ERR_ACCESS).startswith("MP_ERR_ACCESS")


def test_graph_step_argument_checks(mp):
    L = mp.lib()
    tab = mp.TensorTable([(0, 100, 1)])
    hyper = mp.MpHyper(float("nan"), 0.9, 0.95, 1e-8, 0.1, 1.0)  # lr is read from the device state

    def call(**kw):
        a = dict(params=FAKE, master=FAKE, n=100, state=FAKE, bias=FAKE, blen=338, norm=FAKE)
        a.update(kw)
        return L.mp_optimizer_step_graph(a["params"], FAKE, None, a["master"], FAKE, FAKE, a["n"],
                                         tab.ctypes_array, tab.n_tensors, ctypes.byref(hyper), a["state"],
                                         a["bias"], a["blen"], FAKE, 4096, None, 0.0, None, a["norm"], FAKE,
                                         None, None, None)
    assert call(state=None) == mp.MP_ERR_NULL
    assert call(bias=None) == mp.MP_ERR_NULL
    assert call(state=FAKE + 8) == mp.MP_ERR_ALIGN
    assert call(bias=FAKE + 2) == mp.MP_ERR_ALIGN
    assert call(blen=0) == mp.MP_ERR_RANGE
    assert call(blen=(1 << 26) + 1) == mp.MP_ERR_RANGE
    assert call(norm=None) == mp.MP_ERR_NULL
    assert call(master=FAKE + 2) == mp.MP_ERR_ALIGN
    assert call(n=101) == mp.MP_ERR_TABLE


@pytest.mark.parametrize("b1,b2", [(0.9, 0.95), (0.9, 0.999), (0.8, 0.99), (0.0, 0.5), (0.0, 0.0),
                                   (0.5, 0.9999)])
def test_bias_table_matches_the_oracle(mp, b1, b2):
    """The device table of replayable steps holds, for every t up to its
    length, the bias corrections the oracle computes for step t, and its
    last entry is the first (1, 1): every later step has the same values."""
    import oracle
    n = mp.mp_bias_table_len(b1, b2)
    assert n >= 1
    tab = mp.mp_bias_table(b1, b2).numpy()
    assert tab.size == 2 * n
    got = tab.view("u4").reshape(n, 2)
    for t in range(1, n + 1):
        bc1, bc2 = oracle.bias_corrections(b1, b2, t)
        assert (int(got[t - 1, 0]), int(got[t - 1, 1])) == (
            int(np.float32(bc1).view("u4")), int(np.float32(bc2).view("u4"))), t
    assert tuple(tab[-2:]) == (1.0, 1.0)
    if n > 1:
        assert tuple(tab[-4:-2]) != (1.0, 1.0)
    assert oracle.bias_corrections(b1, b2, n + 12345) == (1.0, 1.0)


def test_bias_table_checks(mp):
    L = mp.lib()
    assert mp.mp_bias_table_len(1.0, 0.9) == 0
    assert mp.mp_bias_table_len(0.9, -0.1) == 0
    assert mp.mp_bias_table_len(0.9, float("nan")) == 0
    assert mp.mp_bias_table_len(0.9, 1.0 - 2.0 ** -24) == 0  # would need more than 2^26 entries
    assert L.mp_bias_table(0.9, 0.95, 4, None) == mp.MP_ERR_NULL
    assert L.mp_bias_table(0.9, 0.95, 0, FAKE) == mp.MP_ERR_RANGE
    assert L.mp_bias_table(1.0, 0.95, 4, FAKE) == mp.MP_ERR_RANGE


@pytest.mark.parametrize("seed,n,goff,tmax", [(1, 10, 0, 3), (2, 100_000, 0, 5000), (3, 100_003, 17, 40),
                                           (4, 2_000_000, 5, 300), (5, (3 << 26) * 2 + 999, 0, 10 ** 7),
                                           (6, (3 << 26) + 1, 3, 200_000)])
def test_step_launch_plan_invariants(mp, seed, n, goff, tmax):
    """mp_step_launches (the split mp_adamw_step launches with): launches tile
    the range in order, each holds at most 201,326,592 elements and at most
    1024 decay segments, starts stay 4-element aligned from the range start,
    and the segment counts and first flags match the table."""
    import torch
    import workloads as W
    gen = torch.Generator().manual_seed(seed)
    tab = W.random_table(goff + n, gen, 1, tmax)
    plan = mp.mp_step_launches(goff, n, mp.TensorTable(tab))
    assert plan and plan[0][0] == goff and plan[-1][0] + plan[-1][1] == goff + n
    for (o0, s0, _, _), (o1, _, _, _) in zip(plan, plan[1:]):
        assert o0 + s0 == o1
    # decay flag of every element boundary, from the table
    starts = [o for o, _, _ in tab]
    import bisect

    def flag_at(i):
        return tab[bisect.bisect_right(starts, i) - 1][2]

    def segments(a, b):
        cnt, prev, i = 0, None, a
        k = bisect.bisect_right(starts, a) - 1
        while i < b:
            o, sz, d = tab[k]
            if d != prev:
                cnt, prev = cnt + 1, d
            i = o + sz
            k += 1
        return cnt
    for off, size, nseg, first in plan:
        assert 1 <= size <= 3 << 26 and (off - goff) % 4 == 0
        assert 1 <= nseg <= 1024 and first == flag_at(off)
        assert nseg == segments(off, off + size)
    if n <= 3 << 26 and segments(goff, goff + n) <= 1024:
        assert len(plan) == 1


def test_step_launch_plan_checks(mp):
    L = mp.lib()
    tab = mp.TensorTable([(0, 100, 1)])
    import ctypes as C
    cnt = C.c_int64()
    assert L.mp_step_launches(0, 100, tab.ctypes_array, 1, None, 0, None) == mp.MP_ERR_NULL
    assert L.mp_step_launches(0, 100, tab.ctypes_array, 1, None, 4, C.byref(cnt)) == mp.MP_ERR_NULL
    assert L.mp_step_launches(0, 100, tab.ctypes_array, 1, None, -1, C.byref(cnt)) == mp.MP_ERR_RANGE
    assert L.mp_step_launches(0, 101, tab.ctypes_array, 1, None, 0, C.byref(cnt)) == mp.MP_ERR_TABLE
    assert L.mp_step_launches(0, 100, None, 1, None, 0, C.byref(cnt)) == mp.MP_ERR_NULL
    assert L.mp_step_launches(0, 100, tab.ctypes_array, 1, None, 0, C.byref(cnt)) == mp.MP_OK and cnt.value == 1


def test_split_norm_argument_checks(mp):
    """mp_grad_sumsq and mp_clip_scale_from_sumsq reject bad input before any
    device work (the ZeRO-1 norm's two halves)."""
    L = mp.lib()
    assert L.mp_grad_sumsq(None, 10, FAKE, 4096, FAKE, None) == mp.MP_ERR_NULL
    assert L.mp_grad_sumsq(FAKE, 10, FAKE, 4096, None, None) == mp.MP_ERR_NULL
    assert L.mp_grad_sumsq(FAKE, 10, None, 4096, FAKE, None) == mp.MP_ERR_WORKSPACE
    assert L.mp_grad_sumsq(FAKE + 1, 10, FAKE, 4096, FAKE, None) == mp.MP_ERR_ALIGN
    assert L.mp_grad_sumsq(FAKE, 10, FAKE + 4, 4096, FAKE, None) == mp.MP_ERR_ALIGN
    assert L.mp_grad_sumsq(FAKE, 10, FAKE, 4096, FAKE + 4, None) == mp.MP_ERR_ALIGN
    assert L.mp_grad_sumsq(FAKE, (1 << 62) + 1, FAKE, 4096, FAKE, None) == mp.MP_ERR_RANGE
    assert L.mp_clip_scale_from_sumsq(None, 2, 1.0, FAKE, FAKE, None, None) == mp.MP_ERR_NULL
    assert L.mp_clip_scale_from_sumsq(FAKE, 2, 1.0, None, FAKE, None, None) == mp.MP_ERR_NULL
    assert L.mp_clip_scale_from_sumsq(FAKE, 2, 1.0, FAKE, None, None, None) == mp.MP_ERR_NULL
    assert L.mp_clip_scale_from_sumsq(FAKE + 4, 2, 1.0, FAKE, FAKE, None, None) == mp.MP_ERR_ALIGN
    assert L.mp_clip_scale_from_sumsq(FAKE, 2, 1.0, FAKE + 2, FAKE, None, None) == mp.MP_ERR_ALIGN
    assert L.mp_clip_scale_from_sumsq(FAKE, 2, 1.0, FAKE, FAKE, FAKE + 4, None) == mp.MP_ERR_ALIGN
    assert L.mp_clip_scale_from_sumsq(FAKE, 0, 1.0, FAKE, FAKE, None, None) == mp.MP_ERR_RANGE
    assert L.mp_clip_scale_from_sumsq(FAKE, (1 << 20) + 1, 1.0, FAKE, FAKE, None, None) == mp.MP_ERR_RANGE
    assert L.mp_clip_scale_from_sumsq(FAKE, 2, 0.0, FAKE, FAKE, None, None) == mp.MP_ERR_RANGE
    assert L.mp_clip_scale_from_sumsq(FAKE, 2, float("nan"), FAKE, FAKE, None, None) == mp.MP_ERR_RANGE


@pytest.mark.parametrize("kind", ["constant", "cosine", "linear", "wsd"])
def test_lr_schedule_matches_the_oracle(mp, kind):
    """mp_lr_at (host only) against the oracle's schedule, bit for bit, over
    warm-up, decay and past the end, for several shapes of run."""
    import oracle
    for warmup, total, hi, lo, f in ((0, 1, 3e-4, 0.0, 1.0), (10, 110, 6e-4, 6e-5, 0.2), (2000, 60000, 1e-3, 1e-5, 0.1),
                                     (7, 13, 0.5, 0.25, 0.5)):
        s = mp.LRSchedule(kind, lr_max=hi, lr_min=lo, warmup=warmup, total=total, decay_frac=f)
        for t in list(range(1, min(total, 400) + 3)) + [total - 1, total, total + 1, 10 * total + 5]:
            if t < 1:
                continue
            ref = oracle.lr(mp.LR_KINDS[kind], warmup, total, hi, lo, f, t)
            assert s.lr(t) == float(ref), (kind, warmup, total, t)


def test_lr_schedule_checks(mp):
    L = mp.lib()
    out = ctypes.c_float()

    def call(kind, warmup, total, hi, lo, f, t, reserved=0):
        s = mp.MpLrSchedule(kind, reserved, warmup, total, hi, lo, f, 0.0)
        return L.mp_lr_at(ctypes.byref(s), t, ctypes.byref(out))

    assert L.mp_lr_at(None, 1, ctypes.byref(out)) == mp.MP_ERR_NULL
    assert call(1, 10, 100, 1e-3, 0.0, 0.0, 0) == mp.MP_ERR_RANGE        # t < 1
    assert call(4, 10, 100, 1e-3, 0.0, 0.0, 5) == mp.MP_ERR_RANGE        # unknown kind
    assert call(1, 100, 100, 1e-3, 0.0, 0.0, 5) == mp.MP_ERR_RANGE       # total <= warmup
    assert call(1, -1, 100, 1e-3, 0.0, 0.0, 5) == mp.MP_ERR_RANGE        # negative warm-up
    assert call(3, 10, 100, 1e-3, 0.0, 0.0, 5) == mp.MP_ERR_RANGE        # WSD without a decay fraction
    assert call(3, 10, 100, 1e-3, 0.0, 1.5, 5) == mp.MP_ERR_RANGE
    assert call(1, 10, 100, float("inf"), 0.0, 0.0, 5) == mp.MP_ERR_RANGE
    assert call(1, 10, 100, 1e-3, 0.0, 0.0, 5, reserved=1) == mp.MP_ERR_RANGE
    assert call(0, 0, 0, 1e-3, 0.0, 0.0, 5) == mp.MP_OK and out.value == np.float32(1e-3)  # constant needs no total
    with pytest.raises(ValueError):
        mp.LRSchedule("step", lr_max=1e-3)
    with pytest.raises(mp.MpError):
        mp.LRSchedule("cosine", lr_max=1e-3, warmup=5, total=5)


def test_copy_from_host_argument_checks(mp):
    L = mp.lib()
    assert L.mp_copy_from_host(None, None, 0, 1, None) == mp.MP_OK  # nothing to copy
    assert L.mp_copy_from_host(None, FAKE, 16, 1, None) == mp.MP_ERR_NULL
    assert L.mp_copy_from_host(FAKE, None, 16, 1, None) == mp.MP_ERR_NULL
    assert L.mp_copy_from_host(FAKE, FAKE, 16, 0, None) == mp.MP_ERR_RANGE
    assert L.mp_copy_from_host(FAKE, FAKE, 16, 33, None) == mp.MP_ERR_RANGE
