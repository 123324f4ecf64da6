"""The oracle's command-line front end (oracle/mp_oracle_cli.c) gives the
library's results on raw binary files (no GPU)."""
import os
import subprocess

import numpy as np
import torch

import oracle
import workloads as W
from oracle import build as ob


def _cli(*args):
    ob.build()
    return subprocess.run([ob.CLI, *map(str, args)], capture_output=True, text=True, timeout=120)


def test_step_files_equal_the_library(tmp_path):
    name = "tiny"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    n = W.total(entries)
    st = W.make_state(name)
    g = W.bf16_bits(W.make_grads(name, 3)).copy()
    H = W.HYPER
    files = {k: tmp_path / k for k in ("params", "grads", "master", "m", "v", "table")}
    host = dict(params=W.bf16_bits(st["params"]).copy(), master=st["master"].numpy().copy(),
                m=(np.arange(n, dtype=np.float32) * 1e-6), v=np.full(n, 1e-8, np.float32))
    host["params"].tofile(files["params"])
    g.tofile(files["grads"])
    for k in ("master", "m", "v"):
        host[k].tofile(files[k])
    files["table"].write_text("".join(f"{o} {s} {d}\n" for o, s, d in tab))
    r = _cli("step", n, files["table"], files["params"], files["grads"], files["master"], files["m"], files["v"],
             H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], H["clip"], 3, 77)
    assert r.returncode == 0, r.stderr
    _, nrm, sc = oracle.grad_norm(g, H["clip"])
    assert r.stdout.split()[:4] == ["norm", f"{float(nrm):.9g}", "scale", f"{float(sc):.9g}"]
    assert oracle.adamw_step(host["params"], g, host["master"], host["m"], host["v"], 0, tab, H["lr"], H["beta1"],
                             H["beta2"], H["eps"], H["weight_decay"], float(sc), 3, 77) == 0
    assert np.array_equal(np.fromfile(files["params"], np.uint16), host["params"])
    for k in ("master", "m", "v"):
        assert np.array_equal(np.fromfile(files[k], np.float32).view(np.uint32), host[k].view(np.uint32)), k


def test_no_master_step_and_bad_table(tmp_path):
    n = 1000
    rng = np.random.default_rng(1)
    p = W.bf16_bits(torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)).copy()
    g = W.bf16_bits(torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 0.01).to(torch.bfloat16)).copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    for a, name in ((p, "p"), (g, "g"), (m, "m"), (v, "v")):
        a.tofile(tmp_path / name)
    (tmp_path / "t").write_text("0 600 1\n600 400 0\n")
    r = _cli("step", n, tmp_path / "t", tmp_path / "p", tmp_path / "g", "-", tmp_path / "m", tmp_path / "v",
             1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1, 5)
    assert r.returncode == 0, r.stderr
    ref = p.copy()
    _, _, sc = oracle.grad_norm(g, 1.0)
    mm, vv = np.zeros(n, np.float32), np.zeros(n, np.float32)
    assert oracle.adamw_step(ref, g, None, mm, vv, 0, [(0, 600, 1), (600, 400, 0)], 1e-3, 0.9, 0.95, 1e-8, 0.1,
                             float(sc), 1, 5) == 0
    assert np.array_equal(np.fromfile(tmp_path / "p", np.uint16), ref)
    (tmp_path / "bad").write_text("0 600 1\n601 399 0\n")  # a gap: not a tiling of [0, n)
    r = _cli("step", n, tmp_path / "bad", tmp_path / "p", tmp_path / "g", "-", tmp_path / "m", tmp_path / "v",
             1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1, 5)
    assert r.returncode == 1


def test_sr_sr16_and_noise_equal_the_library(tmp_path):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(5000) * 10.0 ** rng.uniform(-5, 5, 5000)).astype(np.float32)
    x.tofile(tmp_path / "x")
    r = _cli("sr", x.size, tmp_path / "x", tmp_path / "y", (1 << 32) - 77, 123)
    assert r.returncode == 0, r.stderr
    assert np.array_equal(np.fromfile(tmp_path / "y", np.uint16), oracle.stochastic_round(x, (1 << 32) - 77, 123))
    r = _cli("sr16", x.size, tmp_path / "x", tmp_path / "h", (1 << 32) - 77, 123)
    assert r.returncode == 0, r.stderr
    assert np.array_equal(np.fromfile(tmp_path / "h", np.uint16),
                          oracle.stochastic_round_fp16(x, (1 << 32) - 77, 123))
    r = _cli("noise", (1 << 32) - 2, 5, 9)
    assert r.returncode == 0
    got = [int(w, 16) for w in r.stdout.split()]
    assert got == [oracle.noise_u32((1 << 32) - 2 + i, 9) for i in range(5)]
    assert _cli("frobnicate").returncode == 1
