"""libmpadamw.so used from plain C: tests/c_abi/c_abi_check.c allocates its
own device buffers, calls the ABI (mp_optimizer_step, mp_grad_norm,
mp_adamw_step, the roundings, mp_optimizer_step_graph captured into a CUDA
graph with the runtime's own stream capture, the ZeRO-1 norm's two halves,
mp_lr_at and mp_copy_from_host) and compares every output bit for bit with
the CPU oracle linked into the same program, which computes its own norm,
clip scale and steps. No Python or PyTorch on that path. On CPU the program is only compiled and linked (the header is
valid C and every symbol resolves); on a GPU it runs."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "_build", "c_abi")
EXE = os.path.join(OUT, "c_abi_check")


def _build_program():
    import __graft_entry__
    __graft_entry__.build()
    from oracle import build as ob
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    os.makedirs(OUT, exist_ok=True)
    libdir = os.path.join(ROOT, "mixed_precision_adamw_gb300")
    oracle_flags = [f for f in ob.CFLAGS if f not in ("-shared", "-fPIC")]
    subprocess.run(["gcc", *oracle_flags, "-c", ob.SRC, "-o", os.path.join(OUT, "mp_oracle.o")], check=True)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "oracle"), "-I", cuda_inc, "-c",
                    os.path.join(ROOT, "tests", "c_abi", "c_abi_check.c"), "-o", os.path.join(OUT, "c_abi_check.o")],
                   check=True)
    subprocess.run([nvcc, "-o", EXE, os.path.join(OUT, "c_abi_check.o"), os.path.join(OUT, "mp_oracle.o"),
                    "-L", libdir, "-lmpadamw", "-Xlinker", f"-rpath,{libdir}", "-lm"], check=True)
    return EXE


def test_c_program_compiles_and_links():
    assert os.access(_build_program(), os.X_OK)


@pytest.mark.gpu
def test_c_program_matches_the_oracle():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = _build_program()
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bit-identical to the oracle" in r.stdout
