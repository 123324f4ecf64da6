"""Seeded synthetic workloads: parameter-set shapes, initial state and gradients.

This module is the only thing the CUDA path's tests/benchmark and the CPU
oracle's tests share. It holds none of the optimizer's arithmetic: only
tensor tables (names, shapes, offsets, decay flags), seeded random draws and
dtype casts (bf16 inputs are the round-to-nearest-even cast of fp32 draws).

Parameter sets (one flat buffer each, tensors in the order listed):
  tiny        28,672 params: the d=32, 2-layer GPT-style model of CMU 11-667
              lecture 13 notes §0.3 (wte 64x32, wpe 36x32, 2 blocks, lnf).
  gpt2_124m   GPT-2 small: V=50304, T=1024, d=768, 12 layers, 4x MLP, tied wte.
  gpt2_1558m  GPT-2 XL: same layout with d=1600, 48 layers.
  llama3_8b   Llama-3-8B: d=4096, 32 layers, 32 query / 8 KV heads of 128,
              SwiGLU FFN 14336, V=128256, untied embeddings, RMSNorm weights.
Decay follows llm.c ch. 04 "Multi-GPU and mixed precision" §2.2: 2D tensors
(embeddings and matrices) decay, 1D tensors (norm weights, biases) do not.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import torch

BASE_SEED = 1234

# Optimizer hyperparameters used by every parameter set (llm.c ch. 04 §4 uses
# beta2 = 0.95; the CMU 11-667 lecture 13 notes §1.7 give beta1 0.9,
# beta2 0.95, weight decay 0.1 as the common LLM setting).
HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0)


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: Tuple[int, ...]
    kind: str  # "matrix" | "norm" | "bias"

    @property
    def size(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n

    @property
    def decay(self) -> bool:
        return len(self.shape) == 2


@dataclasses.dataclass(frozen=True)
class Entry:
    spec: TensorSpec
    offset: int

    @property
    def size(self) -> int:
        return self.spec.size


def _gpt_specs(V: int, T: int, d: int, L: int) -> List[TensorSpec]:
    specs = [TensorSpec("wte", (V, d), "matrix"), TensorSpec("wpe", (T, d), "matrix")]
    for l in range(L):
        p = f"h.{l}."
        specs += [
            TensorSpec(p + "ln_1.weight", (d,), "norm"),
            TensorSpec(p + "ln_1.bias", (d,), "bias"),
            TensorSpec(p + "attn.c_attn.weight", (d, 3 * d), "matrix"),
            TensorSpec(p + "attn.c_attn.bias", (3 * d,), "bias"),
            TensorSpec(p + "attn.c_proj.weight", (d, d), "matrix"),
            TensorSpec(p + "attn.c_proj.bias", (d,), "bias"),
            TensorSpec(p + "ln_2.weight", (d,), "norm"),
            TensorSpec(p + "ln_2.bias", (d,), "bias"),
            TensorSpec(p + "mlp.c_fc.weight", (d, 4 * d), "matrix"),
            TensorSpec(p + "mlp.c_fc.bias", (4 * d,), "bias"),
            TensorSpec(p + "mlp.c_proj.weight", (4 * d, d), "matrix"),
            TensorSpec(p + "mlp.c_proj.bias", (d,), "bias"),
        ]
    specs += [TensorSpec("ln_f.weight", (d,), "norm"), TensorSpec("ln_f.bias", (d,), "bias")]
    return specs


def _llama_specs(V=128256, d=4096, L=32, n_heads=32, n_kv=8, ffn=14336) -> List[TensorSpec]:
    hd = d // n_heads
    kv = n_kv * hd
    specs = [TensorSpec("tok_embeddings.weight", (V, d), "matrix")]
    for l in range(L):
        p = f"layers.{l}."
        specs += [
            TensorSpec(p + "attention_norm.weight", (d,), "norm"),
            TensorSpec(p + "attention.wq.weight", (d, d), "matrix"),
            TensorSpec(p + "attention.wk.weight", (kv, d), "matrix"),
            TensorSpec(p + "attention.wv.weight", (kv, d), "matrix"),
            TensorSpec(p + "attention.wo.weight", (d, d), "matrix"),
            TensorSpec(p + "ffn_norm.weight", (d,), "norm"),
            TensorSpec(p + "feed_forward.w1.weight", (ffn, d), "matrix"),
            TensorSpec(p + "feed_forward.w2.weight", (d, ffn), "matrix"),
            TensorSpec(p + "feed_forward.w3.weight", (ffn, d), "matrix"),
        ]
    specs += [TensorSpec("norm.weight", (d,), "norm"), TensorSpec("output.weight", (V, d), "matrix")]
    return specs


def specs_for(name: str) -> List[TensorSpec]:
    if name == "tiny":
        return _gpt_specs(V=64, T=36, d=32, L=2)
    if name == "gpt2_124m":
        return _gpt_specs(V=50304, T=1024, d=768, L=12)
    if name == "gpt2_1558m":
        return _gpt_specs(V=50304, T=1024, d=1600, L=48)
    if name == "llama3_8b":
        return _llama_specs()
    raise KeyError(name)


def layout(specs: List[TensorSpec]) -> List[Entry]:
    out, off = [], 0
    for s in specs:
        out.append(Entry(s, off))
        off += s.size
    return out


def table(entries: List[Entry]) -> List[Tuple[int, int, int]]:
    """(offset, size, decay) per tensor, in buffer order."""
    return [(e.offset, e.size, int(e.spec.decay)) for e in entries]


def total(entries: List[Entry]) -> int:
    return entries[-1].offset + entries[-1].size if entries else 0


# Gradient recipes: standard deviation per tensor for each parameter set.
def grad_std(name: str, entries: List[Entry]) -> List[float]:
    if name == "tiny":
        # N(0, 1e-3 * (1 + tensor index)), fresh per step.
        return [1e-3 * (1 + k) for k in range(len(entries))]
    if name == "gpt2_124m":
        # N(0, 1e-3), with the first MLP matrix scaled x1e3 so clipping fires.
        return [1.0 if e.spec.name == "h.0.mlp.c_fc.weight" else 1e-3 for e in entries]
    if name == "gpt2_1558m":
        return [1e-3] * len(entries)
    if name == "llama3_8b":
        return [1e-4] * len(entries)
    raise KeyError(name)


def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


_CHUNK = 1 << 26


def _fill_normal(out: torch.Tensor, std: float, gen: torch.Generator):
    """out[:] = bf16/fp32 cast of N(0, std) draws, generated in chunks."""
    n = out.numel()
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        x = torch.randn(b - a, generator=gen, device=out.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[a:b].copy_(x)


def make_state(name: str, device="cpu", seed: int = BASE_SEED, with_master: bool = True,
               entries: Optional[List[Entry]] = None) -> Dict[str, torch.Tensor]:
    """Initial optimizer state: fp32 master ~N(0, 0.02) on matrices, norm
    weights 1, biases 0; bf16 params = round-to-nearest cast of the master;
    m = v = 0."""
    entries = entries or layout(specs_for(name))
    N = total(entries)
    gen = _generator(device, seed)
    master = torch.empty(N, dtype=torch.float32, device=device)
    for e in entries:
        sl = master[e.offset:e.offset + e.size]
        if e.spec.kind == "matrix":
            _fill_normal(sl, 0.02, gen)
        elif e.spec.kind == "norm":
            sl.fill_(1.0)
        else:
            sl.zero_()
    params = master.to(torch.bfloat16)
    st = dict(params=params,
              m=torch.zeros(N, dtype=torch.float32, device=device),
              v=torch.zeros(N, dtype=torch.float32, device=device))
    if with_master:
        st["master"] = master
    else:
        del master
    return st


def make_grads(name: str, step: int, device="cpu", seed: int = BASE_SEED,
               entries: Optional[List[Entry]] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16 gradients for 1-based step `step`, drawn from seed + step."""
    entries = entries or layout(specs_for(name))
    N = total(entries)
    if out is None:
        out = torch.empty(N, dtype=torch.bfloat16, device=device)
    gen = _generator(out.device, seed + 1000003 * step)
    for e, std in zip(entries, grad_std(name, entries)):
        _fill_normal(out[e.offset:e.offset + e.size], std, gen)
    return out


def step_seed(step: int, seed: int = BASE_SEED) -> int:
    """Per-step rounding seed (a host-side counter, like llm.c's rng state)."""
    return (seed + step) & 0xFFFFFFFF


def sr_stress_weights(n: int = 64 << 20, device="cpu", seed: int = BASE_SEED) -> torch.Tensor:
    """fp32 weights with |w| log-uniform in [1e-3, 1e1] and random sign."""
    gen = _generator(device, seed)
    u = torch.rand(n, generator=gen, device=device, dtype=torch.float64)
    mag = torch.pow(10.0, u * 4.0 - 3.0)
    sign = torch.where(torch.rand(n, generator=gen, device=device) < 0.5, -1.0, 1.0)
    return (mag * sign).to(torch.float32)


def random_table(n: int, gen: torch.Generator, min_size: int = 1, max_size: int = 5000,
                 ) -> List[Tuple[int, int, int]]:
    """A random tensor table tiling [0, n): ragged sizes, random decay flags."""
    out, off = [], 0
    while off < n:
        size = int(torch.randint(min_size, max_size + 1, (1,), generator=gen))
        size = min(size, n - off)
        decay = int(torch.randint(0, 2, (1,), generator=gen))
        out.append((off, size, decay))
        off += size
    return out


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor's raw patterns."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
