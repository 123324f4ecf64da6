"""Shapes of the synthetic parameter sets (no GPU)."""
import pytest
import torch

import workloads as W


@pytest.mark.parametrize("name,n_params,n_tensors,n_decay", [
    ("tiny", 28_672, 28, 27_776),
    ("gpt2_124m", 124_475_904, 148, 124_354_560),
    ("gpt2_1558m", 1_557_686_400, 580, None),
    ("llama3_8b", 8_030_261_248, 291, None),
])
def test_parameter_set_sizes(name, n_params, n_tensors, n_decay):
    entries = W.layout(W.specs_for(name))
    assert len(entries) == n_tensors
    assert W.total(entries) == n_params
    if n_decay is not None:
        assert sum(e.size for e in entries if e.spec.decay) == n_decay
    # contiguous tiling from 0
    off = 0
    for e in entries:
        assert e.offset == off
        off += e.size
    # decay exactly on the 2D tensors
    assert all(e.spec.decay == (len(e.spec.shape) == 2) for e in entries)


def test_gpt2_1558m_splits_into_eight_equal_shards_of_whole_vectors():
    n = W.total(W.layout(W.specs_for("gpt2_1558m")))
    assert n % 8 == 0 and (n // 8) % 8 == 0
    assert n // 8 == 194_710_800


def test_tiny_state_and_grads_are_seeded():
    a = W.make_state("tiny")
    b = W.make_state("tiny")
    assert torch.equal(a["master"], b["master"]) and torch.equal(a["params"], b["params"])
    assert torch.equal(a["params"], a["master"].to(torch.bfloat16))
    g1 = W.make_grads("tiny", 1)
    assert torch.equal(g1, W.make_grads("tiny", 1))
    assert not torch.equal(g1, W.make_grads("tiny", 2))
    entries = W.layout(W.specs_for("tiny"))
    for e in entries:
        sl = a["master"][e.offset:e.offset + e.size]
        if e.spec.kind == "norm":
            assert torch.all(sl == 1)
        elif e.spec.kind == "bias":
            assert torch.all(sl == 0)


def test_random_table_tiles_the_range():
    g = torch.Generator().manual_seed(0)
    t = W.random_table(100_000, g, 1, 3000)
    off = 0
    for o, s, d in t:
        assert o == off and s >= 1 and d in (0, 1)
        off += s
    assert off == 100_000
