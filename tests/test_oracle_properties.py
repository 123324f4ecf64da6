"""Property-based pins of the oracle's stochastic rounding (CPU only).

For any fp32 value and any 16-bit draw, the rounding to bf16 and to fp16
(llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §2.3: keep the
value's neighbour toward zero, or move one step away from zero when the
discarded fraction of a step, as 16 bits, exceeds the draw) must:
  - land on one of the value's two neighbours on the target grid, found here
    with torch's bf16 cast and numpy's fp16 cast (round to nearest even,
    library routines that share nothing with the oracle);
  - leave values already on the grid unchanged, whatever the draw;
  - go away from zero exactly when floor(f * 65536) > draw, with f the
    fraction of one step computed here in float64 from those neighbours.
hypothesis draws the values (all fp32 magnitudes, subnormals and the
largest finite values included) and shrinks any counterexample."""
import math

import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402

FINITE_F32 = st.floats(width=32, allow_nan=False, allow_infinity=False)
DRAW = st.integers(min_value=0, max_value=0xFFFF)
SETTINGS = settings(max_examples=3000, deadline=None)
BELOW_65536 = float(np.nextafter(np.float32(65536.0), np.float32(0.0)))  # the largest fp32 below 65536


def _f32_bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def _bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def _bf16_toward_zero(x: float) -> int:
    """Pattern of the bf16 neighbour of x toward zero, from torch's cast."""
    with np.errstate(over="ignore"):
        b = int(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)[0]) & 0xFFFF
    if abs(_bf16_value(b)) > abs(x):  # the cast went away from zero (or to infinity): step back
        b -= 1
    return b


def _fp16_toward_zero(x: float) -> int:
    """Pattern of the fp16 neighbour of x toward zero, from numpy's cast."""
    with np.errstate(over="ignore"):
        h = int(np.array([x], np.float16).view(np.uint16)[0])
    if abs(float(np.array([h], np.uint16).view(np.float16)[0])) > abs(x):
        h -= 1
    return h


def _fp16_value(bits: int) -> float:
    return float(np.array([bits], np.uint16).view(np.float16)[0])


@SETTINGS
@given(x=FINITE_F32, draw=DRAW)
def test_bf16_rounding_lands_on_a_neighbour_by_the_fraction_rule(x, draw):
    x = float(np.float32(x))
    lo = _bf16_toward_zero(x)
    hi = lo + 1  # one step away from zero (sign bit unchanged)
    got = oracle.sr_with_rand(x, draw)
    assert got in (lo, hi), (x, hex(got), hex(lo))
    a = abs(_bf16_value(lo))
    step = abs(_bf16_value(hi)) - a if (hi & 0x7FFF) < 0x7F80 else 2.0 ** ((lo >> 7 & 0xFF) - 127 - 7)
    f = (abs(x) - a) / step
    assert 0.0 <= f < 1.0
    assert (got == hi) == (math.floor(f * 65536) > draw), (x, draw, f)


@SETTINGS
@given(x=FINITE_F32, draw=DRAW)
def test_bf16_rounding_keeps_values_on_the_grid(x, draw):
    b = _f32_bits(float(np.float32(x))) & 0xFFFF0000
    v = float(np.array([b], np.uint32).view(np.float32)[0])
    assert oracle.sr_with_rand(v, draw) == b >> 16


@SETTINGS
@given(x=st.floats(width=32, min_value=-BELOW_65536, max_value=BELOW_65536), draw=DRAW)
def test_fp16_rounding_lands_on_a_neighbour_by_the_fraction_rule(x, draw):
    x = float(np.float32(x))
    lo = _fp16_toward_zero(x)
    hi = lo + 1
    got = oracle.sr_fp16_with_rand(x, draw)
    assert got in (lo, hi), (x, hex(got), hex(lo))
    a = abs(_fp16_value(lo))
    step = 32.0 if (lo & 0x7FFF) == 0x7BFF else abs(_fp16_value(hi)) - a
    f = (abs(x) - a) / step
    assert 0.0 <= f < 1.0
    assert (got == hi) == (math.floor(f * 65536) > draw), (x, draw, f)


@SETTINGS
@given(h=st.integers(min_value=0, max_value=0xFFFF), draw=DRAW)
def test_fp16_rounding_keeps_values_on_the_grid(h, draw):
    v = _fp16_value(h)
    if not math.isfinite(v):
        return
    assert oracle.sr_fp16_with_rand(v, draw) == h


@SETTINGS
@given(x=st.floats(width=32, min_value=65536.0, allow_infinity=True, allow_nan=False),
       neg=st.booleans(), draw=DRAW)
def test_fp16_rounding_past_the_range_is_infinity(x, neg, draw):
    v = -x if neg else x
    assert oracle.sr_fp16_with_rand(v, draw) == (0xFC00 if neg else 0x7C00)
