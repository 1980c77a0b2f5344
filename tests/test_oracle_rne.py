"""Pins for the oracle's FP32 -> BF16 round-to-nearest-even cast.

Each test checks the oracle against something other than itself:
  * the pages' worked values at theta = 1 (tests/golden/rne_worked_values.txt);
  * IEEE-754 special cases derived by hand in the comments below;
  * exact rational rounding (nearest of the two neighbouring BF16 values,
    ties to the even pattern) computed in float64, where every quantity
    involved is exact;
  * torch's CPU cast ``.to(torch.bfloat16)`` on all 2^32 FP32 patterns
    (NaN excluded; the oracle maps every NaN to 0x7FC0).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rne_worked_values.txt")


def _read_golden(path):
    rows = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split(None, 2)
            rows.append((int(parts[0], 16), int(parts[1], 16), parts[2] if len(parts) > 2 else ""))
    return rows


def test_worked_values_from_the_talk():
    rows = _read_golden(GOLDEN)
    assert len(rows) >= 8
    for f32, bf16, note in rows:
        assert oracle.bf16_rne(f32) == bf16, (hex(f32), hex(bf16), note)


def test_adam_step_is_a_thousand_times_below_the_floor():
    # The talk's arithmetic: boundary 2^-8 at theta=1 versus a 3e-6 step.
    assert 2.0 ** -8 / 3e-6 > 1000
    one = int(np.float32(1.0).view(np.uint32))
    step = int((np.float32(1.0) + np.float32(3e-6)).view(np.uint32))
    assert oracle.bf16_rne(step) == oracle.bf16_rne(one) == 0x3F80


# IEEE-754 special cases (hand-derived):
SPECIAL = [
    (0x00000000, 0x0000),  # +0 keeps its sign
    (0x80000000, 0x8000),  # -0 keeps its sign
    (0x00000001, 0x0000),  # smallest subnormal (2^-149) is far below half of BF16's 2^-133
    (0x80000001, 0x8000),  # ... and keeps the sign of zero
    (0x007FFFFF, 0x0080),  # largest subnormal: remainder 0xFFFF > half, carries into the smallest normal
    (0x00800000, 0x0080),  # smallest normal is exact
    (0x00018000, 0x0002),  # subnormal tie, kept 0x0001 is odd -> up to 0x0002
    (0x00008000, 0x0000),  # subnormal tie, kept 0x0000 is even -> stays
    (0x3F808000, 0x3F80),  # tie at 1 + 2^-8, kept even -> stays
    (0x3F818000, 0x3F82),  # tie, kept 0x3F81 odd -> up
    (0x7F7FFFFF, 0x7F80),  # FLT_MAX is past the midpoint above the largest finite BF16 -> +inf
    (0x7F7F8000, 0x7F80),  # exact midpoint above 0x7F7F; 0x7F7F is odd -> up to +inf
    (0x7F7F7FFF, 0x7F7F),  # just below that midpoint stays finite
    (0xFF7FFFFF, 0xFF80),  # -FLT_MAX -> -inf
    (0x7F800000, 0x7F80),  # +inf
    (0xFF800000, 0xFF80),  # -inf
    (0x7FC00000, 0x7FC0),  # quiet NaN -> canonical
    (0x7F800001, 0x7FC0),  # signalling NaN -> canonical (not infinity)
    (0xFFC00000, 0x7FC0),  # negative NaN -> canonical, sign dropped
    (0x7FFFFFFF, 0x7FC0),  # NaN with all payload bits -> canonical (no carry into the sign)
    (0xFFFFFFFF, 0x7FC0),
]


@pytest.mark.parametrize("f32,bf16", SPECIAL)
def test_ieee_special_cases(f32, bf16):
    assert oracle.bf16_rne(f32) == bf16


def _exact_rne(bits: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even by distance, in float64 (exact for these values).

    For a finite FP32 value v with pattern u, the two BF16 candidates are the
    truncation toward zero (pattern u >> 16) and the next BF16 value away from
    zero; past the largest finite BF16 that neighbour is 2^128 (roundTiesToEven
    with an unbounded exponent), which maps to infinity. The nearer candidate
    wins; on a tie the one whose last pattern bit is 0 wins.
    """
    bits = bits.astype(np.uint32)
    v = bits.view(np.float32).astype(np.float64)
    lo_bits = (bits >> 16).astype(np.uint32)
    hi_bits = lo_bits + 1
    lo = (lo_bits << 16).view(np.float32).astype(np.float64)
    hi_is_inf = (hi_bits & 0x7FFF) == 0x7F80
    hi = np.where(hi_is_inf, np.copysign(2.0 ** 128, v),
                  (hi_bits << 16).astype(np.uint32).view(np.float32).astype(np.float64))
    d_lo = np.abs(v - lo)
    d_hi = np.abs(hi - v)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo_bits & 1) == 1))
    return np.where(pick_hi, hi_bits, lo_bits).astype(np.uint16)


def _finite_only(bits):
    mag = bits & np.uint32(0x7FFFFFFF)
    return bits[mag < np.uint32(0x7F800000)]


def test_exact_rational_rounding_structured():
    # every one of the 65536 upper halves (all signs, binades, mantissas)
    # with the remainders that decide the rounding
    upper = np.arange(1 << 16, dtype=np.uint32) << 16
    rems = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = _finite_only((upper[:, None] | rems[None, :]).reshape(-1))
    np.testing.assert_array_equal(oracle.bf16_rne(bits), _exact_rne(bits))


def test_exact_rational_rounding_random():
    rng = np.random.default_rng(12345)
    bits = _finite_only(rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32))
    np.testing.assert_array_equal(oracle.bf16_rne(bits), _exact_rne(bits))


def _torch_chunk(start: int, size: int):
    bits = np.arange(start, start + size, dtype=np.uint64).astype(np.uint32)
    ours = oracle.bf16_rne(bits)
    ref = torch.from_numpy(bits.view(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = (bits & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    bad_nan = int(np.count_nonzero(ours[nan] != 0x7FC0))
    mism = np.nonzero((ours != ref) & ~nan)[0]
    first = None if mism.size == 0 else (hex(int(bits[mism[0]])), hex(int(ours[mism[0]])), hex(int(ref[mism[0]])))
    return int(mism.size), bad_nan, first


def test_exhaustive_all_fp32_patterns_against_torch_cpu_cast():
    """All 2^32 FP32 patterns: oracle == torch CPU cast on every non-NaN input,
    and every NaN maps to 0x7FC0."""
    chunk = 1 << 25
    starts = range(0, 1 << 32, chunk)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda s: _torch_chunk(s, chunk), starts))
    mism = sum(r[0] for r in results)
    bad_nan = sum(r[1] for r in results)
    firsts = [r[2] for r in results if r[2] is not None]
    assert mism == 0, f"{mism} mismatches, first: {firsts[:3]}"
    assert bad_nan == 0
