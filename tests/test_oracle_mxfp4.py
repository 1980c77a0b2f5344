"""Pins for the oracle's MXFP4 serving view (quantize / encode / apply).

What fixes the expected results here is independent of the oracle's code:
  * an E2M1 decoder written from the format's definition (sign, 2-bit
    exponent with bias 1, 1-bit mantissa, subnormal at exponent 0, no
    infinities or NaN): every code must encode back to itself;
  * a brute-force rounding: the nearest of the 8 magnitudes, a tie going to
    the code whose mantissa bit is 0, anything past 6 clamped to 6;
  * a brute-force exponent search for the block scale of the OCP MX v1.0
    specification (2^(floor(log2 amax) - 2), limited to 2^-127 .. 2^127) and
    its closed forms;
  * the pages' statements: a coarser float format hides more of an update
    (talk "Taking Reinforcement Learning Cross Datacenter", 13:25-13:59; PULSE
    summary, "Potenziale Futuro": MXFP4 should be sparser still);
  * the patch definition built from a view decoded and re-derived in numpy,
    and the reconstruction invariant apply(encode(old -> new), old) == new
    view, bit for bit;
  * brute force over short vectors of special values.
"""
import itertools
import math

import numpy as np
import pytest

import oracle

MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # magnitudes of codes 0..7


def decode_e2m1(code: int) -> float:
    """Value of an E2M1 code from the format's definition."""
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * m * 0.5
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


def brute_e2m1(y: float) -> int:
    """Nearest magnitude by exhaustive search; ties to the even code; clamp."""
    a = abs(y)
    best = min(range(8), key=lambda c: (abs(MAGS[c] - a), c & 1))
    return best | (0x8 if math.copysign(1.0, y) < 0 else 0)


def brute_scale(block) -> int:
    """E8M0 byte by searching the exponent: largest k with 2^k <= amax."""
    vals = [float(v) for v in block]
    if any(not math.isfinite(v) for v in vals):
        return 0xFF
    amax = max(abs(v) for v in vals)
    if amax == 0.0:
        return 0
    k = -160
    while 2.0 ** (k + 1) <= amax:
        k += 1
    return min(max(k - 2, -127), 127) + 127


def test_decoder_grid():
    assert [decode_e2m1(c) for c in range(8)] == MAGS
    assert [decode_e2m1(c | 8) for c in range(8)] == [-m for m in MAGS]


def test_every_code_encodes_back_to_itself():
    for c in range(16):
        assert oracle.e2m1_rne(decode_e2m1(c) if c != 8 else -0.0) == c, c


@pytest.mark.parametrize("y", [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
def test_ties_go_to_the_even_code(y):
    for s in (1.0, -1.0):
        got = oracle.e2m1_rne(s * y)
        assert got == brute_e2m1(s * y)
        assert got & 1 == 0  # mantissa bit 0


def test_matches_brute_force_on_random_values():
    rng = np.random.default_rng(0)
    ys = np.concatenate([rng.uniform(-8, 8, 20000), rng.uniform(-1, 1, 5000),
                         np.array([m + d for m in MAGS for d in (-1e-9, 0.0, 1e-9)])])
    for y in ys:
        assert oracle.e2m1_rne(float(y)) == brute_e2m1(float(y)), y


@pytest.mark.parametrize("y", [6.0, 6.5, 7.999, 1e30])
def test_saturates_to_6(y):
    assert oracle.e2m1_rne(y) == 0x7
    assert oracle.e2m1_rne(-y) == 0xF


def test_negative_values_rounding_to_zero_keep_the_sign():
    assert oracle.e2m1_rne(-0.0) == 0x8
    assert oracle.e2m1_rne(-0.1) == 0x8
    assert oracle.e2m1_rne(0.1) == 0x0


def test_block_scale_closed_forms_and_search():
    f = np.float32
    cases = [
        (np.array([6.0], f), 127),            # floor(log2 6) = 2 -> 2^0
        (np.array([4.0, -7.99], f), 127),
        (np.array([3.99], f), 126),
        (np.array([6.0 * 2 ** 10], f), 137),
        (np.array([0.0, -0.0], f), 0),         # all zero: the smallest scale
        (np.array([1e-40], f), 0),             # subnormal maximum: raised to 2^-127
        (np.array([3e38], f), 127 + 125),      # floor(log2 3e38) = 127
        (np.array([1.0, np.nan], f), 0xFF),
        (np.array([np.inf], f), 0xFF),
        (np.array([-np.inf, 2.0], f), 0xFF),
    ]
    for block, want in cases:
        assert oracle.mxfp4_block_scale(block) == want, block
        assert brute_scale(block) == want, block
    rng = np.random.default_rng(1)
    for _ in range(2000):
        blk = (rng.standard_normal(int(rng.integers(1, 33))) *
               10.0 ** rng.uniform(-30, 30)).astype(f)
        assert oracle.mxfp4_block_scale(blk) == brute_scale(blk)


def _view_numpy(master: np.ndarray):
    """The MXFP4 view from brute-force pieces: per block the searched scale,
    per element the brute-force code of v / 2^(s - 127), packed two per byte."""
    n = master.size
    codes = np.zeros((n + 1) // 2, np.uint8)
    scales = np.zeros((n + 31) // 32, np.uint8)
    for b in range(scales.size):
        blk = master[32 * b:32 * b + 32]
        s = brute_scale(blk)
        scales[b] = s
        for i, v in enumerate(blk):
            c = 0 if s == 0xFF else brute_e2m1(float(v) * 2.0 ** (127 - s))
            e = 32 * b + i
            codes[e // 2] |= c << (4 * (e & 1))
    return codes, scales


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 63, 64, 65, 257])
def test_quantize_matches_brute_force_view(n):
    rng = np.random.default_rng(n)
    m = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m[rng.random(n) < 0.05] = 0.0
    codes, scales = oracle.mxfp4_quantize(m)
    ec, es = _view_numpy(m)
    np.testing.assert_array_equal(codes, ec)
    np.testing.assert_array_equal(scales, es)


def test_quantize_special_blocks():
    f = np.float32
    m = np.concatenate([np.zeros(32, f), np.full(32, np.nan, f), np.array([np.inf] + [1.0] * 31, f),
                        np.array([1e-42] * 32, f), np.array([-5.0, 5.0, 6.0, -6.0] * 8, f)])
    codes, scales = oracle.mxfp4_quantize(m)
    assert scales[0] == 0 and np.all(codes[0:16] == 0)
    assert scales[1] == 0xFF and np.all(codes[16:32] == 0)
    assert scales[2] == 0xFF and np.all(codes[32:48] == 0)
    assert scales[3] == 0  # subnormal block maximum: scale 2^-127, values round to 0
    # amax 6 -> scale 2^0: -5 -> -4 (tie to even), 5 -> 4, 6 -> 6, -6 -> -6
    assert scales[4] == 127
    assert list(codes[64:66]) == [0x6E, 0xF7]


def test_reconstruction_error_is_within_half_a_grid_step():
    """Every finite element decodes to the nearest grid value of its block
    (or to +-6 times the scale when it was clamped)."""
    rng = np.random.default_rng(4)
    m = (rng.standard_normal(32 * 200) * 10.0 ** rng.uniform(-3, 3, 32 * 200)).astype(np.float32)
    codes, scales = oracle.mxfp4_quantize(m)
    for i, v in enumerate(m):
        s = int(scales[i // 32])
        c = (int(codes[i // 2]) >> (4 * (i & 1))) & 0xF
        x = 2.0 ** (s - 127)
        y = float(v) / x
        got = decode_e2m1(c)
        assert abs(got - y) <= min(abs(mg - abs(y)) for mg in MAGS) + 1e-12
        assert abs(y) < 8.0  # the block scale keeps every element below 2^3


@pytest.mark.parametrize("n,eta", [(1, 1e-3), (33, 1e-2), (4096 + 17, 3e-6), (5000, 1e-3)])
def test_encode_matches_definition_and_reconstructs(n, eta):
    rng = np.random.default_rng(n)
    m0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m1 = (m0 + np.float32(eta) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
    pc, ps = oracle.mxfp4_quantize(m0)
    old_c, old_s = pc.copy(), ps.copy()
    idx, val, sidx, sval = oracle.mxfp4_encode(m1, pc, ps)
    nc, ns = oracle.mxfp4_quantize(m1)
    # the definition: changed bytes / scales in ascending order
    np.testing.assert_array_equal(idx, np.flatnonzero(nc != old_c).astype(np.uint32))
    np.testing.assert_array_equal(val, nc[idx])
    np.testing.assert_array_equal(sidx, np.flatnonzero(ns != old_s).astype(np.uint32))
    np.testing.assert_array_equal(sval, ns[sidx])
    # refreshed previous view, and apply on a receiver reconstructs the view
    np.testing.assert_array_equal(pc, nc)
    np.testing.assert_array_equal(ps, ns)
    rc, rs = old_c.copy(), old_s.copy()
    oracle.mxfp4_apply(rc, rs, (idx, val, sidx, sval))
    np.testing.assert_array_equal(rc, nc)
    np.testing.assert_array_equal(rs, ns)
    # encoding the same master again changes nothing
    again = oracle.mxfp4_encode(m1, pc, ps)
    assert all(a.size == 0 for a in again)


def test_odd_length_pads_the_last_high_nibble_with_zero():
    m = np.array([1.0, -1.0, 6.0], np.float32)
    codes, scales = oracle.mxfp4_quantize(m)
    assert scales[0] == 127 and list(codes) == [0xA2, 0x07]
    # garbage in a previous padding nibble is a change of that byte
    pc, ps = codes.copy(), scales.copy()
    pc[1] |= 0x50
    idx, val, sidx, sval = oracle.mxfp4_encode(m, pc, ps)
    assert list(idx) == [1] and list(val) == [0x07] and sidx.size == 0


def test_fp4_view_changes_less_than_fp8_and_bf16_views():
    """Coarser cells hide more of the same update (pages: FP8 and MXFP4 views
    should be sparser than BF16)."""
    rng = np.random.default_rng(9)
    n = 1 << 16
    m0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m1 = (m0 + np.float32(3e-6) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
    c4, s4 = oracle.mxfp4_quantize(m0)
    k4 = oracle.mxfp4_encode(m1, c4, s4)[0].size * 2       # bytes -> at most 2 elements each
    c8, s8 = oracle.mxfp8_quantize(m0)
    k8 = oracle.mxfp8_encode(m1, c8, s8)[0].size
    prev = oracle.bf16_rne(m0.view(np.uint32)).astype(np.uint16)
    kb = oracle.encode(m1, prev)[0].size
    assert k4 < k8 < kb


def test_brute_force_pairs_of_special_values():
    specials = [0.0, -0.0, 0.25, -0.75, 1.0, 5.0, 6.0, 100.0, 1e-40, np.nan, np.inf, -np.inf]
    for a, b in itertools.product(specials, repeat=2):
        m = np.array([a, b], np.float32)
        codes, scales = oracle.mxfp4_quantize(m)
        ec, es = _view_numpy(m)
        assert codes[0] == ec[0] and scales[0] == es[0], (a, b)
