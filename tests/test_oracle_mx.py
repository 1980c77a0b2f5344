"""Pins for the oracle's MXFP8 serving view (quantize / encode / apply).

What fixes the expected results here is independent of the oracle's code:
  * an E4M3 decoder written from the format's definition (sign, 4-bit
    exponent with bias 7, 3-bit mantissa, subnormals at exponent 0, no
    infinities, S.1111.111 is NaN): every finite code must encode back to
    itself;
  * torch's CPU ``float8_e4m3fn`` cast (a library routine, round to nearest
    even) for every magnitude up to the saturation point 464 -- torch returns
    NaN past it, where the view clamps to 448;
  * closed forms of the block scale of the OCP MX v1.0 specification (scale
    2^(floor(log2 amax) - 8), limited to 2^-127 .. 2^127) and of the
    saturation rule;
  * the pages' statements: a plain float format hides updates below about
    theta / 2^(mantissa bits + 1) (talk "Taking Reinforcement Learning Cross
    Datacenter", 13:25-13:42), so an FP8 view changes less than the BF16 view
    under the same update (PULSE summary, "Potenziale Futuro");
  * the patch definition built directly from a view computed with numpy and
    torch, and the reconstruction invariant apply(encode(old -> new), old) ==
    new view, bit for bit;
  * brute force over short vectors of special values.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads


def decode_e4m3(code: int) -> float:
    """Value of an E4M3 code from the format's definition (NaN for S.1111.111)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


FINITE_CODES = [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_every_finite_code_encodes_back_to_itself():
    for c in FINITE_CODES:
        assert oracle.e4m3_rne(decode_e4m3(c)) == c, hex(c)


def test_grid_is_the_expected_one():
    # 126 positive finite codes, strictly increasing values, largest 448
    pos = [decode_e4m3(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9 and pos[8] == 2.0 ** -6


def _torch_e4m3(y32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(y32).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _oracle_e4m3(y32: np.ndarray) -> np.ndarray:
    return np.array([oracle.e4m3_rne(float(v)) for v in y32], dtype=np.uint8)


def test_matches_torch_cast_on_midpoints_and_neighbours():
    # every midpoint between neighbouring grid values (ties), and the FP32
    # values just below and above it, for both signs
    pos = [decode_e4m3(c) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])] + [464.0]
    vals = []
    for m in mids:
        m32 = np.float32(m)
        assert float(m32) == m  # midpoints are exact in FP32
        vals += [m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))]
    vals = np.array(vals + [np.float32(v) for v in pos], dtype=np.float32)
    vals = vals[np.abs(vals) <= 464.0]
    vals = np.concatenate([vals, -vals])
    np.testing.assert_array_equal(_oracle_e4m3(vals), _torch_e4m3(vals))


def test_matches_torch_cast_on_random_magnitudes():
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-14.0, math.log2(464.0), 20000)).astype(np.float32)
    sign = rng.choice(np.array([-1.0, 1.0], dtype=np.float32), mag.size)
    y = (mag * sign).astype(np.float32)
    y = y[np.abs(y) <= 464.0]
    np.testing.assert_array_equal(_oracle_e4m3(y), _torch_e4m3(y))


def test_named_ties_go_to_even():
    assert oracle.e4m3_rne(1.0625) == 0x38      # 1 + 1/16: between 1 and 1.125
    assert oracle.e4m3_rne(1.1875) == 0x3A      # between 1.125 and 1.25
    assert oracle.e4m3_rne(2.0 ** -10) == 0x00  # half the smallest subnormal
    assert oracle.e4m3_rne(3 * 2.0 ** -10) == 0x02
    assert oracle.e4m3_rne(7 * 2.0 ** -10) == 0x04
    assert oracle.e4m3_rne(15 * 2.0 ** -10) == 0x08  # up into the smallest normal
    assert oracle.e4m3_rne(464.0) == 0x7E       # between 448 and (absent) 480
    assert oracle.e4m3_rne(-0.0) == 0x80 and oracle.e4m3_rne(0.0) == 0x00


@pytest.mark.parametrize("y", [448.0, 449.0, 463.99, 464.0, 465.0, 480.0, 500.0, 511.9, 1e30, 3.4e38])
def test_saturates_to_448(y):
    assert oracle.e4m3_rne(y) == 0x7E
    assert oracle.e4m3_rne(-y) == 0xFE


def test_plain_float_visibility_floor():
    # at a fixed scale, E4M3 (3 mantissa bits) hides any update below
    # theta / 2^(3 + 1) = half the grid spacing theta / 8 of the binade
    # [theta, 2 theta), and shows one just above it
    for e in range(-6, 8):
        theta = 2.0 ** e
        for m in range(1, 7):
            y = theta * (1 + m / 8)
            c = oracle.e4m3_rne(y)
            floor = theta / 16
            assert oracle.e4m3_rne(y + 0.99 * floor) == c
            assert oracle.e4m3_rne(y - 0.99 * floor) == c
            assert oracle.e4m3_rne(y + 1.01 * floor) == c + 1
            assert oracle.e4m3_rne(y - 1.01 * floor) == c - 1


# ------------------------------------------------------------ block scale

def _scale(vals):
    return oracle.mx_block_scale(np.array(vals, dtype=np.float32))


def test_block_scale_closed_forms():
    assert _scale([1.0]) == 127 - 8
    assert _scale([1.0, -0.5, 0.25]) == 119
    assert _scale([-1.999]) == 119                 # floor(log2) = 0
    assert _scale([2.0]) == 120
    assert _scale([0.02, 0.06, -0.01]) == 127 + (-5) - 8   # 0.06 in [2^-5, 2^-4)
    assert _scale([0.0] * 32) == 0                 # all zero: smallest scale
    assert _scale([-0.0, 0.0]) == 0
    assert _scale([2.0 ** -119]) == 0              # e = -127 exactly
    assert _scale([2.0 ** -118]) == 1
    assert _scale([2.0 ** -120]) == 0              # raised to 2^-127
    assert _scale([1.4e-45]) == 0                  # the smallest FP32 subnormal
    assert _scale([1.5 * 2.0 ** 127]) == 127 + 127 - 8
    assert _scale([3.4028235e38]) == 246           # FLT_MAX
    assert _scale([1.0, np.inf]) == 0xFF
    assert _scale([np.nan, 1.0]) == 0xFF
    assert _scale([-np.inf]) == 0xFF


def _view_codes(vals):
    codes, scales = oracle.mxfp8_quantize(np.array(vals, dtype=np.float32))
    return codes.tolist(), scales.tolist()


def test_quantize_closed_forms():
    assert _view_codes([1.0, 0.5, -1.0]) == ([0x78, 0x70, 0xF8], [119])     # 256, 128, -256
    assert _view_codes([1.75, 0.0]) == ([0x7E, 0x00], [119])                 # 448
    assert _view_codes([1.99, -1.99]) == ([0x7E, 0xFE], [119])               # 509.4 clamps to 448
    assert _view_codes([2.0 ** -130]) == ([0x20], [0])                       # 2^-130 * 2^127 = 1/8
    assert _view_codes([2.0 ** -120]) == ([0x70], [0])                       # 128
    assert _view_codes([-0.0, 0.0]) == ([0x80, 0x00], [0])
    assert _view_codes([1.5 * 2.0 ** 127, 1.0]) == ([0x7C, 0x00], [246])     # 384; 1.0 underflows
    assert _view_codes([1.0, np.inf, -2.0]) == ([0x7F, 0x7F, 0x7F], [0xFF])
    assert _view_codes([np.nan]) == ([0x7F], [0xFF])


def _numpy_torch_view(master: np.ndarray):
    """MXFP8 view computed with numpy's frexp and torch's E4M3 cast."""
    n = master.size
    nb = (n + 31) // 32
    pad = np.zeros(nb * 32, dtype=np.float32)
    pad[:n] = master
    blocks = pad.reshape(nb, 32)
    finite = np.isfinite(blocks).all(axis=1)
    amax = np.where(finite, np.abs(np.where(np.isfinite(blocks), blocks, 0)).max(axis=1), 0.0)
    _, ex = np.frexp(amax.astype(np.float64))
    e = np.where(amax > 0, ex - 1 - 8, -127).clip(-127, 127)
    scales = np.where(finite, e + 127, 255).astype(np.uint8)
    y = blocks.astype(np.float64) * np.exp2(-e.astype(np.float64))[:, None]
    y = np.where(np.isfinite(y), y, 0.0)
    with np.errstate(over="ignore"):  # only in non-finite blocks, overwritten below
        codes = _torch_e4m3(y.astype(np.float32))
    big = np.abs(y) > 464.0
    codes[big] = np.where(y[big] < 0, 0xFE, 0x7E)
    codes[~finite] = 0x7F
    return codes.reshape(-1)[:n].copy(), scales


SIZES = [1, 31, 32, 33, 4095, 4096, 4097, 3 * 4096 + 77]


@pytest.mark.parametrize("n", SIZES)
def test_quantize_matches_numpy_torch_view(n):
    m, _ = workloads.np_pair(n, seed=500 + n)
    codes, scales = oracle.mxfp8_quantize(m)
    ec, es = _numpy_torch_view(m)
    np.testing.assert_array_equal(scales, es)
    np.testing.assert_array_equal(codes, ec)


def test_quantize_matches_on_wide_magnitudes():
    rng = np.random.default_rng(11)
    n = 32 * 2000
    scale = np.exp2(rng.integers(-140, 120, n // 32)).repeat(32)
    m = (rng.standard_normal(n) * scale).astype(np.float32)
    m[::97] = 0.0
    m[5::389] = -0.0
    m[7::1001] = np.nan
    m[9::1703] = -np.inf
    codes, scales = oracle.mxfp8_quantize(m)
    ec, es = _numpy_torch_view(m)
    np.testing.assert_array_equal(scales, es)
    np.testing.assert_array_equal(codes, ec)


# ----------------------------------------------------------------- encode

def _expected_patch(master, prev_codes, prev_scales):
    codes, scales = _numpy_torch_view(master)
    idx = np.nonzero(codes != prev_codes)[0].astype(np.uint32)
    sidx = np.nonzero(scales != prev_scales)[0].astype(np.uint32)
    return (idx, codes[idx], sidx, scales[sidx]), codes, scales


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("eta", [3e-6, 1e-4, 3e-3])
def test_encode_matches_definition_and_reconstructs(n, eta):
    m0, _ = workloads.np_pair(n, seed=600 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=600 + n, eta=eta)
    old_codes, old_scales = _numpy_torch_view(m0)
    prev_c, prev_s = old_codes.copy(), old_scales.copy()
    patch = oracle.mxfp8_encode(m1, prev_c, prev_s)
    (ei, ev, esi, esv), new_c, new_s = _expected_patch(m1, old_codes, old_scales)
    for got, exp in zip(patch, (ei, ev, esi, esv)):
        np.testing.assert_array_equal(got, exp)
    np.testing.assert_array_equal(prev_c, new_c)
    np.testing.assert_array_equal(prev_s, new_s)
    # the receiver holding the old view reconstructs the new one bit for bit
    w_c, w_s = old_codes.copy(), old_scales.copy()
    oracle.mxfp8_apply(w_c, w_s, patch)
    np.testing.assert_array_equal(w_c, new_c)
    np.testing.assert_array_equal(w_s, new_s)
    # a second encode of the same master is empty
    again = oracle.mxfp8_encode(m1, prev_c, prev_s)
    assert all(a.size == 0 for a in again)


def test_scale_change_moves_the_whole_block():
    # the block's largest value crosses a power of two: the scale changes and
    # every non-zero code of the block changes with it ([TALK] 13:45-13:59)
    m0 = np.full(32, 0.01, dtype=np.float32)
    m0[0] = 0.99
    prev_c, prev_s = oracle.mxfp8_quantize(m0)
    assert prev_s.tolist() == [118]
    m1 = m0.copy()
    m1[0] = 1.01
    idx, val, sidx, sval = oracle.mxfp8_encode(m1, prev_c, prev_s)
    assert sidx.tolist() == [0] and sval.tolist() == [119]
    assert idx.tolist() == list(range(32))


def test_fp8_view_changes_less_than_bf16_view():
    n = 1 << 18
    m0, p0 = workloads.np_pair(n, seed=77, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=77, eta=3e-6)
    k_bf16 = oracle.count_changed(m1, p0)
    c0, s0 = oracle.mxfp8_quantize(m0)
    idx, _, _, _ = oracle.mxfp8_encode(m1, c0, s0)
    assert 0 < idx.size < k_bf16 / 4


SPECIALS = np.array([0.0, -0.0, 1.0, -1.0, 1.0625, 1.75, 1.99, 2.0 ** -130, 1e-3,
                     448.0, 3e38, np.inf, np.nan], dtype=np.float32)


def test_brute_force_pairs_of_special_values():
    for a, b in itertools.product(SPECIALS, repeat=2):
        m0 = np.array([a, b], dtype=np.float32)
        for c, d in itertools.product(SPECIALS[::3], repeat=2):
            m1 = np.array([c, d], dtype=np.float32)
            old_c, old_s = _numpy_torch_view(m0)
            prev_c, prev_s = old_c.copy(), old_s.copy()
            patch = oracle.mxfp8_encode(m1, prev_c, prev_s)
            expected, new_c, new_s = _expected_patch(m1, old_c, old_s)
            for got, exp in zip(patch, expected):
                np.testing.assert_array_equal(got, exp)
            np.testing.assert_array_equal(prev_c, new_c)
            np.testing.assert_array_equal(prev_s, new_s)


def test_apply_u8_is_a_plain_scatter():
    rng = np.random.default_rng(3)
    w = rng.integers(0, 256, 1000, dtype=np.uint8)
    idx = np.sort(rng.choice(1000, 300, replace=False)).astype(np.uint32)
    val = rng.integers(0, 256, 300, dtype=np.uint8)
    expected = torch.from_numpy(w.copy())
    expected[torch.from_numpy(idx.astype(np.int64))] = torch.from_numpy(val)
    oracle.apply_u8(w, idx, val)
    np.testing.assert_array_equal(w, expected.numpy())
    with pytest.raises(IndexError):
        oracle.apply_u8(w, np.array([1000], dtype=np.uint32), np.array([1], dtype=np.uint8))
