"""Pins for the oracle's NVFP4 serving view (E2M1 codes, E4M3 scale per 16
elements, FP32 scale per tensor).

What fixes the expected results here is independent of the oracle's code:
  * the view re-derived with library primitives: numpy float32 arithmetic for
    every scale step (each operation rounded to FP32, in the reading's order),
    torch's CPU float8_e4m3fn cast for the block scale byte and its decode,
    and a brute-force nearest-value search for the E2M1 codes;
  * closed forms: S = 1 when the largest magnitude is 2688; a block reaching
    the tensor maximum gets the largest block scale 448 and its maximum the
    code for 6; NaN blocks, zero blocks and all-zero tensors;
  * the reconstruction invariant apply(encode(old -> new), old) == new view,
    and the pages' claim that coarser views change less.
"""
import math

import numpy as np
import pytest
import torch

import oracle

F = np.float32
MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def brute_e2m1(y: float) -> int:
    if math.isnan(y):
        raise ValueError("no E2M1 code for NaN")
    a = abs(y)
    best = min(range(8), key=lambda c: (abs(MAGS[c] - a), c & 1))
    return best | (0x8 if math.copysign(1.0, y) < 0 else 0)


def e4m3_byte(u: np.float32) -> int:
    """torch's RNE cast to float8_e4m3fn (u <= 448 * (1 + 2^-23) here)."""
    t = torch.tensor([float(u)], dtype=torch.float32).to(torch.float8_e4m3fn)
    return int(t.view(torch.uint8).item())


def e4m3_value(b: int) -> np.float32:
    t = torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    return F(t.item())


def view_reference(master: np.ndarray):
    """The NVFP4 view from library pieces, following the reading step by step."""
    n = master.size
    fin = master[np.isfinite(master)]
    A = F(np.max(np.abs(fin))) if fin.size else F(0.0)
    S = F(A / F(2688.0))
    codes = np.zeros((n + 1) // 2, np.uint8)
    scales = np.zeros((n + 15) // 16, np.uint8)
    for b in range(scales.size):
        blk = master[16 * b:16 * b + 16]
        cs = [0] * blk.size
        if not np.all(np.isfinite(blk)):
            d = 0x7F
        elif S == F(0.0):
            d = 0
        else:
            t = F(F(np.max(np.abs(blk))) / F(6.0))
            u = F(t / S)
            d = e4m3_byte(u)
            if d != 0:
                x = F(e4m3_value(d) * S)
                if x != F(0.0):
                    r = F(F(1.0) / x)
                    if np.isfinite(r):
                        cs = [brute_e2m1(float(F(v * r))) for v in blk]
        scales[b] = d
        for i, c in enumerate(cs):
            e = 16 * b + i
            codes[e // 2] |= c << (4 * (e & 1))
    return codes, scales, S


@pytest.mark.parametrize("n,seed", [(1, 0), (15, 1), (16, 2), (17, 3), (33, 4), (257, 5), (1000, 6)])
def test_quantize_matches_library_derivation(n, seed):
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(n) * 0.02).astype(F)
    m[rng.random(n) < 0.05] = 0.0
    if n > 40:
        m[rng.integers(0, n, 5)] *= F(50.0)   # blocks well below the tensor maximum
    c, s, S = oracle.nvfp4_quantize(m)
    ec, es, eS = view_reference(m)
    assert S == eS
    np.testing.assert_array_equal(s, es)
    np.testing.assert_array_equal(c, ec)


def test_wide_magnitudes_and_specials():
    rng = np.random.default_rng(9)
    n = 16 * 40 + 7
    m = (rng.standard_normal(n) * np.exp2(rng.integers(-60, 20, n))).astype(F)
    m[[3, 100, 200]] = [np.nan, np.inf, -np.inf]
    m[16 * 5:16 * 6] = 0.0
    m[16 * 7:16 * 8] = -0.0
    c, s, S = oracle.nvfp4_quantize(m)
    ec, es, eS = view_reference(m)
    assert S == eS
    np.testing.assert_array_equal(s, es)
    np.testing.assert_array_equal(c, ec)
    assert s[0] == 0x7F and s[100 // 16] == 0x7F and s[200 // 16] == 0x7F
    assert s[5] == 0 and s[7] == 0


def test_closed_forms():
    m = np.zeros(32, F)
    m[0] = 2688.0          # S = 1, block scale 448, code 6
    m[1] = -1344.0         # half the block maximum: 3 -> code 0xD with sign
    m[16] = 6.0            # small block: (6 / 6) / 1 = 1 -> block scale 1.0 (0x38)
    m[17] = 1.5
    c, s, S = oracle.nvfp4_quantize(m)
    assert S == F(1.0)
    assert s[0] == 0x7E and s[1] == 0x38
    assert c[0] == (0x7 | (0xD << 4))
    assert c[8] == (0x7 | (0x3 << 4))
    # an all-zero tensor has S = 0, every scale 0 and every code 0
    z, zs, zS = oracle.nvfp4_quantize(np.zeros(40, F))
    assert zS == F(0.0) and not z.any() and not zs.any()


def test_tensor_scale_ignores_non_finite_values():
    m = np.array([1.0, np.nan, -5376.0, np.inf], F)
    assert oracle.nvfp4_tensor_scale(m) == F(2.0)


@pytest.mark.parametrize("n,eta", [(16, 1e-2), (1000, 1e-3), (4096 + 9, 3e-6)])
def test_encode_matches_definition_and_reconstructs(n, eta):
    rng = np.random.default_rng(n)
    m0 = (rng.standard_normal(n) * 0.02).astype(F)
    m1 = (m0 + F(eta) * rng.standard_normal(n).astype(F)).astype(F)
    pc, ps, _ = oracle.nvfp4_quantize(m0)
    old_c, old_s = pc.copy(), ps.copy()
    idx, val, sidx, sval, S = oracle.nvfp4_encode(m1, pc, ps)
    nc, ns, nS = oracle.nvfp4_quantize(m1)
    assert S == nS
    np.testing.assert_array_equal(idx, np.flatnonzero(nc != old_c).astype(np.uint32))
    np.testing.assert_array_equal(val, nc[idx])
    np.testing.assert_array_equal(sidx, np.flatnonzero(ns != old_s).astype(np.uint32))
    np.testing.assert_array_equal(sval, ns[sidx])
    np.testing.assert_array_equal(pc, nc)
    np.testing.assert_array_equal(ps, ns)
    rc, rs = old_c.copy(), old_s.copy()
    oracle.apply_u8(rc, idx, val)
    oracle.apply_u8(rs, sidx, sval)
    np.testing.assert_array_equal(rc, nc)
    np.testing.assert_array_equal(rs, ns)
    again = oracle.nvfp4_encode(m1, pc, ps)
    assert all(a.size == 0 for a in again[:4])


def test_nvfp4_view_changes_less_than_bf16_view():
    rng = np.random.default_rng(11)
    n = 1 << 16
    m0 = (rng.standard_normal(n) * 0.02).astype(F)
    m1 = (m0 + F(3e-6) * rng.standard_normal(n).astype(F)).astype(F)
    c, s, _ = oracle.nvfp4_quantize(m0)
    k4 = oracle.nvfp4_encode(m1, c, s)[0].size * 2
    prev = oracle.bf16_rne(m0.view(np.uint32)).astype(np.uint16)
    kb = oracle.encode(m1, prev)[0].size
    assert k4 < kb
