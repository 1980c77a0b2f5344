"""Pins for the oracle's PULSELoCo gate with FP32 error feedback.

What fixes the expected results here is independent of the oracle's code:
  * numpy FP32 arithmetic (IEEE, one rounding per operation) for the
    pseudo-gradient and the error-feedback sum (a NaN sum stored as the quiet
    NaN 0x7FC00000), and torch's CPU BF16 cast (every NaN read as 0x7FC0)
    for the visibility test, on random and special-value inputs;
  * conservation: for every entry, the value sent (or 0) plus the new error
    equals pseudo-gradient + old error, bit for bit (nothing is lost or
    created, PULSE summary "2. PULSELoCo": what does not pass is kept);
  * the BF16 visibility floor at theta = 1 (boundary 2^-8, tie to even);
  * a sub-threshold update repeated each round is sent in the round where
    the accumulated error first crosses the boundary (closed form);
  * numpy's np.add.at (a library routine) for the receiver's accumulation.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle


def _bf16(x: np.ndarray) -> np.ndarray:
    out = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    out[np.isnan(x)] = 0x7FC0
    return out


def _expected(g, w, e):
    with np.errstate(all="ignore"):
        u = (w - g) + e                      # numpy float32: one rounding per op
        u[np.isnan(u)] = np.uint32(0x7FC00000).view(np.float32)   # the quiet NaN
        s = g + u
    passed = _bf16(s) != _bf16(g)
    idx = np.nonzero(passed)[0].astype(np.uint32)
    e_new = np.where(passed, np.float32(0.0), u).astype(np.float32)
    return idx, u[idx], e_new, u


def _same_bits(a, b):
    np.testing.assert_array_equal(np.asarray(a, np.float32).view(np.uint32),
                                  np.asarray(b, np.float32).view(np.uint32))


@pytest.mark.parametrize("n,seed,scale", [(1, 0, 1e-3), (1000, 1, 1e-4), (4097, 2, 3e-5), (65539, 3, 1e-5)])
def test_gate_matches_numpy_and_torch(n, seed, scale):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    w = (g + rng.standard_normal(n).astype(np.float32) * np.float32(scale)).astype(np.float32)
    e = (rng.standard_normal(n) * scale * 0.3).astype(np.float32)
    ei, ev, e_new, _ = _expected(g, w, e)
    err = e.copy()
    idx, val = oracle.loco_gate(g, w, err)
    np.testing.assert_array_equal(idx, ei)
    _same_bits(val, ev)
    _same_bits(err, e_new)
    assert 0 < idx.size < n or n == 1


def test_conservation_is_exact():
    rng = np.random.default_rng(9)
    n = 20000
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    w = (g + rng.standard_normal(n).astype(np.float32) * np.float32(2e-5)).astype(np.float32)
    e = (rng.standard_normal(n) * 1e-5).astype(np.float32)
    _, _, _, u = _expected(g, w, e)
    err = e.copy()
    idx, val = oracle.loco_gate(g, w, err)
    sent = np.zeros(n, np.float32)
    sent[idx.astype(np.int64)] = val
    total = np.where(np.isin(np.arange(n), idx), sent, err)
    _same_bits(total, u)
    assert np.all(err[idx.astype(np.int64)] == 0)


def test_visibility_floor_at_one():
    g = np.ones(5, np.float32)
    half = 2.0 ** -8                       # half a BF16 ULP at theta = 1
    w = np.array([1.0 + 0.9 * half, 1.0 + half, 1.0 + 1.1 * half, 1.0 - 0.45 * half, 1.0 - 0.55 * half],
                 np.float32)
    err = np.zeros(5, np.float32)
    idx, _ = oracle.loco_gate(g, w, err)
    # +half is a tie that rounds to even (1.0): not visible; below 1 the
    # spacing halves, so -0.55 * half crosses the lower midpoint
    assert idx.tolist() == [2, 4]


def test_sub_threshold_update_is_sent_once_accumulated():
    g = np.ones(1, np.float32)
    w = np.array([1.001], np.float32)      # 0.001 < 2^-8 = 0.0039: invisible alone
    err = np.zeros(1, np.float32)
    sent_round = None
    for r in range(1, 8):
        idx, val = oracle.loco_gate(g, w, err)
        if idx.size:
            sent_round = r
            assert val[0] > 2.0 ** -8
            assert err[0] == 0
            break
    d = np.float32(1.001) - np.float32(1.0)
    assert sent_round == int(np.ceil(2.0 ** -8 / float(d)))   # 4 rounds of ~0.000999


SPECIALS = np.array([0.0, -0.0, 1.0, -1.0, 1e-40, -1e-40, 3e38, np.inf, -np.inf, np.nan, 0.0039, 1.00390625],
                    np.float32)


def test_brute_force_special_values():
    for gv, wv, ev in itertools.product(SPECIALS, SPECIALS, SPECIALS[::2]):
        g = np.array([gv], np.float32)
        w = np.array([wv], np.float32)
        e = np.array([ev], np.float32)
        ei, evals, e_new, _ = _expected(g, w, e)
        err = e.copy()
        idx, val = oracle.loco_gate(g, w, err)
        np.testing.assert_array_equal(idx, ei)
        _same_bits(val, evals)
        _same_bits(err, e_new)


def test_accumulate_matches_add_at():
    rng = np.random.default_rng(4)
    acc = rng.standard_normal(3000).astype(np.float32)
    idx = np.sort(rng.choice(3000, 700, replace=False)).astype(np.uint32)
    val = rng.standard_normal(700).astype(np.float32)
    exp = acc.copy()
    np.add.at(exp, idx.astype(np.int64), val)
    oracle.loco_accumulate(acc, idx, val)
    _same_bits(acc, exp)
