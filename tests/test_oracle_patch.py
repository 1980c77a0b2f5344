"""Pins for the oracle's encode / apply / XOR mask / XOR apply.

What fixes the expected results here is independent of the oracle's code:
  * torch's CPU cast gives the new BF16 view (``_view``), NaN -> 0x7FC0;
  * the definition of the patch (changed positions, ascending, with the new
    absolute value) is built directly from that view with numpy;
  * the pages' invariants: apply(encode(old -> new), old) is the new view bit
    for bit; re-encoding the same weights and eta = 0 give an empty patch;
    a double XOR restores the original and XOR-ing the mask into the old view
    gives the new one; an update smaller than about |w|/256 leaves the view
    unchanged;
  * brute force over every vector of length <= 2 (and a subset of length 3)
    drawn from a set of special values.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads


def _view(master: np.ndarray) -> np.ndarray:
    """New BF16 view by torch's CPU cast; every NaN becomes 0x7FC0."""
    out = torch.from_numpy(np.ascontiguousarray(master)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    nan = np.isnan(master)
    out[nan] = 0x7FC0
    return out


def _expected_patch(master, prev):
    b = _view(master)
    idx = np.nonzero(b != prev)[0].astype(np.uint32)
    return idx, b[idx], b


SIZES = [0, 1, 7, 8, 9, 4095, 4096, 4097, 65536 + 3]


@pytest.mark.parametrize("n", SIZES)
def test_encode_matches_definition(n):
    master, prev = workloads.np_pair(n, seed=100 + n)
    old = prev.copy()
    e_idx, e_val, b = _expected_patch(master, prev)
    idx, val = oracle.encode(master, prev)
    np.testing.assert_array_equal(idx, e_idx)
    np.testing.assert_array_equal(val, e_val)
    np.testing.assert_array_equal(prev, b)            # prev refreshed to the new view
    # structural: strictly ascending, every entry a real change
    assert np.all(np.diff(idx.astype(np.int64)) > 0)
    assert np.all(val != old[idx])
    assert oracle.count_changed(master, old) == idx.size


@pytest.mark.parametrize("n", [1, 4097, 1 << 16])
def test_reconstruction_is_bit_identical(n):
    # Talk 11:14-11:30 and PULSE "1. PULSESync": applying the patch of
    # absolute values to the old view gives exactly the new checkpoint.
    master, prev = workloads.np_pair(n, seed=7)
    receiver = prev.copy()
    idx, val = oracle.encode(master, prev)
    oracle.apply(receiver, idx, val)
    np.testing.assert_array_equal(receiver, _view(master))
    np.testing.assert_array_equal(receiver, prev)


def test_reencode_same_weights_is_empty_and_eta_zero_is_empty():
    master, prev = workloads.np_pair(1 << 14, seed=3)
    oracle.encode(master, prev)
    before = prev.copy()
    idx, val = oracle.encode(master, prev)
    assert idx.size == 0 and val.size == 0
    np.testing.assert_array_equal(prev, before)
    # eta = 0: master is exactly w0 and prev is its torch cast
    m0, p0 = workloads.np_pair(1 << 14, seed=5, eta=0.0)
    keep = p0.copy()
    idx, _ = oracle.encode(m0, p0)
    assert idx.size == 0
    np.testing.assert_array_equal(p0, keep)


def test_apply_equals_numpy_fancy_index_assignment():
    rng = np.random.default_rng(11)
    w = rng.integers(0, 1 << 16, size=5000, dtype=np.uint64).astype(np.uint16)
    idx = np.sort(rng.choice(5000, size=700, replace=False)).astype(np.uint32)
    val = rng.integers(0, 1 << 16, size=700, dtype=np.uint64).astype(np.uint16)
    ref = w.copy()
    ref[idx] = val
    oracle.apply(w, idx, val)
    np.testing.assert_array_equal(w, ref)


def test_apply_later_entry_wins_on_duplicate_index():
    w = np.zeros(4, dtype=np.uint16)
    oracle.apply(w, np.array([2, 2], dtype=np.uint32), np.array([5, 9], dtype=np.uint16))
    assert list(w) == [0, 0, 9, 0]


@pytest.mark.parametrize("n", [0, 1, 9, 4097, 1 << 15])
def test_xor_mask_and_apply(n):
    # humansand.ai summary, "XOR maskeleri ile delta senkronizasyonu":
    # mask = old XOR new; the old weights XOR the mask give the new weights;
    # the XOR acts on raw bits.
    master, prev = workloads.np_pair(n, seed=21)
    old = prev.copy()
    b = _view(master)
    mask = oracle.xor_mask(master, prev)
    np.testing.assert_array_equal(mask, old ^ b)
    np.testing.assert_array_equal(prev, b)
    w = old.copy()
    oracle.xor_apply(w, mask)
    np.testing.assert_array_equal(w, b)               # old ^ mask == new
    oracle.xor_apply(w, mask)
    np.testing.assert_array_equal(w, old)             # double XOR restores
    # cross-mode: non-zero mask words are exactly the patch positions
    p2 = old.copy()
    idx, _ = oracle.encode(master, p2)
    np.testing.assert_array_equal(np.nonzero(mask)[0].astype(np.uint32), idx)


# ------------------------------------------------------------- brute force

# FP32 special values (bit patterns)
S_MASTER = [0x00000000, 0x80000000, 0x00000001, 0x007FFFFF, 0x00800000,
            0x7F7FFFFF, 0x7F7F7FFF, 0x7F800000, 0xFF800000, 0x7FC00000,
            0x7F800001, 0xFFC00000, 0x3F808000, 0x3F818000, 0x00018000,
            0x3F800000, 0xBF800000, 0x3F800019]
# BF16 prev values (bit patterns)
S_PREV = [0x0000, 0x8000, 0x0001, 0x0002, 0x0080, 0x7F7F, 0x7F80, 0xFF80,
          0x7FC0, 0x7FFF, 0x3F80, 0x3F81, 0x3F82, 0xBF80]


def _torch_view_bits(bits):
    arr = np.array(bits, dtype=np.uint32).view(np.float32)
    return _view(arr)


def _brute(cases_master, cases_prev):
    view_of = dict(zip(S_MASTER, (int(x) for x in _torch_view_bits(S_MASTER))))
    bad = 0
    for mb, pv in zip(cases_master, cases_prev):
        master = np.array(mb, dtype=np.uint32).view(np.float32)
        prev = np.array(pv, dtype=np.uint16)
        b = [view_of[x] for x in mb]
        e_idx = [i for i in range(len(mb)) if b[i] != pv[i]]
        e_val = [b[i] for i in e_idx]
        idx, val = oracle.encode(master, prev)
        if list(idx) != e_idx or list(val) != e_val or list(prev) != b:
            bad += 1
        # mask of the same step
        p2 = np.array(pv, dtype=np.uint16)
        mask = oracle.xor_mask(master, p2)
        if list(mask) != [b[i] ^ pv[i] for i in range(len(mb))]:
            bad += 1
    return bad


def test_bruteforce_length_1_and_2():
    pairs = list(itertools.product(S_MASTER, S_PREV))
    cm, cp = [], []
    for (m, p) in pairs:
        cm.append((m,))
        cp.append((p,))
    for (m1, p1), (m2, p2) in itertools.product(pairs, repeat=2):
        cm.append((m1, m2))
        cp.append((p1, p2))
    assert len(cm) == len(pairs) + len(pairs) ** 2
    assert _brute(cm, cp) == 0


def test_bruteforce_length_3_subset():
    sm = [0x80000000, 0x00018000, 0x7F7FFFFF, 0x7F800001, 0x3F808000, 0x3F818000]
    sp = [0x0000, 0x8000, 0x7FC0, 0x3F80, 0x3F82]
    pairs = list(itertools.product(sm, sp))
    cm, cp = [], []
    for trip in itertools.product(pairs, repeat=3):
        cm.append(tuple(t[0] for t in trip))
        cp.append(tuple(t[1] for t in trip))
    assert _brute(cm, cp) == 0


# ------------------------------------------------------- visibility floor

def _bf16_grid_values(rng, count):
    """Random finite, normal BF16 values (as float64) away from the overflow edge."""
    sign = rng.integers(0, 2, size=count, dtype=np.uint32) << 15
    exp = rng.integers(1 + 8, 254 - 8, size=count, dtype=np.uint32) << 7
    man = rng.integers(0, 128, size=count, dtype=np.uint32)
    # include exact powers of two (mantissa 0) where the lower gap halves
    man[: count // 4] = 0
    bits = (sign | exp | man).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64), (bits >> 16).astype(np.uint16)


def test_update_below_the_floor_is_invisible_and_above_is_visible():
    # PULSE "Osservazione Centrale": updates below about |w|/256 are absorbed
    # by the BF16 cast; the talk (07:36-08:00) puts the floor at half a ULP.
    # For w on the BF16 grid the half-gap to either neighbour lies in
    # [|w|/512, |w|/256], so |d| < |w|/512 never changes the view and
    # |d| > |w|/256 always does.
    rng = np.random.default_rng(2024)
    w, wbits = _bf16_grid_values(rng, 20000)
    frac = rng.uniform(0.0, 0.999, size=w.size)
    sgn = np.where(rng.integers(0, 2, size=w.size) == 0, -1.0, 1.0)
    small = (w + sgn * frac * np.abs(w) / 512).astype(np.float32)
    prev = wbits.copy()
    idx, _ = oracle.encode(small, prev)
    assert idx.size == 0
    big = (w + sgn * (1.001 + frac) * np.abs(w) / 256).astype(np.float32)
    prev = wbits.copy()
    idx, _ = oracle.encode(big, prev)
    assert idx.size == w.size


def test_exact_floor_is_half_the_gap_in_the_update_direction():
    # the exact reading: invisible iff w + d stays on w's side of the
    # rounding midpoint toward the neighbour in d's direction
    rng = np.random.default_rng(99)
    w, wbits = _bf16_grid_values(rng, 4000)
    up_bits = (wbits.astype(np.uint32) + 1) << 16
    dn_bits = (wbits.astype(np.uint32) - 1) << 16
    up = up_bits.astype(np.uint32).view(np.float32).astype(np.float64)
    dn = dn_bits.astype(np.uint32).view(np.float32).astype(np.float64)
    for toward, nb in ((+1, up), (-1, dn)):
        half = np.abs(nb - w) / 2
        inside = (w + toward * np.sign(w) * 0.98 * half).astype(np.float32)
        outside = (w + toward * np.sign(w) * 1.02 * half).astype(np.float32)
        p = wbits.copy()
        assert oracle.encode(inside, p)[0].size == 0
        p = wbits.copy()
        assert oracle.encode(outside, p)[0].size == w.size


# ---------------------------------------------------------- chain / multi

def _small_model_specs():
    # a miniature of the Qwen2.5 layout (tiny tensors, biases, norms)
    return [workloads.TensorSpec("emb", (97, 16), "weight")] + [
        workloads.TensorSpec(f"l{i}.{nm}", shp, kind)
        for i in range(2)
        for nm, shp, kind in (("q", (16, 16), "weight"), ("qb", (16,), "bias"),
                              ("k", (4, 16), "weight"), ("kb", (4,), "bias"),
                              ("gate", (40, 16), "weight"), ("ln", (16,), "norm"))
    ] + [workloads.TensorSpec("norm", (16,), "norm")]


@pytest.mark.parametrize("eta", [3e-6, 1e-4])
def test_twenty_step_chain_receiver_stays_bit_identical(eta):
    # Talk 11:19-11:30: patches are bit-level replacements, not floating-point
    # additions, so a chain of them does not drift. Both modes, every step.
    specs = _small_model_specs()
    rng = np.random.default_rng(4)
    masters = [workloads.np_init(s, rng) for s in specs]
    trainer_p = [workloads.np_bf16_view_torch(m) for m in masters]
    trainer_x = [p.copy() for p in trainer_p]
    recv_p = [p.copy() for p in trainer_p]
    recv_x = [p.copy() for p in trainer_p]
    total_changed = 0
    for step in range(workloads.CHAIN_STEPS):
        srng = np.random.default_rng(workloads.CHAIN_SEED_BASE + step)
        masters = [workloads.np_update(m, eta, srng) for m in masters]
        patches = oracle.encode_multi(masters, trainer_p)
        oracle.apply_multi(recv_p, patches)
        masks = oracle.xor_mask_multi(masters, trainer_x)
        oracle.xor_apply_multi(recv_x, masks)
        for m, tp, tx, rp, rx, (idx, _), mk in zip(masters, trainer_p, trainer_x, recv_p, recv_x, patches, masks):
            full = _view(m)                       # what a full checkpoint would carry
            np.testing.assert_array_equal(tp, full)
            np.testing.assert_array_equal(tx, full)
            np.testing.assert_array_equal(rp, full)
            np.testing.assert_array_equal(rx, full)
            assert np.count_nonzero(mk) == idx.size
            total_changed += idx.size
    assert total_changed > 0


@pytest.mark.parametrize("n,parts", [(0, 4), (1, 4), (4097, 3), (1 << 16, 7), (1 << 16, 64)])
def test_chunked_encode_and_apply_equal_the_single_thread_oracle(n, parts):
    # The all-cores CPU baseline runs the same scalar loops on contiguous
    # chunks (count pass, scan, emit pass); its patch must be the definition's.
    from concurrent.futures import ThreadPoolExecutor
    master, prev = workloads.np_pair(n, seed=300 + n)
    old = prev.copy()
    e_idx, e_val, b = _expected_patch(master, prev)
    with ThreadPoolExecutor(max_workers=4) as pool:
        idx, val = oracle.encode_chunked(master, prev, pool, parts)
        np.testing.assert_array_equal(idx, e_idx)
        np.testing.assert_array_equal(val, e_val)
        np.testing.assert_array_equal(prev, b)
        w = old.copy()
        oracle.apply_chunked(w, idx, val, pool, parts)
    np.testing.assert_array_equal(w, b)
