"""Pins for the oracle's codec-friendly index packing (gap + bit-packing).

What fixes the expected results here is independent of the oracle's code:
  * a worked example done by hand (tests/golden/pack_example.txt);
  * numpy for the gaps (np.diff), Python's int.bit_length for the widths,
    np.cumsum for the chunk offsets, and np.unpackbits (little bit order) to
    read every slot back out of the payload;
  * the round trip unpack(pack(idx)) == idx on every size edge and on gaps up
    to 2^32 - 2.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pack_example.txt")


def _golden():
    fields = {}
    for line in open(GOLDEN):
        if line.startswith("#") or ":" not in line:
            continue
        k, v = line.split(":", 1)
        fields[k.strip()] = v.split()
    return fields


def test_hand_worked_example():
    f = _golden()
    idx = np.array([int(x) for x in f["indices"]], np.uint32)
    firsts, widths, chunk_off, payload = oracle.pack_indices(idx)
    assert firsts.tolist() == [int(x) for x in f["firsts"]]
    assert widths.tolist() == [int(x) for x in f["widths"]]
    assert chunk_off.tolist() == [int(x) for x in f["chunk_off"]]
    assert payload.size == int(f["payload_len"][0])
    expected = np.zeros(payload.size, np.uint8)
    for item in f["payload_nonzero"]:
        pos, val = item.split(":")
        expected[int(pos)] = int(val, 16)
    np.testing.assert_array_equal(payload, expected)


def _random_idx(rng, k, mean_gap, big=False):
    gaps = rng.geometric(1.0 / (mean_gap + 1), size=k).astype(np.uint64) - 1
    if big and k > 3:
        gaps[rng.integers(1, k, 3)] = rng.integers(1 << 20, 1 << 29, 3)
    idx = np.cumsum(gaps + 1, dtype=np.uint64) - 1
    assert idx[-1] < (1 << 32) - 1
    return idx.astype(np.uint32)


def _check_layout(idx):
    firsts, widths, chunk_off, payload = oracle.pack_indices(idx)
    k = idx.size
    nb = (k + 127) // 128
    assert firsts.size == nb and widths.size == nb
    assert chunk_off.size == (k + 4095) // 4096
    offs = np.concatenate([[0], np.cumsum(16 * widths.astype(np.uint64))])
    np.testing.assert_array_equal(chunk_off, offs[:-1][::32])
    assert payload.size == offs[-1]
    for i in range(nb):
        blk = idx[128 * i:128 * (i + 1)].astype(np.int64)
        assert firsts[i] == blk[0]
        gaps = np.diff(blk) - 1
        b = int(gaps.max()).bit_length() if gaps.size else 0
        assert widths[i] == b
        if b == 0:
            continue
        o = int(offs[i])
        bits = np.unpackbits(payload[o:o + 16 * b], bitorder="little")
        slots = bits.reshape(128, b).astype(np.int64) @ (1 << np.arange(b, dtype=np.int64))
        np.testing.assert_array_equal(slots[:gaps.size], gaps)
        assert not slots[gaps.size:].any()
    return firsts, widths, chunk_off, payload


@pytest.mark.parametrize("k", [1, 2, 127, 128, 129, 4095, 4096, 4097, 3 * 4096 + 500])
@pytest.mark.parametrize("mean_gap", [0, 3, 12, 1000])
def test_layout_and_round_trip(k, mean_gap):
    rng = np.random.default_rng(k * 31 + mean_gap)
    idx = _random_idx(rng, k, mean_gap, big=(mean_gap == 12))
    parts = _check_layout(idx)
    np.testing.assert_array_equal(oracle.unpack_indices(*parts, k), idx)


def test_extremes():
    idx = np.array([0, 4294967294], np.uint32)          # gap 2^32 - 3: width 32
    firsts, widths, chunk_off, payload = _check_layout(idx)
    assert widths.tolist() == [32]
    np.testing.assert_array_equal(oracle.unpack_indices(firsts, widths, chunk_off, payload, 2), idx)
    dense = np.arange(10000, 20000, dtype=np.uint32)   # consecutive: every width 0
    firsts, widths, chunk_off, payload = _check_layout(dense)
    assert payload.size == 0 and not widths.any()
    np.testing.assert_array_equal(oracle.unpack_indices(firsts, widths, chunk_off, payload, dense.size), dense)
    e = oracle.pack_indices(np.zeros(0, np.uint32))
    assert all(x.size == 0 for x in e)


def test_packing_shrinks_an_encode_patch():
    # indices of an 8%-dense patch: about 6 bits per entry instead of 32
    rng = np.random.default_rng(5)
    idx = np.nonzero(rng.random(1 << 20) < 0.08)[0].astype(np.uint32)
    firsts, widths, chunk_off, payload = oracle.pack_indices(idx)
    packed = payload.size + 4 * firsts.size + widths.size + 8 * chunk_off.size
    assert packed < 0.25 * 4 * idx.size
