"""Pins for the oracle's patch-chain composition (sidecar catch-up).

What fixes the expected results here is independent of the oracle's code:
  * a Python dictionary filled patch by patch (a later patch overwrites), read
    out in sorted order;
  * applying the patches one after another with numpy fancy assignment
    (a library routine) gives the same weights as applying the composition
    once (the talk's "apply the missing transitions", 16:40-17:04);
  * on a chain of real steps (views from torch's BF16 cast, patches by numpy
    comparison) the composition holds every position whose view changed over
    the span, with the final value, and nothing else but positions that
    changed and changed back;
  * associativity, identities and the edge cases (empty, equal, disjoint,
    nested index sets).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _rand_patch(rng, n, k, dtype=np.uint16):
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
    hi = 1 << (8 * np.dtype(dtype).itemsize)
    val = rng.integers(0, hi, size=k).astype(dtype)
    return idx, val


def _dict_compose(patches):
    d = {}
    for idx, val in patches:
        for i, v in zip(idx.tolist(), val.tolist()):
            d[i] = v
    keys = sorted(d)
    return np.array(keys, dtype=np.uint32), np.array([d[k] for k in keys])


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
@pytest.mark.parametrize("seed", range(6))
def test_compose_matches_dictionary(dtype, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 3000))
    chain = [_rand_patch(rng, n, int(rng.integers(0, n + 1)), dtype) for _ in range(int(rng.integers(2, 6)))]
    got_i, got_v = oracle.compose_chain(chain)
    exp_i, exp_v = _dict_compose(chain)
    np.testing.assert_array_equal(got_i, exp_i)
    np.testing.assert_array_equal(got_v, exp_v.astype(dtype))
    assert got_v.dtype == dtype
    assert np.all(np.diff(got_i.astype(np.int64)) > 0)


@pytest.mark.parametrize("seed", range(4))
def test_compose_then_apply_equals_sequential_apply(seed):
    rng = np.random.default_rng(100 + seed)
    n = 5000
    w0 = rng.integers(0, 1 << 16, size=n).astype(np.uint16)
    chain = [_rand_patch(rng, n, int(rng.integers(0, 2000))) for _ in range(5)]
    seq = w0.copy()
    for idx, val in chain:
        seq[idx.astype(np.int64)] = val
    idx, val = oracle.compose_chain(chain)
    once = w0.copy()
    once[idx.astype(np.int64)] = val
    np.testing.assert_array_equal(once, seq)


def _view(master):
    return torch.from_numpy(master).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def test_chain_of_real_steps_covers_the_span():
    n = 1 << 16
    rng = np.random.default_rng(7)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    views = [_view(w)]
    for _ in range(4):
        w = (w + np.float32(3e-5) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
        views.append(_view(w))
    chain = []
    for a, b in zip(views, views[1:]):
        idx = np.nonzero(a != b)[0].astype(np.uint32)
        chain.append((idx, b[idx]))
    idx, val = oracle.compose_chain(chain)
    first, last = views[0], views[-1]
    np.testing.assert_array_equal(val, last[idx])                  # final values
    span = np.nonzero(first != last)[0].astype(np.uint32)
    assert np.isin(span, idx).all()                                 # every change over the span
    extra = np.setdiff1d(idx, span)
    np.testing.assert_array_equal(last[extra], first[extra])       # the rest changed back
    union = np.unique(np.concatenate([p[0] for p in chain]))
    np.testing.assert_array_equal(idx, union)
    assert extra.size > 0   # at this step size some positions do change back


def test_edge_cases():
    e = (np.zeros(0, np.uint32), np.zeros(0, np.uint16))
    a = (np.array([0, 5, 9], np.uint32), np.array([1, 2, 3], np.uint16))
    b = (np.array([5], np.uint32), np.array([7], np.uint16))
    c = (np.array([1, 2, 10, 4000000000], np.uint32), np.array([4, 5, 6, 8], np.uint16))
    for x, y, ei, ev in [
        (e, e, [], []),
        (a, e, [0, 5, 9], [1, 2, 3]),
        (e, a, [0, 5, 9], [1, 2, 3]),
        (a, a, [0, 5, 9], [1, 2, 3]),
        (a, b, [0, 5, 9], [1, 7, 3]),           # nested: the later value wins
        (b, a, [0, 5, 9], [1, 2, 3]),
        (a, c, [0, 1, 2, 5, 9, 10, 4000000000], [1, 4, 5, 2, 3, 6, 8]),   # disjoint
    ]:
        gi, gv = oracle.compose(x, y)
        assert gi.tolist() == ei and gv.tolist() == ev


def test_associative():
    rng = np.random.default_rng(11)
    a, b, c = (_rand_patch(rng, 500, k) for k in (100, 300, 250))
    left = oracle.compose(oracle.compose(a, b), c)
    right = oracle.compose(a, oracle.compose(b, c))
    np.testing.assert_array_equal(left[0], right[0])
    np.testing.assert_array_equal(left[1], right[1])


def test_rejects_mixed_value_types():
    a = (np.array([1], np.uint32), np.array([1], np.uint16))
    b = (np.array([1], np.uint32), np.array([1], np.uint8))
    with pytest.raises(TypeError):
        oracle.compose(a, b)
