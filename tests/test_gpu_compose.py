"""GPU vs oracle for patch-chain composition through the C ABI: random
patches across many tiles (shared indices straddling tile edges, nested,
disjoint and identical index sets), both value widths, chains of real encode
patches, and the multi-segment form. Every comparison is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_u32, host_u32

pytestmark = pytest.mark.gpu

TILE = 2048  # merged positions per compose tile


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _rand_patch(rng, n, k, dtype):
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32)
    hi = 1 << (8 * np.dtype(dtype).itemsize)
    return idx, rng.integers(0, hi, size=k).astype(dtype)


def _to_dev(p, dev):
    idx, val = p
    t_idx = dev_u32(idx, dev) if idx.size else torch.empty(0, dtype=torch.int32, device=dev)
    tv = torch.from_numpy(val.view(np.int16) if val.dtype == np.uint16 else val).to(dev)
    return t_idx, tv


def _host_val(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == np.uint16 else a.view(np.uint8)


def _gpu_compose(a, b, dev):
    ia, va = _to_dev(a, dev)
    ib, vb = _to_dev(b, dev)
    cap = max(a[0].size + b[0].size, 1)
    gi, gv = Guarded(cap, torch.int32, dev), Guarded(cap, va.dtype, dev)
    gc = Guarded(1, torch.int64, dev)
    idx, val, cnt = pulse.compose(ia, va, a[0].size, ib, vb, b[0].size, gi.t, gv.t, gc.t)
    k = int(cnt.item())
    for name, g in (("idx", gi), ("val", gv), ("count", gc)):
        g.check(name)
    return host_u32(idx[:k]), _host_val(val[:k], a[1].dtype)


def _check(a, b, dev):
    gi, gv = _gpu_compose(a, b, dev)
    oi, ov = oracle.compose(a, b)
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov)
    return oi.size


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
@pytest.mark.parametrize("ka,kb,n", [(1, 0, 10), (0, 1, 10), (5, 7, 12), (TILE, TILE, 3 * TILE),
                                     (3 * TILE + 5, 2 * TILE - 3, 6 * TILE),
                                     (40000, 35000, 100000), (200000, 1000, 10 ** 9)])
def test_random_patches(dtype, ka, kb, n):
    dev = _dev()
    rng = np.random.default_rng(ka * 7 + kb)
    _check(_rand_patch(rng, n, ka, dtype), _rand_patch(rng, n, kb, dtype), dev)


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_structured_index_sets(dtype):
    dev = _dev()
    rng = np.random.default_rng(5)
    n = 50000
    a = _rand_patch(rng, n, 20000, dtype)
    same = (a[0].copy(), rng.integers(0, 200, size=a[0].size).astype(dtype))
    assert _check(a, same, dev) == a[0].size                      # identical: B wins everywhere
    sub = (a[0][::3].copy(), a[1][::3].copy())
    _check(a, sub, dev)                                          # nested
    _check(sub, a, dev)
    evens = (np.arange(0, 2 * 9000, 2, dtype=np.uint32), np.ones(9000, dtype))
    odds = (np.arange(1, 2 * 9000, 2, dtype=np.uint32), np.full(9000, 2, dtype))
    assert _check(evens, odds, dev) == 18000                     # interleaved, disjoint
    # shared indices placed exactly at the tile edges of the merged order
    idx = np.arange(0, 4 * TILE, dtype=np.uint32) * 3
    a2 = (idx, np.zeros(idx.size, dtype))
    b2 = (idx[TILE // 2 - 1::TILE // 2].copy(), np.ones(idx[TILE // 2 - 1::TILE // 2].size, dtype))
    _check(a2, b2, dev)
    _check((np.zeros(0, np.uint32), np.zeros(0, dtype)), (np.zeros(0, np.uint32), np.zeros(0, dtype)), dev)


def test_chain_of_encode_patches_then_apply():
    """Four consecutive steps of one Llama decoder-layer tensor, encoded on
    the GPU; the composed patch applied once equals the final view."""
    dev = _dev()
    spec = workloads.llama_layer()[4]            # gate_proj, 58.7M params
    gen = workloads.torch_generator(dev, 31)
    w = torch.empty(spec.numel, dtype=torch.float32, device=dev)
    workloads.torch_init_(w, spec, gen)
    prev = torch.empty(spec.numel, dtype=torch.int16, device=dev)
    workloads.torch_bf16_view_(prev, w)
    view0 = prev.clone()
    patches = []
    for step in range(4):
        workloads.torch_update_(w, 3e-5, gen)
        idx, val, cnt = pulse.encode(w, prev)
        k = int(cnt.item())
        patches.append((idx[:k].clone(), val[:k].clone(), k))
    ci, cv, ck = patches[0]
    for ib, vb, kb in patches[1:]:
        ci, cv, cnt = pulse.compose(ci, cv, ck, ib, vb, kb)
        ck = int(cnt.item())
    recv = view0.clone()
    pulse.apply(recv, ci, cv, ck)
    torch.cuda.synchronize()
    assert torch.equal(recv, prev)
    host = [(host_u32(i), v.cpu().numpy().view(np.uint16)) for i, v, _ in patches]
    oi, ov = oracle.compose_chain(host)
    np.testing.assert_array_equal(host_u32(ci[:ck]), oi)
    np.testing.assert_array_equal(cv[:ck].cpu().numpy().view(np.uint16), ov)
    assert pulse.get_error(dev) == 0


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_multi_segment(dtype):
    dev = _dev()
    rng = np.random.default_rng(9)
    shapes = [(0, 0, 10), (3, 0, 10), (0, 4, 10), (TILE, TILE + 1, 10 * TILE), (70000, 50000, 200000),
              (1, 1, 2), (5000, 6000, 9000)]
    segs, host, guards = [], [], []
    for ka, kb, n in shapes:
        a, b = _rand_patch(rng, n, ka, dtype), _rand_patch(rng, n, kb, dtype)
        ia, va = _to_dev(a, dev)
        ib, vb = _to_dev(b, dev)
        cap = max(ka + kb, 1)
        gio, gvo = Guarded(cap, torch.int32, dev), Guarded(cap, va.dtype, dev)
        guards += [gio, gvo]
        segs.append((ia, va, ka, ib, vb, kb, gio.t, gvo.t))
        host.append((a, b))
    counts = pulse.compose_multi(segs).cpu().tolist()
    for (a, b), s, k in zip(host, segs, counts):
        oi, ov = oracle.compose(a, b)
        assert k == oi.size
        np.testing.assert_array_equal(host_u32(s[6][:k]), oi)
        np.testing.assert_array_equal(_host_val(s[7][:k], dtype), ov)
    assert pulse.get_error(dev) == 0
    for g in guards:
        g.check()
