"""GPU vs oracle for the PULSELoCo gate with FP32 error feedback and the
receiver's accumulation, through the C ABI: sizes across many tiles with
ragged tails, unaligned views, special values, several rounds on one error
buffer, multi-tensor plans. Every comparison is bit-exact (FP32 bit patterns
included)."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_f32, host_f32, host_u32

pytestmark = pytest.mark.gpu

TILE = 2048


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def _round(n, seed, scale=2e-5, err_scale=1e-5):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    w = (g + rng.standard_normal(n).astype(np.float32) * np.float32(scale)).astype(np.float32)
    e = (rng.standard_normal(n) * err_scale).astype(np.float32)
    return g, w, e


def _check(g, w, e, dev, offset=0):
    n = g.size

    guards = []

    def placed(a):
        gb = Guarded(n + offset, torch.float32, dev)
        guards.append(gb)
        v = gb.t[offset:]
        v.copy_(torch.from_numpy(a).to(dev))
        return v

    gt, wt, et = placed(g), placed(w), placed(e)
    gi, gv = Guarded(max(n, 1), torch.int32, dev), Guarded(max(n, 1), torch.float32, dev)
    gc = Guarded(1, torch.int64, dev)
    guards += [gi, gv, gc]
    idx, val, cnt = pulse.loco_gate(gt, wt, et, gi.t, gv.t, gc.t)
    torch.cuda.synchronize()
    k = int(cnt.item())
    oe = e.copy()
    oi, ov = oracle.loco_gate(g, w, oe)
    assert k == oi.size
    np.testing.assert_array_equal(host_u32(idx[:k]), oi)
    np.testing.assert_array_equal(_bits(host_f32(val[:k])), _bits(ov))
    np.testing.assert_array_equal(_bits(host_f32(et)), _bits(oe))
    assert pulse.get_error(dev) == 0
    for gb in guards:
        gb.check()
    return k


@pytest.mark.parametrize("n", [1, 3, 4, 5, TILE - 1, TILE, TILE + 1, 7 * TILE + 13, 1 << 20])
def test_gate_matches_oracle(n):
    dev = _dev()
    k = _check(*_round(n, 100 + n), dev)
    if n >= TILE:
        assert 0 < k < n


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_gate_unaligned_views(offset):
    dev = _dev()
    _check(*_round(5 * TILE + 77, 7 + offset), dev, offset=offset)


def test_gate_special_values():
    dev = _dev()
    n = 3 * TILE + 5
    g, w, e = _round(n, 55)
    rng = np.random.default_rng(56)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1e-40, -1e-40, 3e38, 1.0, 1.00390625],
                        np.float32)
    for arr in (g, w, e):
        pick = rng.random(n) < 0.01
        arr[pick] = rng.choice(specials, int(pick.sum()))
    _check(g, w, e, dev)


def test_rounds_on_one_error_buffer():
    """Five rounds of local steps against a fixed global checkpoint: the
    error buffer carries over, and entries below the gate are sent once
    their accumulated error crosses it (same rounds as the oracle)."""
    dev = _dev()
    n = 6 * TILE + 3
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    e_gpu = torch.zeros(n, dtype=torch.float32, device=dev)
    e_cpu = np.zeros(n, np.float32)
    gt = dev_f32(g, dev)
    total = 0
    for r in range(5):
        w = (g + rng.standard_normal(n).astype(np.float32) * np.float32(1.5e-5)).astype(np.float32)
        idx, val, cnt = pulse.loco_gate(gt, dev_f32(w, dev), e_gpu)
        k = int(cnt.item())
        oi, ov = oracle.loco_gate(g, w, e_cpu)
        np.testing.assert_array_equal(host_u32(idx[:k]), oi)
        np.testing.assert_array_equal(_bits(host_f32(val[:k])), _bits(ov))
        np.testing.assert_array_equal(_bits(host_f32(e_gpu)), _bits(e_cpu))
        total += k
    assert total > 0


def test_accumulate_matches_oracle_and_checks_indices():
    dev = _dev()
    rng = np.random.default_rng(8)
    n = 100000
    acc = rng.standard_normal(n).astype(np.float32)
    idx = np.sort(rng.choice(n, 30000, replace=False)).astype(np.uint32)
    val = rng.standard_normal(30000).astype(np.float32)
    ga = Guarded(n, torch.float32, dev, init=acc)
    at = ga.t
    pulse.loco_accumulate(at, torch.from_numpy(idx.view(np.int32)).to(dev), dev_f32(val, dev), idx.size)
    torch.cuda.synchronize()
    exp = acc.copy()
    oracle.loco_accumulate(exp, idx, val)
    np.testing.assert_array_equal(_bits(host_f32(at)), _bits(exp))
    assert pulse.get_error(dev) == 0
    bad = torch.tensor([5, n, 7], dtype=torch.int32, device=dev)
    pulse.loco_accumulate(at, bad, torch.ones(3, device=dev), 3)
    assert pulse.get_error(dev) == pulse.pulse.PULSE_ERR_INDEX
    ga.check("acc")


def test_plan_gate_then_accumulate():
    """A decoder layer's worth of tensors (plus tiny and empty ones): the
    gate of every tensor in one launch equals the oracle per tensor, and a
    receiver accumulating the sent entries ends at global + sent values."""
    dev = _dev()
    specs = workloads.llama_layer()[-4:] + [workloads.TensorSpec(f"t{i}", (n,), "weight")
                                            for i, n in enumerate([0, 1, 5, TILE + 3])]
    rng = np.random.default_rng(21)
    host, slots, guards = [], [], []
    for s in specs:
        g, w, e = _round(s.numel, int(rng.integers(1 << 30)))
        gt, wt = dev_f32(g, dev), dev_f32(w, dev)
        bufs = [Guarded(s.numel, torch.float32, dev, init=e),
                Guarded(max(s.numel, 1), torch.int32, dev),
                Guarded(max(s.numel, 1), torch.float32, dev),
                Guarded(s.numel, torch.float32, dev, init=g)]
        guards += bufs
        et, idx, val, acc = (b.t for b in bufs)
        host.append((g, w, e))
        slots.append(pulse.LocoTensorSlot(s.numel, global_w=gt, local_w=wt, err=et, idx=idx, val=val,
                                          acc=acc))
    with pulse.LocoPlan(slots) as plan:
        counts = plan.gate()
        plan.accumulate(counts)
        torch.cuda.synchronize()
        assert plan.get_error() == 0
        c = counts.cpu().tolist()
        for (g, w, e), sl, k in zip(host, slots, c):
            oe = e.copy()
            oi, ov = oracle.loco_gate(g, w, oe)
            assert k == oi.size
            np.testing.assert_array_equal(host_u32(sl.idx[:k]), oi)
            np.testing.assert_array_equal(_bits(host_f32(sl.val[:k])), _bits(ov))
            np.testing.assert_array_equal(_bits(host_f32(sl.err)), _bits(oe))
            acc = g.copy()
            oracle.loco_accumulate(acc, oi, ov)
            np.testing.assert_array_equal(_bits(host_f32(sl.acc)), _bits(acc))
    for b in guards:
        b.check()
