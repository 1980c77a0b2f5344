"""GPU vs oracle for the NVFP4 serving view (E2M1 codes two per byte, E4M3
scale per 16 elements, FP32 scale per tensor): every E4M3 block scale code
at a unit tensor scale, quantize, encode (changed code bytes and block
scales, the new tensor scale, refreshed previous view) and apply, single
tensor and multi-tensor plans, odd lengths, unaligned views, special values.
Every comparison is bit-exact (the tensor scale as an FP32 bit pattern)."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_f32, host_f32, host_u32

pytestmark = pytest.mark.gpu

TILE = 4096
NV = pulse.MX_NVFP4


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def _bits(x) -> int:
    return int(np.asarray(x, np.float32).reshape(-1).view(np.uint32)[0])


def _e4m3_value(c: int) -> float:
    e, m = (c >> 3) & 0xF, c & 7
    return m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)


def test_every_block_scale_code_at_unit_tensor_scale():
    """Block b's maximum is 6 * dec(b + 1), so with S = 1 (a 2688 in the last
    block) its scale byte is b + 1 for every positive finite E4M3 code; the
    other elements spread over the block's E2M1 grid and its ties."""
    dev = _dev()
    rng = np.random.default_rng(3)
    blocks = []
    for c in range(1, 0x7F):
        top = 6.0 * _e4m3_value(c)
        blk = (rng.uniform(-1, 1, 16) * top).astype(np.float32)
        ties = np.float32(top) * np.array([0.25, 0.75, 1.25, 2.5, 5.0], np.float32) / np.float32(6.0)
        blk[1:6] = ties
        blk[0] = np.float32(top) * np.float32(rng.choice([-1.0, 1.0]))  # the block maximum
        blocks.append(blk)
    blocks.append(np.full(16, 2688.0, np.float32))
    m = np.concatenate(blocks)
    codes, scales, ts = pulse.nvfp4_quantize(dev_f32(m, dev))
    oc, osc, oS = oracle.nvfp4_quantize(m)
    assert oS == np.float32(1.0) and _bits(host_f32(ts)) == _bits(oS)
    assert list(osc[:-1]) == list(range(1, 0x7F))
    np.testing.assert_array_equal(host_u8(scales), osc)
    np.testing.assert_array_equal(host_u8(codes), oc)


SIZES = [1, 2, 15, 16, 17, 33, 4095, TILE, TILE + 1, 3 * TILE + 77, 64 * TILE + 5]


def _special_master(n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(n) * 0.02).astype(np.float32)
    nb = (n + 15) // 16
    scale = np.exp2(rng.integers(-40, 10, nb)).repeat(16)[:n]
    wide = rng.random(nb).repeat(16)[:n] < 0.2
    m = np.where(wide, (rng.standard_normal(n) * scale).astype(np.float32), m).astype(np.float32)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1.4e-45, -1e-40, 0.5, 3.0],
                        dtype=np.float32)
    pick = rng.random(n) < 0.002
    m[pick] = rng.choice(specials, int(pick.sum()))
    zero_blocks = rng.random(nb) < 0.01
    m[np.repeat(zero_blocks, 16)[:n]] = 0.0
    return m


@pytest.mark.parametrize("n", SIZES)
def test_quantize_matches_oracle(n):
    dev = _dev()
    m = _special_master(n, 1200 + n)
    codes, scales, ts = pulse.nvfp4_quantize(dev_f32(m, dev))
    oc, osc, oS = oracle.nvfp4_quantize(m)
    assert _bits(host_f32(ts)) == _bits(oS)
    np.testing.assert_array_equal(host_u8(scales), osc)
    np.testing.assert_array_equal(host_u8(codes), oc)


def test_tiny_and_zero_tensors():
    dev = _dev()
    for m in (np.zeros(40, np.float32), np.full(33, 1e-41, np.float32),
              np.array([np.nan, 1.0, -np.inf] + [0.0] * 20, np.float32)):
        codes, scales, ts = pulse.nvfp4_quantize(dev_f32(m, dev))
        oc, osc, oS = oracle.nvfp4_quantize(m)
        assert _bits(host_f32(ts)) == _bits(oS)
        np.testing.assert_array_equal(host_u8(scales), osc)
        np.testing.assert_array_equal(host_u8(codes), oc)


def _encode_both(m_old, m_new, dev, offset=0):
    n = m_new.size
    nb, ncb = (n + 15) // 16, (n + 1) // 2
    oc, osc, _ = oracle.nvfp4_quantize(m_old)
    o_pc, o_ps = oc.copy(), osc.copy()
    o_patch = oracle.nvfp4_encode(m_new, o_pc, o_ps)

    guards = []

    def placed(a, dtype, numel=None):
        # `offset` elements into a guarded allocation; filled from `a` if given
        g = Guarded((a.size if numel is None else numel) + offset, dtype, dev)
        guards.append(g)
        view = g.t[offset:]
        if a is not None:
            view.copy_(torch.from_numpy(np.ascontiguousarray(a)).to(dev))
        return view

    master = placed(m_new, torch.float32)
    prev_c, prev_s = placed(oc, torch.uint8), placed(osc, torch.uint8)
    idx = placed(None, torch.int32, max(ncb, 1))
    val = placed(None, torch.uint8, max(ncb, 1))
    sidx = placed(None, torch.int32, max(nb, 1))
    sval = placed(None, torch.uint8, max(nb, 1))
    *_, counts, ts = pulse.nvfp4_encode(master, prev_c, prev_s, idx, val, sidx, sval)
    torch.cuda.synchronize()
    k, ks = (int(c) for c in counts.cpu().tolist())
    g_patch = (host_u32(idx[:k]), host_u8(val[:k]), host_u32(sidx[:ks]), host_u8(sval[:ks]))
    for name, g, o in zip(("idx", "val", "sidx", "sval"), g_patch, o_patch[:4]):
        np.testing.assert_array_equal(g, o, err_msg=name)
    assert _bits(host_f32(ts)) == _bits(o_patch[4])
    np.testing.assert_array_equal(host_u8(prev_c), o_pc)
    np.testing.assert_array_equal(host_u8(prev_s), o_ps)
    w_c, w_s = placed(oc, torch.uint8), placed(osc, torch.uint8)
    pulse.mx_apply(w_c, w_s, idx, val, k, sidx, sval, ks, fmt=NV, n=n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u8(w_c), o_pc)
    np.testing.assert_array_equal(host_u8(w_s), o_ps)
    assert pulse.get_error(dev) == 0
    for g in guards:
        g.check()
    return k, ks


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("eta", [3e-6, 1e-3, 3e-2])
def test_encode_matches_oracle(n, eta):
    dev = _dev()
    m0, _ = workloads.np_pair(n, seed=2200 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=2200 + n, eta=eta)
    _encode_both(m0, m1, dev)


@pytest.mark.parametrize("n", [TILE + 1, 5 * TILE + 333])
@pytest.mark.parametrize("offset", [1, 3, 4])
def test_encode_unaligned_views(n, offset):
    dev = _dev()
    m0, _ = workloads.np_pair(n, seed=3200 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=3200 + n, eta=3e-3)
    _encode_both(m0, m1, dev, offset=offset)


@pytest.mark.parametrize("n", [33, TILE, 7 * TILE + 19])
def test_encode_special_values(n):
    dev = _dev()
    m0 = _special_master(n, 4200 + n)
    m1 = _special_master(n, 5200 + n)
    keep = np.random.default_rng(n).random(n) < 0.5
    _encode_both(m0, np.where(keep, m0, m1).astype(np.float32), dev)


def test_tensor_scale_change_moves_blocks():
    """Raising the tensor maximum changes S, and with it block scales and
    codes all over the tensor, exactly as the oracle says."""
    dev = _dev()
    n = 3 * TILE + 5
    m0, _ = workloads.np_pair(n, seed=90, eta=0.0)
    m1 = m0.copy()
    m1[7] = np.float32(np.abs(m0).max() * 1.7)
    k, ks = _encode_both(m0, m1, dev)
    assert ks > 100


@pytest.mark.parametrize("device_counts", [True, False])
def test_plan_matches_oracle(device_counts):
    dev = _dev()
    specs = workloads.llama_layer()[-3:] + [workloads.TensorSpec(f"t{i}", (n,), "weight") for i, n in
                                            enumerate([5, 0, 33, 4096, 4097, 15, 3 * 4096 + 1, 1])]
    states = workloads.torch_model_states(specs, 29, 1e-3, dev)
    prev_c, prev_s, codes, scales, idx, val, sidx, sval, c0, s0 = ([] for _ in range(10))
    guards = []

    def guard(t, numel=0, dtype=torch.uint8):
        # a copy of t (or numel elements) between guard zones
        g = Guarded(t.numel() if t is not None else numel, t.dtype if t is not None else dtype,
                    dev, init=t)
        guards.append(g)
        return g.t

    for (w, _), s in zip(states, specs):
        c, sc, _ = pulse.nvfp4_quantize(w)
        prev_c.append(guard(c))
        prev_s.append(guard(sc))
        c0.append(host_u8(c))
        s0.append(host_u8(sc))
        codes.append(guard(c))
        scales.append(guard(sc))
        ncb, nb = pulse.mx_code_bytes(s.numel, NV), pulse.mx_scale_count(s.numel, NV)
        idx.append(guard(None, max(ncb, 1), torch.int32))
        val.append(guard(None, max(ncb, 1)))
        sidx.append(guard(None, max(nb, 1), torch.int32))
        sval.append(guard(None, max(nb, 1)))
    slots = [pulse.MxTensorSlot(s.numel, master=states[i][1], prev_codes=prev_c[i],
                                prev_scales=prev_s[i], codes=codes[i], scales=scales[i],
                                idx=idx[i], val=val[i], sidx=sidx[i], sval=sval[i])
             for i, s in enumerate(specs)]
    with pulse.MxPlan(slots, fmt=NV) as plan:
        counts = plan.encode()
        plan.apply(counts if device_counts else counts.cpu().tolist())
        torch.cuda.synchronize()
        assert plan.get_error() == 0
        cnt = counts.cpu().tolist()
        tsc = host_f32(plan.tscales)
        for t, s in enumerate(specs):
            o_c, o_s = c0[t].copy(), s0[t].copy()
            o_patch = oracle.nvfp4_encode(host_f32(states[t][1]), o_c, o_s)
            k, ks = cnt[2 * t], cnt[2 * t + 1]
            assert (k, ks) == (o_patch[0].size, o_patch[2].size), t
            np.testing.assert_array_equal(host_u32(idx[t][:k]), o_patch[0])
            np.testing.assert_array_equal(host_u8(val[t][:k]), o_patch[1])
            np.testing.assert_array_equal(host_u32(sidx[t][:ks]), o_patch[2])
            np.testing.assert_array_equal(host_u8(sval[t][:ks]), o_patch[3])
            assert _bits(tsc[t]) == _bits(o_patch[4]), t
            np.testing.assert_array_equal(host_u8(prev_c[t]), o_c)
            np.testing.assert_array_equal(host_u8(codes[t]), o_c)
            np.testing.assert_array_equal(host_u8(scales[t]), o_s)
    for g in guards:
        g.check()


def test_mx_calls_refuse_nvfp4():
    dev = _dev()
    m = torch.zeros(32, device=dev)
    with pytest.raises(pulse.PulseError):
        pulse.mx_quantize(m, fmt=NV)
