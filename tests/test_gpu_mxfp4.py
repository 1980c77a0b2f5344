"""GPU vs oracle for the MXFP4 serving view (E2M1 codes two per byte, E8M0
scale per 32 elements): the convert over every FP32 pattern below 8 at unit
scale, quantize, encode (changed code bytes and scales, refreshed previous
view) and apply, single tensor and multi-tensor plans, odd lengths,
unaligned views, special values. Every comparison is bit-exact."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_f32, host_f32, host_u32

pytestmark = pytest.mark.gpu

WORKERS = max(1, min(8, (os.cpu_count() or 2) // 2))
TILE = 4096
FP4 = pulse.MX_E2M1


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


# ------------------------------------------------- the E2M1 convert, exhaustive

def _blocks_with_leader(vals: np.ndarray) -> np.ndarray:
    """31 values per block after a leading 6.0, which fixes the block scale at
    2^0 (E8M0 byte 127) while every |value| < 8."""
    nb = (vals.size + 30) // 31
    pad = np.zeros(nb * 31, dtype=np.float32)
    pad[:vals.size] = vals
    out = np.empty((nb, 32), dtype=np.float32)
    out[:, 0] = 6.0
    out[:, 1:] = pad.reshape(nb, 31)
    return out.reshape(-1)


def test_e2m1_convert_exhaustive_below_8():
    """Every FP32 pattern with |y| < 8 (biased exponent <= 129), both signs,
    quantized at unit scale on the GPU, equals the oracle's code."""
    dev = _dev()
    top = 130 << 23
    chunk = 31 * (1 << 21)
    jobs = [(lo, min(lo + chunk, top), sign) for sign in (0, 0x80000000) for lo in range(0, top, chunk)]

    def blocks_of(job):
        lo, hi, sign = job
        return _blocks_with_leader((np.arange(lo, hi, dtype=np.uint32) | np.uint32(sign)).view(np.float32))

    def run(job):
        return oracle.mxfp4_quantize(blocks_of(job))

    with ThreadPoolExecutor(WORKERS) as ex:
        futures = [ex.submit(run, j) for j in jobs]
        for job, fut in zip(jobs, futures):
            blocks = blocks_of(job)
            g_codes, g_scales = pulse.mx_quantize(dev_f32(blocks, dev), fmt=FP4)
            o_codes, o_scales = fut.result()
            assert (o_scales == 127).all()
            np.testing.assert_array_equal(host_u8(g_scales), o_scales)
            g = host_u8(g_codes)
            if not np.array_equal(g, o_codes):
                bad = np.nonzero(g != o_codes)[0][:8]
                raise AssertionError(
                    f"code bytes differ at {bad.tolist()}: inputs "
                    f"{[blocks[2 * b:2 * b + 2].tolist() for b in bad]} "
                    f"gpu {g[bad].tolist()} oracle {o_codes[bad].tolist()}")


# ---------------------------------------------------------------- quantize

SIZES = [1, 2, 31, 32, 33, 127, 4095, TILE, TILE + 1, 3 * TILE + 77, 64 * TILE + 5]


def _special_master(n: int, seed: int) -> np.ndarray:
    """Normal weights with scale-stressing blocks: wide magnitudes, zeros,
    signed zeros, NaN, infinities, subnormals, grid points and ties."""
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(n) * 0.02).astype(np.float32)
    nb = (n + 31) // 32
    scale = np.exp2(rng.integers(-140, 120, nb)).repeat(32)[:n]
    wide = rng.random(nb).repeat(32)[:n] < 0.2
    m = np.where(wide, (rng.standard_normal(n) * scale).astype(np.float32), m).astype(np.float32)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1.4e-45, -1e-40, 0.25, 0.75, 1.25,
                         2.5, 5.0, 6.0, 3.4e38], dtype=np.float32)
    pick = rng.random(n) < 0.002
    m[pick] = rng.choice(specials, int(pick.sum()))
    zero_blocks = rng.random(nb) < 0.01
    m[np.repeat(zero_blocks, 32)[:n]] = 0.0
    return m


@pytest.mark.parametrize("n", SIZES)
def test_quantize_matches_oracle(n):
    dev = _dev()
    m = _special_master(n, 1100 + n)
    codes, scales = pulse.mx_quantize(dev_f32(m, dev), fmt=FP4)
    o_codes, o_scales = oracle.mxfp4_quantize(m)
    np.testing.assert_array_equal(host_u8(scales), o_scales)
    np.testing.assert_array_equal(host_u8(codes), o_codes)


# ------------------------------------------------------------------ encode

def _encode_both(m_old: np.ndarray, m_new: np.ndarray, dev, offset: int = 0):
    """GPU and oracle encode of m_new against the MXFP4 view of m_old. With
    offset > 0 every device array starts `offset` elements (bytes) into a
    larger allocation: an unaligned view, the kernel's generic path."""
    n = m_new.size
    nb = (n + 31) // 32
    ncb = (n + 1) // 2
    o_codes, o_scales = oracle.mxfp4_quantize(m_old)
    o_pc, o_ps = o_codes.copy(), o_scales.copy()
    o_patch = oracle.mxfp4_encode(m_new, o_pc, o_ps)

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
    prev_c = placed(o_codes, torch.uint8)
    prev_s = placed(o_scales, torch.uint8)
    idx = placed(None, torch.int32, max(ncb, 1))
    val = placed(None, torch.uint8, max(ncb, 1))
    sidx = placed(None, torch.int32, max(nb, 1))
    sval = placed(None, torch.uint8, max(nb, 1))
    _, _, _, _, counts = pulse.mx_encode(master, prev_c, prev_s, idx, val, sidx, sval, fmt=FP4)
    torch.cuda.synchronize()
    k, ks = (int(c) for c in counts.cpu().tolist())
    g_patch = (host_u32(idx[:k]), host_u8(val[:k]), host_u32(sidx[:ks]), host_u8(sval[:ks]))
    for name, g, o in zip(("idx", "val", "sidx", "sval"), g_patch, o_patch):
        np.testing.assert_array_equal(g, o, err_msg=name)
    np.testing.assert_array_equal(host_u8(prev_c), o_pc)
    np.testing.assert_array_equal(host_u8(prev_s), o_ps)
    # receiver: the old view plus the patch is the new view
    w_c, w_s = placed(o_codes, torch.uint8), placed(o_scales, torch.uint8)
    pulse.mx_apply(w_c, w_s, idx, val, k, sidx, sval, ks, fmt=FP4, n=n)
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
    m0, _ = workloads.np_pair(n, seed=2100 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=2100 + n, eta=eta)
    _encode_both(m0, m1, dev)


@pytest.mark.parametrize("n", [TILE + 1, 5 * TILE + 333])
@pytest.mark.parametrize("offset", [1, 3, 4])
def test_encode_unaligned_views(n, offset):
    dev = _dev()
    m0, _ = workloads.np_pair(n, seed=3100 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=3100 + n, eta=3e-3)
    _encode_both(m0, m1, dev, offset=offset)


@pytest.mark.parametrize("n", [33, TILE, 7 * TILE + 19])
def test_encode_special_values_and_scale_changes(n):
    dev = _dev()
    m0 = _special_master(n, 4100 + n)
    m1 = _special_master(n, 5100 + n)
    keep = np.random.default_rng(n).random(n) < 0.5
    m1 = np.where(keep, m0, m1).astype(np.float32)
    k, ks = _encode_both(m0, m1, dev)
    if n >= TILE:  # many blocks: some scale moves
        assert ks > 0


def test_encode_everything_changes_and_nothing_changes():
    dev = _dev()
    n = 9 * TILE + 7
    rng = np.random.default_rng(6)
    m0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    k, ks = _encode_both(m0, -m0, dev)   # every code flips its sign bit, no scale moves
    assert k == (n + 1) // 2 and ks == 0
    k, ks = _encode_both(m0, m0.copy(), dev)
    assert k == 0 and ks == 0


def test_padding_nibble_of_an_odd_tensor():
    """A previous view whose padding nibble is not zero: the last byte is a
    change, exactly as the oracle says."""
    dev = _dev()
    n = 2 * TILE + 33
    m, _ = workloads.np_pair(n, seed=77, eta=0.0)
    o_c, o_s = oracle.mxfp4_quantize(m)
    bad = o_c.copy()
    bad[-1] |= 0x30
    prev_c = torch.from_numpy(bad).to(dev)
    prev_s = torch.from_numpy(o_s.copy()).to(dev)
    idx, val, sidx, sval, counts = pulse.mx_encode(dev_f32(m, dev), prev_c, prev_s, fmt=FP4)
    k, ks = (int(c) for c in counts.cpu().tolist())
    o_patch = oracle.mxfp4_encode(m, bad, o_s.copy())
    assert k == o_patch[0].size == 1 and ks == 0
    assert host_u32(idx[:k]).tolist() == [(n + 1) // 2 - 1]
    np.testing.assert_array_equal(host_u8(prev_c), o_c)


def test_two_steps_in_a_row_on_one_workspace():
    dev = _dev()
    n = 11 * TILE + 5
    m0, _ = workloads.np_pair(n, seed=71, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=71, eta=1e-3)
    m2, _ = workloads.np_pair(n, seed=71, eta=2e-3)
    codes, scales = pulse.mx_quantize(dev_f32(m0, dev), fmt=FP4)
    o_c, o_s = oracle.mxfp4_quantize(m0)
    for m in (m1, m2):
        idx, val, sidx, sval, counts = pulse.mx_encode(dev_f32(m, dev), codes, scales, fmt=FP4)
        o_patch = oracle.mxfp4_encode(m, o_c, o_s)
        k, ks = (int(c) for c in counts.cpu().tolist())
        np.testing.assert_array_equal(host_u32(idx[:k]), o_patch[0])
        np.testing.assert_array_equal(host_u8(val[:k]), o_patch[1])
        np.testing.assert_array_equal(host_u32(sidx[:ks]), o_patch[2])
        np.testing.assert_array_equal(host_u8(sval[:ks]), o_patch[3])
        np.testing.assert_array_equal(host_u8(codes), o_c)
        np.testing.assert_array_equal(host_u8(scales), o_s)


def test_apply_checked_skips_out_of_range_bytes():
    dev = _dev()
    n = 99  # 50 code bytes, 4 scales
    codes = torch.zeros(50, dtype=torch.uint8, device=dev)
    scales = torch.zeros(4, dtype=torch.uint8, device=dev)
    idx = torch.tensor([3, 50, 49], dtype=torch.int32, device=dev)
    val = torch.tensor([1, 2, 3], dtype=torch.uint8, device=dev)
    sidx = torch.tensor([4, 0], dtype=torch.int32, device=dev)
    sval = torch.tensor([9, 8], dtype=torch.uint8, device=dev)
    pulse.mx_apply(codes, scales, idx, val, 3, sidx, sval, 2, fmt=FP4, n=n)
    assert pulse.get_error(dev) == pulse.pulse.PULSE_ERR_INDEX
    assert host_u8(codes)[[3, 49]].tolist() == [1, 3]
    assert host_u8(scales).tolist() == [8, 0, 0, 0]
    assert pulse.get_error(dev) == 0


# -------------------------------------------------------------- multi-tensor

@pytest.mark.parametrize("device_counts", [True, False])
def test_plan_matches_oracle(device_counts):
    dev = _dev()
    specs = workloads.llama_layer()[-3:] + [workloads.TensorSpec(f"t{i}", (n,), "weight") for i, n in
                                            enumerate([5, 0, 33, 4096, 4097, 31, 3 * 4096 + 1, 1])]
    states = workloads.torch_model_states(specs, 23, 1e-3, dev)
    prev_c, prev_s, codes, scales, idx, val, sidx, sval, c0, s0 = ([] for _ in range(10))
    guards = []

    def guard(t, numel=0, dtype=torch.uint8):
        # a copy of t (or numel elements) between guard zones
        g = Guarded(t.numel() if t is not None else numel, t.dtype if t is not None else dtype,
                    dev, init=t)
        guards.append(g)
        return g.t

    for (w, _), s in zip(states, specs):
        c, sc = pulse.mx_quantize(w, fmt=FP4)
        prev_c.append(guard(c))
        prev_s.append(guard(sc))
        c0.append(host_u8(c))
        s0.append(host_u8(sc))
        codes.append(guard(c))
        scales.append(guard(sc))
        ncb, nb = pulse.mx_code_bytes(s.numel, FP4), pulse.mx_blocks(s.numel)
        idx.append(guard(None, max(ncb, 1), torch.int32))
        val.append(guard(None, max(ncb, 1)))
        sidx.append(guard(None, max(nb, 1), torch.int32))
        sval.append(guard(None, max(nb, 1)))
    slots = [pulse.MxTensorSlot(s.numel, master=states[i][1], prev_codes=prev_c[i],
                                prev_scales=prev_s[i], codes=codes[i], scales=scales[i],
                                idx=idx[i], val=val[i], sidx=sidx[i], sval=sval[i])
             for i, s in enumerate(specs)]
    with pulse.MxPlan(slots, fmt=FP4) as plan:
        counts = plan.encode()
        plan.apply(counts if device_counts else counts.cpu().tolist())
        torch.cuda.synchronize()
        assert plan.get_error() == 0
        cnt = counts.cpu().tolist()
        for t, s in enumerate(specs):
            o_c, o_s = c0[t].copy(), s0[t].copy()
            o_patch = oracle.mxfp4_encode(host_f32(states[t][1]), o_c, o_s)
            k, ks = cnt[2 * t], cnt[2 * t + 1]
            assert (k, ks) == (o_patch[0].size, o_patch[2].size), t
            np.testing.assert_array_equal(host_u32(idx[t][:k]), o_patch[0])
            np.testing.assert_array_equal(host_u8(val[t][:k]), o_patch[1])
            np.testing.assert_array_equal(host_u32(sidx[t][:ks]), o_patch[2])
            np.testing.assert_array_equal(host_u8(sval[t][:ks]), o_patch[3])
            np.testing.assert_array_equal(host_u8(prev_c[t]), o_c)
            np.testing.assert_array_equal(host_u8(codes[t]), o_c)
            np.testing.assert_array_equal(host_u8(scales[t]), o_s)
    for g in guards:
        g.check()
