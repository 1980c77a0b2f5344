"""GPU vs oracle for the MXFP8 serving view: quantize, encode (both patch
segments, refreshed previous view) and apply, single tensor and multi-tensor
plans, through the C ABI. Every comparison is bit-exact.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_f32, guarded_u8, host_f32, host_u32

pytestmark = pytest.mark.gpu

WORKERS = max(1, min(8, (os.cpu_count() or 2) // 2))
TILE = 4096


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def dev_u8(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(device)


# ------------------------------------------------- the E4M3 convert, exhaustive

def _patterns(lo: int, hi: int, sign: int) -> np.ndarray:
    return (np.arange(lo, hi, dtype=np.uint32) | np.uint32(sign)).view(np.float32)


def _blocks_with_leader(vals: np.ndarray) -> np.ndarray:
    """31 values per block after a leading 256.0, which fixes the block
    scale at 2^0 (E8M0 byte 127) while every |value| < 512."""
    nb = (vals.size + 30) // 31
    pad = np.zeros(nb * 31, dtype=np.float32)
    pad[:vals.size] = vals
    out = np.empty((nb, 32), dtype=np.float32)
    out[:, 0] = 256.0
    out[:, 1:] = pad.reshape(nb, 31)
    return out.reshape(-1)


def test_e4m3_convert_exhaustive_below_512():
    """Every FP32 pattern with |y| < 512 (biased exponent <= 135), both signs,
    quantized at unit scale on the GPU, equals the oracle's code."""
    dev = _dev()
    top = 136 << 23
    chunk = 31 * (1 << 21)
    jobs = [(lo, min(lo + chunk, top), sign) for sign in (0, 0x80000000) for lo in range(0, top, chunk)]

    def run(job):
        lo, hi, sign = job
        blocks = _blocks_with_leader(_patterns(lo, hi, sign))
        codes, scales = oracle.mxfp8_quantize(blocks)
        return codes, scales

    with ThreadPoolExecutor(WORKERS) as ex:
        futures = [ex.submit(run, j) for j in jobs]
        for job, fut in zip(jobs, futures):
            lo, hi, sign = job
            blocks = _blocks_with_leader(_patterns(lo, hi, sign))
            g_codes, g_scales = pulse.mx_quantize(dev_f32(blocks, dev))
            o_codes, o_scales = fut.result()
            assert (o_scales == 127).all()
            np.testing.assert_array_equal(host_u8(g_scales), o_scales)
            g = host_u8(g_codes)
            if not np.array_equal(g, o_codes):
                bad = np.nonzero(g != o_codes)[0][:8]
                raise AssertionError(
                    f"codes differ at {bad.tolist()}: inputs {blocks[bad].tolist()} "
                    f"gpu {g[bad].tolist()} oracle {o_codes[bad].tolist()}")


# ---------------------------------------------------------------- quantize

SIZES = [1, 31, 32, 33, 127, 4095, TILE, TILE + 1, 3 * TILE + 77, 64 * TILE + 5]


def _special_master(n: int, seed: int) -> np.ndarray:
    """Normal weights with scale-stressing blocks: wide magnitudes, zeros,
    signed zeros, NaN, infinities, subnormals, exact powers of two."""
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(n) * 0.02).astype(np.float32)
    nb = (n + 31) // 32
    scale = np.exp2(rng.integers(-140, 120, nb)).repeat(32)[:n]
    wide = rng.random(nb).repeat(32)[:n] < 0.2
    m = np.where(wide, (rng.standard_normal(n) * scale).astype(np.float32), m).astype(np.float32)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1.4e-45, -1e-40, 1.0, 2.0, 0.5,
                         448.0, 3.4e38], dtype=np.float32)
    pick = rng.random(n) < 0.002
    m[pick] = rng.choice(specials, int(pick.sum()))
    zero_blocks = rng.random(nb) < 0.01
    m[np.repeat(zero_blocks, 32)[:n]] = 0.0
    return m


@pytest.mark.parametrize("n", SIZES)
def test_quantize_matches_oracle(n):
    dev = _dev()
    m = _special_master(n, 1000 + n)
    gc, gs = Guarded(n, torch.uint8, dev), Guarded((n + 31) // 32, torch.uint8, dev)
    codes, scales = pulse.mx_quantize(dev_f32(m, dev), gc.t, gs.t)
    o_codes, o_scales = oracle.mxfp8_quantize(m)
    np.testing.assert_array_equal(host_u8(scales), o_scales)
    np.testing.assert_array_equal(host_u8(codes), o_codes)
    gc.check("codes")
    gs.check("scales")


# ------------------------------------------------------------------ encode

def _encode_both(m_old: np.ndarray, m_new: np.ndarray, dev, offset: int = 0):
    """GPU and oracle encode of m_new against the view of m_old. With
    offset > 0 every device array starts `offset` elements into a larger
    allocation (an unaligned view: the kernel's generic path)."""
    n = m_new.size
    nb = (n + 31) // 32
    o_codes, o_scales = oracle.mxfp8_quantize(m_old)
    o_pc, o_ps = o_codes.copy(), o_scales.copy()
    o_patch = oracle.mxfp8_encode(m_new, o_pc, o_ps)

    guards = {}

    def placed(name, a, dtype, numel=None):
        # `offset` elements into a guarded allocation; filled from `a` if given
        numel = a.size if numel is None else numel
        g = Guarded(numel + offset, dtype, dev)
        guards[name] = g
        view = g.t[offset:]
        if a is not None:
            view.copy_(torch.from_numpy(np.ascontiguousarray(a)).to(dev))
        return view

    master = placed("master", m_new, torch.float32)
    prev_c = placed("prev_codes", o_codes, torch.uint8)
    prev_s = placed("prev_scales", o_scales, torch.uint8)
    idx = placed("idx", None, torch.int32, max(n, 1))
    val = placed("val", None, torch.uint8, max(n, 1))
    sidx = placed("sidx", None, torch.int32, max(nb, 1))
    sval = placed("sval", None, torch.uint8, max(nb, 1))
    _, _, _, _, counts = pulse.mx_encode(master, prev_c, prev_s, idx, val, sidx, sval)
    torch.cuda.synchronize()
    k, ks = (int(c) for c in counts.cpu().tolist())
    g_patch = (host_u32(idx[:k]), host_u8(val[:k]), host_u32(sidx[:ks]), host_u8(sval[:ks]))
    for name, g, o in zip(("idx", "val", "sidx", "sval"), g_patch, o_patch):
        np.testing.assert_array_equal(g, o, err_msg=name)
    np.testing.assert_array_equal(host_u8(prev_c), o_pc)
    np.testing.assert_array_equal(host_u8(prev_s), o_ps)
    # receiver: the old view plus the patch is the new view
    w_c, w_s = placed("codes", o_codes, torch.uint8), placed("scales", o_scales, torch.uint8)
    pulse.mx_apply(w_c, w_s, idx, val, k, sidx, sval, ks)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u8(w_c), o_pc)
    np.testing.assert_array_equal(host_u8(w_s), o_ps)
    assert pulse.get_error(dev) == 0
    for name, g in guards.items():
        g.check(name)
    return k, ks


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("eta", [3e-6, 1e-4, 3e-2])
def test_encode_matches_oracle(n, eta):
    dev = _dev()
    m0, _ = workloads.np_pair(n, seed=2000 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=2000 + n, eta=eta)
    _encode_both(m0, m1, dev)


@pytest.mark.parametrize("n", [TILE + 1, 5 * TILE + 333])
@pytest.mark.parametrize("offset", [1, 3, 4])
def test_encode_unaligned_views(n, offset):
    dev = _dev()
    m0, _ = workloads.np_pair(n, seed=3000 + n, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=3000 + n, eta=1e-3)
    _encode_both(m0, m1, dev, offset=offset)


@pytest.mark.parametrize("n", [33, TILE, 7 * TILE + 19])
def test_encode_special_values_and_scale_changes(n):
    dev = _dev()
    m0 = _special_master(n, 4000 + n)
    m1 = _special_master(n, 5000 + n)
    keep = np.random.default_rng(n).random(n) < 0.5
    m1 = np.where(keep, m0, m1).astype(np.float32)
    k, ks = _encode_both(m0, m1, dev)
    assert ks > 0


def test_encode_everything_changes_and_nothing_changes():
    dev = _dev()
    n = 9 * TILE + 7
    rng = np.random.default_rng(6)
    m0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    k, ks = _encode_both(m0, -m0, dev)   # every code flips its sign bit, no scale moves
    assert k == n and ks == 0
    k, ks = _encode_both(m0, m0.copy(), dev)
    assert k == 0 and ks == 0


def test_two_steps_in_a_row_on_one_workspace():
    dev = _dev()
    n = 11 * TILE + 5
    m0, _ = workloads.np_pair(n, seed=70, eta=0.0)
    m1, _ = workloads.np_pair(n, seed=70, eta=1e-4)
    m2, _ = workloads.np_pair(n, seed=70, eta=2e-4)
    codes, scales = pulse.mx_quantize(dev_f32(m0, dev))
    o_c, o_s = oracle.mxfp8_quantize(m0)
    for m in (m1, m2):
        idx, val, sidx, sval, counts = pulse.mx_encode(dev_f32(m, dev), codes, scales)
        o_patch = oracle.mxfp8_encode(m, o_c, o_s)
        k, ks = (int(c) for c in counts.cpu().tolist())
        np.testing.assert_array_equal(host_u32(idx[:k]), o_patch[0])
        np.testing.assert_array_equal(host_u8(val[:k]), o_patch[1])
        np.testing.assert_array_equal(host_u32(sidx[:ks]), o_patch[2])
        np.testing.assert_array_equal(host_u8(sval[:ks]), o_patch[3])
        np.testing.assert_array_equal(host_u8(codes), o_c)
        np.testing.assert_array_equal(host_u8(scales), o_s)


def test_empty_tensor_and_argument_checks():
    dev = _dev()
    counts = torch.full((2,), 7, dtype=torch.int64, device=dev)
    e = torch.empty(0, device=dev)
    e8 = torch.empty(0, dtype=torch.uint8, device=dev)
    pulse.mx_encode(e, e8, e8, counts_out=counts)
    assert counts.cpu().tolist() == [0, 0]
    with pytest.raises(ValueError):   # 33 elements need 2 scale bytes
        pulse.mx_encode(torch.zeros(33, device=dev), torch.zeros(33, dtype=torch.uint8, device=dev),
                        torch.zeros(1, dtype=torch.uint8, device=dev))


def test_apply_checked_skips_out_of_range_entries():
    dev = _dev()
    n = 100
    codes = torch.zeros(n, dtype=torch.uint8, device=dev)
    scales = torch.zeros(4, dtype=torch.uint8, device=dev)
    idx = torch.tensor([3, 100, 99], dtype=torch.int32, device=dev)
    val = torch.tensor([1, 2, 3], dtype=torch.uint8, device=dev)
    sidx = torch.tensor([4, 0], dtype=torch.int32, device=dev)
    sval = torch.tensor([9, 8], dtype=torch.uint8, device=dev)
    pulse.mx_apply(codes, scales, idx, val, 3, sidx, sval, 2)
    assert pulse.get_error(dev) == pulse.pulse.PULSE_ERR_INDEX
    assert host_u8(codes)[[3, 99]].tolist() == [1, 3]
    assert host_u8(scales).tolist() == [8, 0, 0, 0]
    assert pulse.get_error(dev) == 0


# -------------------------------------------------------------- multi-tensor

class MxModel:
    """Trainer and sampler MXFP8 buffers of one model (one allocation per tensor)."""

    def __init__(self, specs, seed, eta, dev):
        states = workloads.torch_model_states(specs, seed, eta, dev)
        self.specs = specs
        self.w0 = [w for w, _ in states]      # weights before the step
        self.master = [m for _, m in states]  # after it
        # the previous view is the MXFP8 view of the weights before the step
        self.prev_c, self.prev_s = [], []
        for w in self.w0:
            c, sc = pulse.mx_quantize(w)
            self.prev_c.append(c)
            self.prev_s.append(sc)
        self.c0 = [c.clone() for c in self.prev_c]
        self.s0 = [s.clone() for s in self.prev_s]
        # every buffer the encode or the apply writes sits between guard zones
        self.guards = []

        def guarded(t=None, numel=0, dtype=torch.uint8):
            g = Guarded(t.numel() if t is not None else numel, t.dtype if t is not None else dtype,
                        dev, init=t)
            self.guards.append(g)
            return g.t

        self.prev_c = [guarded(c) for c in self.c0]
        self.prev_s = [guarded(x) for x in self.s0]
        self.codes = [guarded(c) for c in self.c0]
        self.scales = [guarded(x) for x in self.s0]
        self.idx = [guarded(numel=max(s.numel, 1), dtype=torch.int32) for s in specs]
        self.val = [guarded(numel=max(s.numel, 1)) for s in specs]
        nb = [pulse.mx_blocks(s.numel) for s in specs]
        self.sidx = [guarded(numel=max(b, 1), dtype=torch.int32) for b in nb]
        self.sval = [guarded(numel=max(b, 1)) for b in nb]
        slots = [pulse.MxTensorSlot(s.numel, master=self.master[i], prev_codes=self.prev_c[i],
                                    prev_scales=self.prev_s[i], codes=self.codes[i],
                                    scales=self.scales[i], idx=self.idx[i], val=self.val[i],
                                    sidx=self.sidx[i], sval=self.sval[i])
                 for i, s in enumerate(specs)]
        self.plan = pulse.MxPlan(slots)

    def check(self, t, counts):
        o_c, o_s = host_u8(self.c0[t]), host_u8(self.s0[t])
        o_patch = oracle.mxfp8_encode(host_f32(self.master[t]), o_c, o_s)
        k, ks = int(counts[2 * t]), int(counts[2 * t + 1])
        assert (k, ks) == (o_patch[0].size, o_patch[2].size), t
        np.testing.assert_array_equal(host_u32(self.idx[t][:k]), o_patch[0])
        np.testing.assert_array_equal(host_u8(self.val[t][:k]), o_patch[1])
        np.testing.assert_array_equal(host_u32(self.sidx[t][:ks]), o_patch[2])
        np.testing.assert_array_equal(host_u8(self.sval[t][:ks]), o_patch[3])
        np.testing.assert_array_equal(host_u8(self.prev_c[t]), o_c)
        np.testing.assert_array_equal(host_u8(self.prev_s[t]), o_s)
        np.testing.assert_array_equal(host_u8(self.codes[t]), o_c)
        np.testing.assert_array_equal(host_u8(self.scales[t]), o_s)
        return k, ks

    def close(self):
        self.plan.close()
        for g in self.guards:
            g.check()


def test_initial_view_matches_oracle_quantize():
    dev = _dev()
    specs = workloads.CONFIGS[2]["specs"]()[-3:]
    model = MxModel(specs, 1, workloads.ETA_DEFAULT, dev)
    for t in range(len(specs)):
        o_c, o_s = oracle.mxfp8_quantize(host_f32(model.w0[t]))
        np.testing.assert_array_equal(host_u8(model.c0[t]), o_c)
        np.testing.assert_array_equal(host_u8(model.s0[t]), o_s)
    model.close()


@pytest.mark.parametrize("device_counts", [True, False])
def test_plan_small_tensors(device_counts):
    dev = _dev()
    specs = [workloads.TensorSpec(f"t{i}", (n,), "weight") for i, n in
             enumerate([5, 0, 32, 4096, 4097, 31, 3 * 4096 + 1, 1])]
    model = MxModel(specs, 17, 3e-4, dev)
    counts = model.plan.encode()
    model.plan.apply(counts if device_counts else counts.cpu().tolist())
    torch.cuda.synchronize()
    assert model.plan.get_error() == 0
    c = counts.cpu().numpy()
    for t in range(len(specs)):
        model.check(t, c)
    model.close()


def test_plan_llama_layer_density_and_parity():
    """One Llama-3-8B decoder layer (9 tensors, 218,112,000 params) at the
    BF16 workload's update (eta = 3e-6): every tensor bit-exact, and the
    MXFP8 view changes far less than the BF16 view (about 8% there)."""
    dev = _dev()
    cfg = workloads.CONFIGS[2]
    specs = cfg["specs"]()
    model = MxModel(specs, cfg["seed"], cfg["eta"], dev)
    counts = model.plan.encode()
    model.plan.apply(counts)
    torch.cuda.synchronize()
    assert model.plan.get_error() == 0
    c = counts.cpu().numpy()
    with ThreadPoolExecutor(WORKERS) as ex:
        ks = list(ex.map(lambda t: model.check(t, c), range(len(specs))))
    density = sum(k for k, _ in ks) / workloads.total_params(specs)
    assert 0.0 < density < 0.02, density
    model.close()
