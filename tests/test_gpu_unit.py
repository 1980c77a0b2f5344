"""GPU vs oracle, bit-exact, on small and edge-case inputs.

Every test runs the CUDA kernels through the C ABI (Python binding) and the
plain-C oracle on the same host copy of the inputs, and compares patch
indices, patch values, counts, refreshed prev, masks and applied weights bit
for bit. Sizes span several 4096-element tiles and ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import (Guarded, dev_f32, dev_u16, dev_u32, guarded_u16, host_u16, host_u32,
                            patch_of)

pytestmark = pytest.mark.gpu

TILE = 4096
SIZES = [1, 7, 8, 9, 31, 33, TILE - 1, TILE, TILE + 1, 3 * TILE + 5, 16 * TILE,
         (1 << 20) + 3]


def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _encode_both(master_np, prev_np, offset=0):
    """Runs GPU encode (optionally on views misaligned by `offset` elements)
    into guarded buffers and the oracle; returns (gpu_idx, gpu_val, k,
    gpu_prev, o_idx, o_val, o_prev)."""
    dev = _cuda()
    n = master_np.size
    gm = Guarded(n + offset, torch.float32, dev)
    gp = Guarded(n + offset, torch.int16, dev)
    gm.t.zero_()
    gp.t.zero_()
    gm.t[offset:] = dev_f32(master_np)
    gp.t[offset:] = dev_u16(prev_np)
    m_t, p_t = gm.t[offset:], gp.t[offset:]
    gi = Guarded(max(n, 1), torch.int32, dev)
    gv = Guarded(max(n, 1), torch.int16, dev)
    gc = Guarded(1, torch.int64, dev)
    idx_t, val_t, cnt_t = pulse.encode(m_t, p_t, idx_out=gi.t, val_out=gv.t, count_out=gc.t)
    torch.cuda.synchronize()
    g_idx, g_val, k = patch_of(idx_t, val_t, cnt_t)
    g_prev = host_u16(p_t)
    o_prev = prev_np.copy()
    o_idx, o_val = oracle.encode(master_np, o_prev)
    assert pulse.get_error() == 0
    for name, g in (("master", gm), ("prev", gp), ("idx", gi), ("val", gv), ("count", gc)):
        g.check(name)
    return g_idx, g_val, k, g_prev, o_idx, o_val, o_prev


def _assert_encode_parity(master_np, prev_np, offset=0):
    g_idx, g_val, k, g_prev, o_idx, o_val, o_prev = _encode_both(master_np, prev_np, offset)
    assert k == o_idx.size
    np.testing.assert_array_equal(g_idx, o_idx)
    np.testing.assert_array_equal(g_val, o_val)
    np.testing.assert_array_equal(g_prev, o_prev)
    return k


@pytest.mark.parametrize("n", SIZES)
def test_encode_parity_sizes(n):
    master, prev = workloads.np_pair(n, seed=1000 + n)
    k = _assert_encode_parity(master, prev)
    assert 0 < k < n or n < 64


def test_encode_empty():
    dev = _cuda()
    m = torch.empty(0, dtype=torch.float32, device=dev)
    p = torch.empty(0, dtype=torch.int16, device=dev)
    cnt = torch.full((1,), 12345, dtype=torch.int64, device=dev)
    pulse.encode(m, p, count_out=cnt)
    assert int(cnt.item()) == 0


@pytest.mark.parametrize("offset", [1, 2, 3, 4, 5, 6, 7])
def test_encode_misaligned_views(offset):
    n = 5 * TILE + 77
    master, prev = workloads.np_pair(n, seed=offset)
    _assert_encode_parity(master, prev, offset=offset)


@pytest.mark.parametrize("pattern", ["all", "none", "alternating", "last_only", "first_only",
                                     "tile_edges"])
def test_encode_change_patterns(pattern):
    n = 7 * TILE + 13
    rng = np.random.default_rng(5)
    master = (rng.standard_normal(n, dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    view = oracle.bf16_rne(master.view(np.uint32))
    prev = view.copy()
    if pattern == "all":
        prev ^= np.uint16(1)
    elif pattern == "alternating":
        prev[::2] ^= np.uint16(1)
    elif pattern == "last_only":
        prev[-1] ^= np.uint16(0x8000)
    elif pattern == "first_only":
        prev[0] ^= np.uint16(0x0040)
    elif pattern == "tile_edges":
        for t in range(0, n, TILE):
            prev[t] ^= np.uint16(1)
            prev[min(n - 1, t + TILE - 1)] ^= np.uint16(1)
    k = _assert_encode_parity(master, prev)
    expected = {"all": n, "none": 0, "alternating": (n + 1) // 2, "last_only": 1,
                "first_only": 1}.get(pattern)
    if expected is not None:
        assert k == expected


def test_encode_special_values():
    rng = np.random.default_rng(77)
    specials = np.array([0x00000000, 0x80000000, 0x00000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF,
                         0x7F7F7FFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0x7F800001, 0xFFC00000,
                         0x3F808000, 0x3F818000, 0x00018000, 0x3F800000, 0xBF800000, 0xFFFFFFFF],
                        dtype=np.uint32)
    n = 9 * TILE + 3
    bits = specials[rng.integers(0, specials.size, size=n)]
    master = bits.view(np.float32)
    pv = np.array([0x0000, 0x8000, 0x0001, 0x0080, 0x7F7F, 0x7F80, 0xFF80, 0x7FC0, 0x7FFF,
                   0x3F80, 0x3F82, 0xBF80], dtype=np.uint16)
    prev = pv[rng.integers(0, pv.size, size=n)]
    _assert_encode_parity(master, prev)


def test_encode_random_bit_patterns():
    # arbitrary FP32 bit patterns (every class) against arbitrary prev
    rng = np.random.default_rng(31337)
    n = 33 * TILE + 1
    master = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    prev = rng.integers(0, 1 << 16, size=n, dtype=np.uint64).astype(np.uint16)
    _assert_encode_parity(master, prev)


def test_encode_twice_second_patch_is_empty():
    dev = _cuda()
    master, prev = workloads.np_pair(10 * TILE + 9, seed=8)
    m_t, p_t = dev_f32(master), dev_u16(prev)
    _, _, c1 = pulse.encode(m_t, p_t)
    _, _, c2 = pulse.encode(m_t, p_t)
    assert int(c1.item()) > 0 and int(c2.item()) == 0


@pytest.mark.parametrize("n", [1, 9, TILE + 1, 3 * TILE + 5, (1 << 20) + 3])
def test_apply_parity_and_reconstruction(n):
    dev = _cuda()
    master, prev = workloads.np_pair(n, seed=2000 + n)
    o_prev = prev.copy()
    o_idx, o_val = oracle.encode(master, o_prev)
    w_np = prev.copy()
    gw = guarded_u16(w_np)
    pulse.apply(gw.t, dev_u32(o_idx), dev_u16(o_val), o_idx.size)
    oracle.apply(w_np, o_idx, o_val)
    got = host_u16(gw.t)
    np.testing.assert_array_equal(got, w_np)
    np.testing.assert_array_equal(got, o_prev)   # bit-identical to the new view
    # checked variant on the same inputs
    gw2 = guarded_u16(prev)
    pulse.apply(gw2.t, dev_u32(o_idx), dev_u16(o_val), o_idx.size, checked=True)
    np.testing.assert_array_equal(host_u16(gw2.t), w_np)
    assert pulse.get_error(dev) == 0
    gw.check("w")
    gw2.check("w (checked)")


def test_apply_misaligned_patch_views():
    dev = _cuda()
    n = 3 * TILE + 1
    master, prev = workloads.np_pair(n, seed=12)
    o_prev = prev.copy()
    o_idx, o_val = oracle.encode(master, o_prev)
    for off in (1, 2, 3):
        ib = torch.zeros(o_idx.size + off, dtype=torch.int32, device=dev)
        vb = torch.zeros(o_idx.size + off, dtype=torch.int16, device=dev)
        ib[off:] = dev_u32(o_idx)
        vb[off:] = dev_u16(o_val)
        gw = guarded_u16(prev)
        pulse.apply(gw.t, ib[off:], vb[off:], o_idx.size)
        np.testing.assert_array_equal(host_u16(gw.t), o_prev)
        gw.check("w")


def test_apply_checked_reports_out_of_range_and_skips_it():
    dev = _cuda()
    n = 1000
    w_np = np.arange(n, dtype=np.uint16)
    idx = np.array([3, n + 5, 10, 0xFFFFFFFF], dtype=np.uint32)
    val = np.array([7, 8, 9, 10], dtype=np.uint16)
    gw = guarded_u16(w_np)
    pulse.apply(gw.t, dev_u32(idx), dev_u16(val), idx.size, checked=True)
    assert pulse.get_error(dev) == pulse.pulse.PULSE_ERR_INDEX
    exp = w_np.copy()
    exp[3] = 7
    exp[10] = 9
    np.testing.assert_array_equal(host_u16(gw.t), exp)
    assert pulse.get_error(dev) == 0   # cleared
    gw.check("w")


@pytest.mark.parametrize("n", [1, 7, TILE - 1, TILE, TILE + 1, 5 * TILE + 3, (1 << 20) + 3])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_xor_parity(n, offset):
    dev = _cuda()
    master, prev = workloads.np_pair(n, seed=3000 + n)
    gm = Guarded(n + offset, torch.float32, dev)
    gp = Guarded(n + offset, torch.int16, dev)
    gm.t[offset:] = dev_f32(master)
    gp.t[offset:] = dev_u16(prev)
    m_t, p_t = gm.t[offset:], gp.t[offset:]
    gx = Guarded(n, torch.int16, dev)
    mask_t = pulse.xor_mask(m_t, p_t, mask_out=gx.t)
    o_prev = prev.copy()
    o_mask = oracle.xor_mask(master, o_prev)
    np.testing.assert_array_equal(host_u16(mask_t), o_mask)
    np.testing.assert_array_equal(host_u16(p_t), o_prev)
    gw = guarded_u16(prev)
    pulse.xor_apply(gw.t, mask_t)
    w_np = prev.copy()
    oracle.xor_apply(w_np, o_mask)
    np.testing.assert_array_equal(host_u16(gw.t), w_np)
    np.testing.assert_array_equal(host_u16(gw.t), o_prev)
    pulse.xor_apply(gw.t, mask_t)                                 # double XOR restores
    np.testing.assert_array_equal(host_u16(gw.t), prev)
    for name, g in (("master", gm), ("prev", gp), ("mask", gx), ("w", gw)):
        g.check(name)


def test_xor_and_patch_modes_agree():
    dev = _cuda()
    n = 37 * TILE + 11
    master, prev = workloads.np_pair(n, seed=42)
    m_t = dev_f32(master)
    p1, p2 = dev_u16(prev), dev_u16(prev)
    idx_t, val_t, cnt_t = pulse.encode(m_t, p1)
    mask_t = pulse.xor_mask(m_t, p2)
    g_idx, _, k = patch_of(idx_t, val_t, cnt_t)
    nz = np.nonzero(host_u16(mask_t))[0].astype(np.uint32)
    np.testing.assert_array_equal(nz, g_idx)
    assert torch.equal(p1, p2)


def test_exhaustive_fp32_patterns_through_the_gpu_cast():
    """Every FP32 bit pattern as master, twice. Against prev = 0 the patch
    lists exactly the patterns whose RNE view is not +0, with the oracle's
    values. Against prev = the oracle's RNE view of the same patterns the
    patch is empty and prev is left as it was."""
    dev = _cuda()
    chunk = 1 << 28
    gi = Guarded(chunk, torch.int32, dev)
    gv = Guarded(chunk, torch.int16, dev)
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device=dev)
        m_t = bits.to(torch.int32).view(torch.float32)   # wraps to the uint32 pattern
        del bits
        p_t = torch.zeros(chunk, dtype=torch.int16, device=dev)
        _, _, cnt = pulse.encode(m_t, p_t, idx_out=gi.t, val_out=gv.t)
        k = int(cnt.item())
        view = oracle.bf16_rne(np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32))
        exp_idx = np.nonzero(view)[0].astype(np.uint32)
        assert k == exp_idx.size, hex(start)
        np.testing.assert_array_equal(host_u32(gi.t[:k]), exp_idx)
        np.testing.assert_array_equal(host_u16(gv.t[:k]), view[exp_idx])
        np.testing.assert_array_equal(host_u16(p_t), view)
        # prev already holds the oracle's view: nothing changes
        p_t = dev_u16(view)
        _, _, cnt = pulse.encode(m_t, p_t, idx_out=gi.t, val_out=gv.t)
        assert int(cnt.item()) == 0, hex(start)
        np.testing.assert_array_equal(host_u16(p_t), view)
        del m_t, p_t
    assert pulse.get_error(dev) == 0
    gi.check("idx")
    gv.check("val")


def _host_mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def test_encode_and_apply_at_the_index_limit():
    """One tensor of 2^32 - 1 elements, the largest a uint32 index can
    address: the patch's indices reach past 2^31 and up to 2^32 - 2. At a
    small update (about 0.4 % changed) the whole patch, the refreshed prev and
    the applied w are compared with the oracle (run chunk-parallel on the host
    cores: the same scalar loops)."""
    from concurrent.futures import ThreadPoolExecutor
    dev = _cuda()
    n = (1 << 32) - 1
    if _host_mem_available() < (96 << 30):
        pytest.skip("needs about 96 GB of host memory for the oracle's copies")
    spec = workloads.single(n)[0]
    gen = workloads.torch_generator(dev, 4242)
    m_t = torch.empty(n, dtype=torch.float32, device=dev)
    workloads.torch_init_(m_t, spec, gen)
    p0_t = torch.empty(n, dtype=torch.int16, device=dev)
    workloads.torch_bf16_view_(p0_t, m_t)
    workloads.torch_update_(m_t, 1e-7, gen)
    master = m_t.cpu().numpy()
    p0 = host_u16(p0_t)
    prev_t = p0_t.clone()
    gi = Guarded(n, torch.int32, dev)
    gv = Guarded(n, torch.int16, dev)
    _, _, cnt = pulse.encode(m_t, prev_t, idx_out=gi.t, val_out=gv.t)
    k = int(cnt.item())
    del m_t
    w_t = p0_t
    pulse.apply(w_t, gi.t, gv.t, k)
    torch.cuda.synchronize()
    assert pulse.get_error(dev) == 0
    o_prev = p0.copy()
    with ThreadPoolExecutor(max_workers=16) as pool:
        o_idx, o_val = oracle.encode_chunked(master, o_prev, pool, 256)
    del master
    assert k == o_idx.size and k > n // 400
    assert int(o_idx[-1]) > (1 << 31)
    np.testing.assert_array_equal(host_u32(gi.t[:k]), o_idx)
    np.testing.assert_array_equal(host_u16(gv.t[:k]), o_val)
    del o_idx, o_val
    assert np.array_equal(host_u16(prev_t), o_prev)
    assert np.array_equal(host_u16(w_t), o_prev)
    gi.check("idx")
    gv.check("val")


def test_lookback_watchdog_gives_up_and_context_survives():
    # tile 0 is never processed, so tile 1's look-back waits for a word that
    # nothing publishes; the bounded wait must give up (50 ms) and report
    dev = _cuda()
    n = 40 * TILE
    master, prev = workloads.np_pair(n, seed=9)
    m_t, p_t = dev_f32(master), dev_u16(prev)
    # guard zone after the patch buffers: the timeout path must stay in bounds
    idx_buf = torch.full((n + 1024,), -7, dtype=torch.int32, device=dev)
    val_buf = torch.full((n + 1024,), -7, dtype=torch.int16, device=dev)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    st = pulse.pulse.debug_encode_orphan_tile(m_t, p_t, idx_buf, val_buf, cnt, 50_000_000)
    assert st == 0
    assert pulse.get_error(dev) == pulse.pulse.PULSE_ERR_TIMEOUT
    assert bool((idx_buf[n:] == -7).all()) and bool((val_buf[n:] == -7).all())
    assert pulse.get_error(dev) == 0
    # the same stream and workspace still produce correct results
    _assert_encode_parity(*workloads.np_pair(6 * TILE + 1, seed=10))


# ------------------------------------------------------------- multi-tensor

def _slots_from_np(masters, prevs, dev, offsets=None, with_w=True, with_mask=True):
    """Plan slots over device copies of (master, prev), optionally shifted by
    `offsets` elements from an aligned start. Every buffer sits between guard
    zones; returns (slots, guards) and the caller checks the guards."""
    slots, guards = [], []
    for i, (m, p) in enumerate(zip(masters, prevs)):
        off = 0 if offsets is None else offsets[i]
        n = m.size
        gm = Guarded(n + off, torch.float32, dev)
        gp = Guarded(n + off, torch.int16, dev)
        gm.t.zero_()
        gp.t.zero_()
        if n:
            gm.t[off:] = dev_f32(m)
            gp.t[off:] = dev_u16(p)
        gw = guarded_u16(p) if with_w else None
        gi = Guarded(max(n, 1), torch.int32, dev)
        gv = Guarded(max(n, 1), torch.int16, dev)
        gx = Guarded(n, torch.int16, dev) if with_mask else None
        s = pulse.TensorSlot(n, master=gm.t[off:], prev=gp.t[off:],
                             w=(gw.t if gw is not None else None), idx=gi.t, val=gv.t,
                             mask=(gx.t if gx is not None else None))
        slots.append(s)
        guards += [g for g in (gm, gp, gw, gi, gv, gx) if g is not None]
    return slots, guards


@pytest.mark.parametrize("aligned", [True, False])
def test_multi_tensor_plan_parity(aligned):
    dev = _cuda()
    rng = np.random.default_rng(123)
    sizes = [4096, 1, 0, 4097, 3 * TILE + 5, 12288, 9, 0, 65536 + 17, TILE - 1]
    masters, prevs = [], []
    for i, n in enumerate(sizes):
        m, p = workloads.np_pair(n, seed=500 + i) if n else (np.zeros(0, np.float32), np.zeros(0, np.uint16))
        masters.append(m)
        prevs.append(p)
    offsets = None if aligned else [int(x) for x in rng.integers(0, 8, size=len(sizes))]
    slots, keep = _slots_from_np(masters, prevs, dev, offsets)
    plan = pulse.Plan(slots)
    assert plan.num_tiles == sum((n + TILE - 1) // TILE for n in sizes)
    counts = plan.encode()
    o_prevs = [p.copy() for p in prevs]
    o_patches = oracle.encode_multi(masters, o_prevs)
    got_counts = counts.cpu().numpy()
    for t, (s, (o_idx, o_val)) in enumerate(zip(slots, o_patches)):
        assert got_counts[t] == o_idx.size, t
        g_idx, g_val, _ = patch_of(s.idx, s.val, o_idx.size)
        np.testing.assert_array_equal(g_idx, o_idx)
        np.testing.assert_array_equal(g_val, o_val)
        np.testing.assert_array_equal(host_u16(s.prev), o_prevs[t])
    # apply: device counts
    plan.apply(counts)
    for t, s in enumerate(slots):
        np.testing.assert_array_equal(host_u16(s.w), o_prevs[t])
    assert plan.get_error() == 0
    for g in keep:
        g.check()
    plan.close()


@pytest.mark.parametrize("eta", [1e-8, 3e-7, 1e-6, 1e-4])
@pytest.mark.parametrize("device_counts", [True, False])
def test_multi_apply_densities(eta, device_counts):
    """Whole-model apply from about 0.05 % to 70 % of the view changed
    (1e-4 also fills a tile with consecutive elements), with device and host
    counts: every segment gives the oracle's view and nothing lands outside
    w."""
    dev = _cuda()
    sizes = [3 * 8192 + 77, 1, 0, 65536 + 5, 8192, 200003]
    masters, prevs = [], []
    for i, n in enumerate(sizes):
        m, p = (workloads.np_pair(n, seed=900 + i, eta=eta) if n
                else (np.zeros(0, np.float32), np.zeros(0, np.uint16)))
        masters.append(m)
        prevs.append(p)
    slots, keep = _slots_from_np(masters, prevs, dev, with_mask=False)
    o_prevs = [p.copy() for p in prevs]
    o_patches = oracle.encode_multi(masters, o_prevs)
    with pulse.Plan(slots) as plan:
        counts = plan.encode()
        plan.apply(counts if device_counts else counts.cpu().numpy().tolist())
        torch.cuda.synchronize()
        for t, s in enumerate(slots):
            np.testing.assert_array_equal(host_u16(s.w), o_prevs[t])
        assert plan.get_error() == 0
        # the same patch again changes nothing; an index past its tensor is
        # skipped and reported
        plan.apply(counts if device_counts else counts.cpu().numpy().tolist())
        assert plan.get_error() == 0
        if o_patches[0][0].size:
            slots[0].idx[0] = sizes[0] + 100
            plan.apply(counts)
            assert plan.get_error() == pulse.pulse.PULSE_ERR_INDEX
        for t, s in enumerate(slots[1:], start=1):
            np.testing.assert_array_equal(host_u16(s.w), o_prevs[t])
    for g in keep:
        g.check()


@pytest.mark.parametrize("per_mille", [1, 15, 300])
@pytest.mark.parametrize("device_counts", [True, False])
def test_multi_apply_sorted_random_patch(per_mille, device_counts):
    """Sorted random patches (arbitrary values, not from an encode) whose
    segments hold room for n entries: the apply writes exactly the patch
    (oracle apply of the same entries) and nothing outside w."""
    dev = _cuda()
    sizes = [8192 * 5 + 11, 3 * 8192, 8192 + 1]
    rng = np.random.default_rng(321 + per_mille)
    slots, w0s, patches, guards = [], [], [], []
    for s in sizes:
        k = max(1, s * per_mille // 1000)
        w0 = rng.integers(0, 1 << 16, s, dtype=np.uint64).astype(np.uint16)
        idx = np.sort(rng.choice(s, size=k, replace=False)).astype(np.uint32)
        val = rng.integers(0, 1 << 16, k, dtype=np.uint64).astype(np.uint16)
        # segments with room for n entries (device counts are checked against that)
        idx_room, val_room = np.zeros(s, np.uint32), np.zeros(s, np.uint16)
        idx_room[:k], val_room[:k] = idx, val
        gw = guarded_u16(w0)
        slot = pulse.TensorSlot(s, w=gw.t, idx=dev_u32(idx_room), val=dev_u16(val_room))
        slots.append(slot)
        guards.append(gw)
        w0s.append(w0)
        patches.append((idx, val))
    with pulse.Plan(slots) as plan:
        counts = [int(p[0].size) for p in patches]
        plan.apply(torch.tensor(counts, dtype=torch.int64, device=dev) if device_counts else counts)
        torch.cuda.synchronize()
        assert plan.get_error() == 0
        for s, w0, (idx, val) in zip(slots, w0s, patches):
            want = w0.copy()
            oracle.apply(want, idx, val)
            np.testing.assert_array_equal(host_u16(s.w), want)
    for g in guards:
        g.check("w")


def test_multi_apply_host_counts_and_out_of_range_segment():
    dev = _cuda()
    sizes = [TILE + 3, 2 * TILE]
    masters, prevs = zip(*[workloads.np_pair(n, seed=60 + n) for n in sizes])
    slots, keep = _slots_from_np(list(masters), list(prevs), dev)
    plan = pulse.Plan(slots)
    counts = plan.encode().cpu().numpy().tolist()
    plan.apply(counts)
    o_prevs = [p.copy() for p in prevs]
    oracle.encode_multi(list(masters), o_prevs)
    for t, s in enumerate(slots):
        np.testing.assert_array_equal(host_u16(s.w), o_prevs[t])
    assert plan.get_error() == 0
    # an index past its tensor is skipped and reported
    slots[0].idx[0] = sizes[0] + 100
    plan.apply([1, 0])
    assert plan.get_error() == pulse.pulse.PULSE_ERR_INDEX
    # a count larger than the tensor is clamped and reported
    plan.apply([sizes[0] + 50, 0])
    assert plan.get_error() == pulse.pulse.PULSE_ERR_INDEX
    for g in keep:
        g.check()
    plan.close()


@pytest.mark.parametrize("aligned", [True, False])
def test_multi_xor_parity(aligned):
    dev = _cuda()
    sizes = [4096, 1, 0, 4097, 3 * TILE + 5, 9, 65536 + 17]
    masters, prevs = [], []
    for i, n in enumerate(sizes):
        m, p = workloads.np_pair(n, seed=700 + i) if n else (np.zeros(0, np.float32), np.zeros(0, np.uint16))
        masters.append(m)
        prevs.append(p)
    offsets = None if aligned else [1, 2, 3, 0, 5, 6, 7]
    slots, keep = _slots_from_np(masters, prevs, dev, offsets)
    plan = pulse.Plan(slots)
    plan.xor_mask()
    o_prevs = [p.copy() for p in prevs]
    o_masks = oracle.xor_mask_multi(masters, o_prevs)
    for t, s in enumerate(slots):
        np.testing.assert_array_equal(host_u16(s.mask), o_masks[t])
        np.testing.assert_array_equal(host_u16(s.prev), o_prevs[t])
    plan.xor_apply()
    for t, s in enumerate(slots):
        np.testing.assert_array_equal(host_u16(s.w), o_prevs[t])
    for g in keep:
        g.check()
    plan.close()


def test_plan_rejects_operations_without_buffers():
    dev = _cuda()
    m, p = workloads.np_pair(100, seed=1)
    slot = pulse.TensorSlot(100, master=dev_f32(m), prev=dev_u16(p),
                            idx=torch.empty(100, dtype=torch.int32, device=dev),
                            val=torch.empty(100, dtype=torch.int16, device=dev))
    plan = pulse.Plan([slot])
    with pytest.raises(pulse.PulseError):
        plan.xor_mask()
    with pytest.raises(pulse.PulseError):
        plan.apply([0])
    plan.encode()
    plan.close()
