"""GPU vs oracle for codec-friendly index packing through the C ABI: every
output array bit for bit (firsts, widths, chunk offsets, payload bytes and
their total), and the GPU unpack of both the GPU's and the oracle's packing,
on all size edges, wide gaps, dense runs and a real encode patch."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_u32, host_u32

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _random_idx(rng, k, mean_gap, big=False):
    gaps = rng.geometric(1.0 / (mean_gap + 1), size=k).astype(np.uint64) - 1
    if big and k > 3:
        gaps[rng.integers(1, k, 3)] = rng.integers(1 << 20, 1 << 29, 3)
    idx = np.cumsum(gaps + 1, dtype=np.uint64) - 1
    return idx.astype(np.uint32)


class _GuardedAlloc:
    """Output buffers between guard zones, checked by check()."""

    def __init__(self):
        self.guards = []

    def __call__(self, numel, dtype, device):
        g = Guarded(numel, dtype, device)
        self.guards.append(g)
        return g.t

    def check(self):
        for g in self.guards:
            g.check()


def _check(idx_np, dev):
    k = idx_np.size
    t = dev_u32(idx_np, dev) if k else torch.empty(0, dtype=torch.int32, device=dev)
    alloc = _GuardedAlloc()
    firsts, widths, chunk_off, payload, nbytes = pulse.pack_indices(t, k, alloc=alloc)
    torch.cuda.synchronize()
    of, ow, oc, op = oracle.pack_indices(idx_np)
    nb, nc = of.size, oc.size
    size = int(nbytes.item())
    assert size == op.size
    np.testing.assert_array_equal(host_u32(firsts[:nb]), of)
    np.testing.assert_array_equal(widths[:nb].cpu().numpy(), ow)
    np.testing.assert_array_equal(chunk_off[:nc].cpu().numpy().view(np.uint64), oc)
    np.testing.assert_array_equal(payload[:size].cpu().numpy(), op)
    if k:
        back = pulse.unpack_indices(firsts, widths, chunk_off, payload, k,
                                    idx_out=alloc(k, torch.int32, dev))
        np.testing.assert_array_equal(host_u32(back[:k]), idx_np)
        # the oracle's packing, unpacked on the GPU
        op_dev = torch.zeros(max(op.size, 16), dtype=torch.uint8, device=dev)
        if op.size:
            op_dev[:op.size] = torch.from_numpy(op).to(dev)
        back2 = pulse.unpack_indices(dev_u32(of, dev), torch.from_numpy(ow).to(dev),
                                     torch.from_numpy(oc.view(np.int64)).to(dev), op_dev, k)
        np.testing.assert_array_equal(host_u32(back2[:k]), idx_np)
    assert pulse.get_error(dev) == 0
    alloc.check()
    return size


@pytest.mark.parametrize("k", [1, 2, 127, 128, 129, 4095, 4096, 4097, 40 * 4096 + 1234])
@pytest.mark.parametrize("mean_gap", [0, 11, 1000])
def test_pack_matches_oracle(k, mean_gap):
    dev = _dev()
    rng = np.random.default_rng(k + 7 * mean_gap)
    _check(_random_idx(rng, k, mean_gap, big=(mean_gap == 11)), dev)


def test_extremes_and_empty():
    dev = _dev()
    _check(np.array([0, 4294967294], np.uint32), dev)
    _check(np.arange(5000, 200000, dtype=np.uint32), dev)
    nbytes = pulse.pack_indices(torch.empty(0, dtype=torch.int32, device=dev), 0)[4]
    assert int(nbytes.item()) == 0


def test_pack_an_encode_patch():
    dev = _dev()
    spec = workloads.llama_layer()[0]   # q_proj, 16.8M params
    (m, p0), = workloads.torch_model([spec], seed=5, eta=workloads.ETA_DEFAULT, device=dev)
    idx, val, cnt = pulse.encode(m, p0)
    k = int(cnt.item())
    size = _check(host_u32(idx[:k]), dev)
    assert size < k   # under one byte per index at about 8 % density


def _check_job(segs_np, dev, offsets=None):
    """Pack a list of segments in one call (PackJob) and compare every
    segment's arrays with the oracle packing that segment alone; unpack
    them all in one call and compare with the input."""
    tens = []
    for i, a in enumerate(segs_np):
        off = 0 if offsets is None else offsets[i]
        buf = torch.zeros(a.size + off + 1, dtype=torch.int32, device=dev)
        if a.size:
            buf[off:off + a.size] = dev_u32(a, dev)
        tens.append((buf[off:], a.size))
    alloc = _GuardedAlloc()
    job = pulse.PackJob(tens, alloc=alloc)
    sizes = job.pack()
    outs = job.unpack()
    torch.cuda.synchronize()
    assert pulse.get_error(dev) == 0
    sizes = sizes.cpu().tolist()
    for a, (firsts, widths, chunk_off, payload), size, back in zip(segs_np, job.packed, sizes, outs):
        of, ow, oc, op = oracle.pack_indices(a)
        nb, nc = of.size, oc.size
        assert size == op.size
        np.testing.assert_array_equal(host_u32(firsts[:nb]), of)
        np.testing.assert_array_equal(widths[:nb].cpu().numpy(), ow)
        np.testing.assert_array_equal(chunk_off[:nc].cpu().numpy().view(np.uint64), oc)
        np.testing.assert_array_equal(payload[:size].cpu().numpy(), op)
        np.testing.assert_array_equal(host_u32(back[:a.size]), a)
    alloc.check()


def test_pack_job_many_segments():
    """Segments of every size edge (empty ones included) in one call: the
    look-back restarts at each segment's first chunk."""
    dev = _dev()
    rng = np.random.default_rng(77)
    ks = [0, 1, 2, 127, 128, 129, 0, 4095, 4096, 4097, 3 * 4096 + 5, 100000, 0, 7]
    segs = [_random_idx(rng, k, int(rng.choice([0, 11, 1000])), big=bool(i % 3 == 0))
            for i, k in enumerate(ks)]
    _check_job(segs, dev)


def test_pack_job_unaligned_inputs_and_model_patch():
    """A model's patch (one segment per tensor, from a GPU encode) with
    index views that start at odd word offsets."""
    dev = _dev()
    rng = np.random.default_rng(5)
    specs = workloads.llama_layer()
    segs = []
    for s in specs:
        n = s.numel // 16
        w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        prev = oracle.bf16_rne(w0.view(np.uint32)).astype(np.uint16)
        w1 = (w0 + np.float32(3e-6) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
        idx, _ = oracle.encode(w1, prev)
        segs.append(idx)
    _check_job(segs, dev, offsets=[i % 4 for i in range(len(segs))])


def test_pack_job_all_empty():
    dev = _dev()
    job = pulse.PackJob([(torch.zeros(1, dtype=torch.int32, device=dev), 0)] * 3)
    assert job.pack().cpu().tolist() == [0, 0, 0]
    job.unpack()
    torch.cuda.synchronize()
    assert pulse.get_error(dev) == 0


def test_segments_spanning_several_scan_tiles():
    """Segments of more than 1024 chunks (4,194,304 entries), alone and in
    one job: long look-back chains within a segment, restarted at each one."""
    dev = _dev()
    rng = np.random.default_rng(99)
    big = 2 * 1024 * 4096 + 4096 * 3 + 17   # three scan tiles
    _check(_random_idx(rng, big, 11), dev)
    segs = [_random_idx(rng, 1024 * 4096 + 1, 5), _random_idx(rng, 300, 1000),
            _random_idx(rng, big, 0)]
    _check_job(segs, dev)


def test_pack_job_more_segments_than_the_shared_table():
    """1100 segments in one call: past the pack kernel's shared copy of the
    segments' chunk ranges (1024 entries), each chunk's segment is found by
    a binary search of the global table."""
    dev = _dev()
    rng = np.random.default_rng(1100)
    ks = [int(k) for k in rng.choice([0, 1, 127, 128, 129, 300, 4096, 4097, 9000], size=1100)]
    segs = [_random_idx(rng, k, int(rng.choice([0, 11, 1000]))) for k in ks]
    _check_job(segs, dev)
