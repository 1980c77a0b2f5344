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
from pulse_testutil import dev_u32, host_u32

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


def _check(idx_np, dev):
    k = idx_np.size
    t = dev_u32(idx_np, dev) if k else torch.empty(0, dtype=torch.int32, device=dev)
    firsts, widths, chunk_off, payload, nbytes = pulse.pack_indices(t, k)
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
        back = pulse.unpack_indices(firsts, widths, chunk_off, payload, k)
        np.testing.assert_array_equal(host_u32(back[:k]), idx_np)
        # the oracle's packing, unpacked on the GPU
        op_dev = torch.zeros(max(op.size, 16), dtype=torch.uint8, device=dev)
        if op.size:
            op_dev[:op.size] = torch.from_numpy(op).to(dev)
        back2 = pulse.unpack_indices(dev_u32(of, dev), torch.from_numpy(ow).to(dev),
                                     torch.from_numpy(oc.view(np.int64)).to(dev), op_dev, k)
        np.testing.assert_array_equal(host_u32(back2[:k]), idx_np)
    assert pulse.get_error(dev) == 0
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
