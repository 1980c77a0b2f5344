"""pulse_encode_noalloc: the encode entry point for callers that must not
allocate device memory (its look-back scratch is a fixed array inside the
library instead of a workspace allocated on first use).

Its results must equal pulse_encode's bit for bit -- patch indices and
values in order, the count, and the refreshed prev -- on consecutive calls,
since every call reuses the same scratch array. Sizes past the array's limit
are refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import dev_f32, dev_u16, host_u16, host_u32, patch_of

pytestmark = pytest.mark.gpu

MAX_ELEMS = 268435456  # PULSE_NOALLOC_MAX_ELEMS in include/pulse.h
TILE = 4096


def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _both(master_np, prev_np):
    dev = _cuda()
    n = master_np.size
    m_t = dev_f32(master_np)
    # the existing entry point (allocating workspace)
    p_ref = dev_u16(prev_np)
    i_ref, v_ref, c_ref = pulse.encode(m_t, p_ref)
    # the allocation-free entry point, through the C ABI, with caller-owned outputs
    p_new = dev_u16(prev_np)
    i_new = torch.full((max(n, 1),), -1, dtype=torch.int32, device=dev)
    v_new = torch.full((max(n, 1),), -1, dtype=torch.int16, device=dev)
    c_new = torch.full((1,), -1, dtype=torch.int64, device=dev)
    pulse.encode_noalloc(m_t, p_new, i_new, v_new, c_new)
    torch.cuda.synchronize()
    ri, rv, rk = patch_of(i_ref, v_ref, c_ref)
    ni, nv, nk = patch_of(i_new, v_new, c_new)
    assert nk == rk
    np.testing.assert_array_equal(ni, ri)
    np.testing.assert_array_equal(nv, rv)
    np.testing.assert_array_equal(host_u16(p_new), host_u16(p_ref))
    return rk


def test_noalloc_equals_pulse_encode_on_two_calls_in_a_row():
    n = 7 * TILE + 123  # several tiles and a ragged tail
    m1, p1 = workloads.np_pair(n, seed=901)
    m2, p2 = workloads.np_pair(n, seed=902, eta=1e-5)
    k1 = _both(m1, p1)
    k2 = _both(m2, p2)
    assert k1 > 0 and k2 > k1  # a larger step changes more of the view


def test_noalloc_second_call_on_the_refreshed_view_is_empty():
    dev = _cuda()
    n = 3 * TILE + 5
    m, p = workloads.np_pair(n, seed=903)
    m_t, p_t = dev_f32(m), dev_u16(p)
    idx = torch.empty(n, dtype=torch.int32, device=dev)
    val = torch.empty(n, dtype=torch.int16, device=dev)
    cnt = torch.empty(1, dtype=torch.int64, device=dev)
    pulse.encode_noalloc(m_t, p_t, idx, val, cnt)
    assert int(cnt.item()) > 0
    pulse.encode_noalloc(m_t, p_t, idx, val, cnt)
    assert int(cnt.item()) == 0


def test_noalloc_refuses_sizes_past_its_scratch():
    dev = _cuda()
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    P = ctypes.c_void_p
    st = pulse.lib().pulse_encode_noalloc(P(0), P(0), MAX_ELEMS + 1, P(0), P(0),
                                          P(cnt.data_ptr()), P(0))
    assert st == pulse.pulse.PULSE_ERR_RANGE
    assert int(cnt.item()) == 0
