"""pulse_encode_noalloc: the encode entry point for callers that must not
allocate device memory (its look-back scratch is a fixed array inside the
library instead of a workspace allocated on first use).

Its results must equal the CPU oracle's and pulse_encode's bit for bit --
patch indices and values in order, the count, and the refreshed prev -- on
consecutive calls, since every call reuses the same scratch array: a smaller
call after a larger one, unaligned views, and a tensor of exactly the array's
limit. Every output buffer sits between guard zones that must stay intact.
Sizes past the limit are refused before anything is launched.

This file is collected last (pytest orders files by name), so a run that stops
at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
import workloads
from pulse_testutil import Guarded, dev_f32, dev_u16, guarded_u16, host_u16, host_u32, patch_of

pytestmark = pytest.mark.gpu

MAX_ELEMS = 268435456  # PULSE_NOALLOC_MAX_ELEMS in include/pulse.h
TILE = 4096


def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _check_against_both(m_t, prev_np, master_np=None):
    """One noalloc call on (m_t, prev_np) with guarded outputs, checked against
    the oracle and against pulse_encode. Returns k."""
    dev = _cuda()
    n = m_t.numel()
    if master_np is None:
        master_np = m_t.cpu().numpy()
    o_prev = prev_np.copy()
    o_idx, o_val = oracle.encode(master_np, o_prev)
    # the existing entry point (allocating workspace)
    p_ref = dev_u16(prev_np)
    i_ref, v_ref, c_ref = pulse.encode(m_t, p_ref)
    # the allocation-free entry point, through the C ABI, with caller-owned outputs
    p_new = guarded_u16(prev_np)
    i_new = Guarded(max(n, 1), torch.int32, dev)
    v_new = Guarded(max(n, 1), torch.int16, dev)
    c_new = Guarded(1, torch.int64, dev)
    pulse.encode_noalloc(m_t, p_new.t, i_new.t, v_new.t, c_new.t)
    torch.cuda.synchronize()
    ri, rv, rk = patch_of(i_ref, v_ref, c_ref)
    ni, nv, nk = patch_of(i_new.t, v_new.t, c_new.t)
    assert nk == o_idx.size == rk
    np.testing.assert_array_equal(ni, o_idx)
    np.testing.assert_array_equal(nv, o_val)
    np.testing.assert_array_equal(ni, ri)
    np.testing.assert_array_equal(nv, rv)
    np.testing.assert_array_equal(host_u16(p_new.t), o_prev)
    np.testing.assert_array_equal(host_u16(p_new.t), host_u16(p_ref))
    for name, b in (("prev", p_new), ("idx", i_new), ("val", v_new), ("count", c_new)):
        b.check(name)
    return nk


def test_noalloc_equals_oracle_and_pulse_encode_on_two_calls_in_a_row():
    n = 7 * TILE + 123  # several tiles and a ragged tail
    m1, p1 = workloads.np_pair(n, seed=901)
    m2, p2 = workloads.np_pair(n, seed=902, eta=1e-5)
    k1 = _check_against_both(dev_f32(m1), p1, m1)
    k2 = _check_against_both(dev_f32(m2), p2, m2)
    assert k1 > 0 and k2 > k1  # a larger step changes more of the view


def test_noalloc_smaller_call_after_a_larger_one():
    # the second call reads only status words it cleared itself, not the
    # larger first call's
    big, small = 40 * TILE + 7, 3 * TILE + 1
    m1, p1 = workloads.np_pair(big, seed=904)
    m2, p2 = workloads.np_pair(small, seed=905)
    assert _check_against_both(dev_f32(m1), p1, m1) > 0
    assert _check_against_both(dev_f32(m2), p2, m2) > 0
    assert _check_against_both(dev_f32(m1), p1, m1) > 0


@pytest.mark.parametrize("offset", [1, 3])
def test_noalloc_unaligned_views(offset):
    # master and prev not 16-byte aligned: the per-element load path
    n = 5 * TILE + 77
    m, p = workloads.np_pair(n + offset, seed=906 + offset)
    m_full = dev_f32(m)
    m_t = m_full[offset:]
    assert m_t.data_ptr() % 16 != 0
    assert _check_against_both(m_t, p[offset:].copy(), m[offset:].copy()) > 0


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


def test_noalloc_at_its_size_limit():
    # n = PULSE_NOALLOC_MAX_ELEMS: every status word of the array is used
    dev = _cuda()
    n = MAX_ELEMS
    spec = workloads.single(n)[0]
    gen = workloads.torch_generator(dev, 907)
    w0 = torch.empty(n, dtype=torch.float32, device=dev)
    workloads.torch_init_(w0, spec, gen)
    prev = torch.empty(n, dtype=torch.int16, device=dev)
    workloads.torch_bf16_view_(prev, w0)
    workloads.torch_update_(w0, workloads.ETA_DEFAULT, gen)
    prev_np = host_u16(prev)
    del prev
    k = _check_against_both(w0, prev_np)
    assert k > n // 20  # about 8 % of the view changes at this update scale


def test_noalloc_refuses_sizes_past_its_scratch():
    dev = _cuda()
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    P = ctypes.c_void_p
    st = pulse.lib().pulse_encode_noalloc(P(0), P(0), MAX_ELEMS + 1, P(0), P(0),
                                          P(cnt.data_ptr()), P(0))
    assert st == pulse.pulse.PULSE_ERR_RANGE
    assert int(cnt.item()) == 0
