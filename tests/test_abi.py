"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/pulse.h declares, and rejects bad arguments on the
host before any CUDA call (no compute calls: this machine may have no GPU)."""
import ctypes
import subprocess

import pytest

import rl_post_trainer_gb300 as pulse
from rl_post_trainer_gb300 import _build
from pulse_testutil import header_functions


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pulse.lib()


def test_header_declares_the_expected_entry_points():
    names = header_functions()
    for must in ("pulse_encode", "pulse_apply", "pulse_xor_mask", "pulse_xor_apply",
                 "pulse_plan_create", "pulse_encode_multi", "pulse_apply_multi",
                 "pulse_xor_mask_multi", "pulse_xor_apply_multi", "pulse_get_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported


def test_build_targets_sm_103a_only():
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_error_strings(lib):
    for code in range(0, 7):
        s = pulse.error_string(code)
        assert s.startswith("PULSE_")
    assert pulse.error_string(4).startswith("PULSE_ERR_TIMEOUT")
    assert pulse.error_string(99) == "PULSE_ERR_UNKNOWN"


def test_tile_constant(lib):
    assert pulse.tile_elems() == 4096


def test_host_side_argument_checks_launch_nothing(lib):
    P = ctypes.c_void_p
    # null count_out, null pointers with n > 0, n >= 2^32: rejected before CUDA is touched
    assert lib.pulse_encode(P(0), P(0), 5, P(0), P(0), P(0), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_encode(P(0), P(0), 1 << 32, P(0), P(0), P(8), P(0)) == pulse.pulse.PULSE_ERR_RANGE
    assert lib.pulse_encode(P(0), P(0), 5, P(0), P(0), P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_apply(P(0), P(0), P(0), 0, P(0)) == pulse.pulse.PULSE_OK       # empty patch: no-op
    assert lib.pulse_apply(P(0), P(0), P(0), 3, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_apply_checked(P(0), 4, P(0), P(0), 3, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_xor_mask(P(0), P(0), 0, P(0), P(0)) == pulse.pulse.PULSE_OK
    assert lib.pulse_xor_mask(P(0), P(0), 9, P(0), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_xor_mask(P(0), P(0), 1 << 32, P(0), P(0)) == pulse.pulse.PULSE_ERR_RANGE
    assert lib.pulse_xor_apply(P(0), P(0), 9, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_xor_apply(P(0), P(0), 1 << 32, P(0)) == pulse.pulse.PULSE_ERR_RANGE
    # plans
    h = P()
    assert lib.pulse_plan_create(None, 0, ctypes.byref(h)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_plan_create(None, 1, None) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_plan_destroy(None) == pulse.pulse.PULSE_OK
    assert lib.pulse_plan_num_tensors(None) == 0
    assert lib.pulse_plan_num_tiles(None) == 0
    assert lib.pulse_encode_multi(None, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_apply_multi(None, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_apply_multi_device(None, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    segs = (pulse.pulse.PulsePackSegment * 1)()
    assert lib.pulse_pack_indices_multi(None, 1, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_pack_indices_multi(segs, 0, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_pack_indices_multi(segs, 1, None, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    segs[0].count = 5  # a non-empty segment with NULL buffers
    assert lib.pulse_pack_indices_multi(segs, 1, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_unpack_indices_multi(segs, 1, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    segs[0].count = 1 << 32
    assert lib.pulse_unpack_indices_multi(segs, 1, P(0)) == pulse.pulse.PULSE_ERR_RANGE
    refs = (pulse.pulse.PulsePatchRef * 1)()
    outs = (pulse.pulse.PulsePatchOut * 1)()
    assert lib.pulse_compose_chain_multi(None, refs, 1, outs, P(8), P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_apply_chain_multi(None, refs, 1, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_apply_chain_multi(None, None, 1, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_xor_mask_multi(None, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_xor_apply_multi(None, P(0)) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_plan_get_error(None) == pulse.pulse.PULSE_ERR_INVALID
    assert lib.pulse_debug_encode_orphan_tile(P(0), P(0), 100, P(0), P(0), P(8), 10, P(0)) \
        == pulse.pulse.PULSE_ERR_INVALID


def test_binding_rejects_cpu_tensors(lib):
    import torch
    m = torch.zeros(8, dtype=torch.float32)
    p = torch.zeros(8, dtype=torch.int16)
    with pytest.raises(TypeError):
        pulse.encode(m, p)
    with pytest.raises(TypeError):
        pulse.xor_mask(m, p)


def test_mx_host_side_argument_checks_launch_nothing(lib):
    P = ctypes.c_void_p
    E = pulse.pulse
    assert lib.pulse_mx_quantize(P(0), 0, P(0), P(0), P(0)) == E.PULSE_OK
    assert lib.pulse_mx_quantize(P(0), 7, P(0), P(0), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_quantize_fmt(2, P(8), 7, P(8), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_quantize_fmt(1, P(0), 7, P(0), P(0), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_encode_fmt(5, P(8), P(8), P(8), 5, P(8), P(8), P(8), P(8), P(8), P(0)) \
        == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_apply_fmt(-1, P(8), P(8), 5, P(8), P(8), 1, P(8), P(8), 1, P(0)) \
        == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_plan_create_fmt(None, 1, 1, None) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_quantize_fmt(2, P(8), 7, P(8), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_nvfp4_quantize(P(8), 7, P(8), P(8), None, P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_nvfp4_encode(P(8), P(8), P(8), 7, P(8), P(8), P(8), P(8), P(8), None, P(0)) \
        == E.PULSE_ERR_INVALID
    assert lib.pulse_nvfp4_encode_multi(None, P(8), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_quantize(P(0), 1 << 32, P(0), P(0), P(0)) == E.PULSE_ERR_RANGE
    assert lib.pulse_mx_encode(P(0), P(0), P(0), 5, P(0), P(0), P(0), P(0), P(0), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_encode(P(0), P(0), P(0), 5, P(0), P(0), P(0), P(0), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_encode(P(0), P(0), P(0), 1 << 32, P(0), P(0), P(0), P(0), P(8), P(0)) == E.PULSE_ERR_RANGE
    assert lib.pulse_mx_apply(P(0), P(0), 10, P(0), P(0), 0, P(0), P(0), 0, P(0)) == E.PULSE_OK
    assert lib.pulse_mx_apply(P(0), P(0), 10, P(0), P(0), 2, P(0), P(0), 0, P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_apply(P(0), P(0), 10, P(0), P(0), 0, P(0), P(0), 1, P(0)) == E.PULSE_ERR_INVALID
    h = P()
    assert lib.pulse_mx_plan_create(None, 0, ctypes.byref(h)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_plan_create(None, 1, None) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_encode_multi(None, P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_apply_multi(None, P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_apply_multi_device(None, P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_mx_plan_destroy(None) == E.PULSE_OK
    assert lib.pulse_mx_plan_num_tensors(None) == 0


def test_compose_host_side_argument_checks_launch_nothing(lib):
    P = ctypes.c_void_p
    E = pulse.pulse
    assert lib.pulse_compose(P(0), P(0), 0, P(0), P(0), 0, P(0), P(0), P(0), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_compose(P(0), P(0), 3, P(0), P(0), 0, P(0), P(0), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_compose(P(8), P(8), 3, P(0), P(0), 0, P(0), P(0), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_compose(P(8), P(8), 1 << 32, P(0), P(0), 0, P(8), P(8), P(8), P(0)) == E.PULSE_ERR_RANGE
    assert lib.pulse_compose_u8(P(0), P(0), 0, P(0), P(0), 2, P(0), P(0), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_compose_multi(None, 1, 2, P(8), P(0)) == E.PULSE_ERR_INVALID
    seg = (pulse.pulse.PulseComposeSegment * 1)()
    assert lib.pulse_compose_multi(seg, 1, 3, P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_compose_multi(seg, 0, 2, P(8), P(0)) == E.PULSE_ERR_INVALID
    seg[0].count_a = 5
    assert lib.pulse_compose_multi(seg, 1, 2, P(8), P(0)) == E.PULSE_ERR_INVALID


def test_loco_host_side_argument_checks_launch_nothing(lib):
    P = ctypes.c_void_p
    E = pulse.pulse
    assert lib.pulse_loco_gate(P(0), P(0), P(0), 4, P(0), P(0), P(0), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_loco_gate(P(0), P(0), P(0), 4, P(0), P(0), P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_loco_gate(P(0), P(0), P(0), 1 << 32, P(0), P(0), P(8), P(0)) == E.PULSE_ERR_RANGE
    assert lib.pulse_loco_accumulate(P(0), 4, P(0), P(0), 0, P(0)) == E.PULSE_OK
    assert lib.pulse_loco_accumulate(P(0), 4, P(0), P(0), 2, P(0)) == E.PULSE_ERR_INVALID
    h = P()
    assert lib.pulse_loco_plan_create(None, 1, ctypes.byref(h)) == E.PULSE_ERR_INVALID
    assert lib.pulse_loco_gate_multi(None, P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_loco_accumulate_multi(None, P(8), P(0)) == E.PULSE_ERR_INVALID
    assert lib.pulse_loco_plan_destroy(None) == E.PULSE_OK
