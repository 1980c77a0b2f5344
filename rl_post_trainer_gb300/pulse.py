"""Python binding of libpulse (include/pulse.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module only
checks tensor types, allocates outputs with torch, and passes raw device
pointers plus torch's current CUDA stream through ctypes. There is no CPU
fallback: if the library is not built, every call raises.

Dtypes: FP32 master weights are ``torch.float32``; BF16 views, patch values
and masks may be ``torch.bfloat16``, ``torch.int16`` or ``torch.uint16``
(their bit patterns are used); patch indices are ``torch.int32`` holding
uint32 values; counts are ``torch.int64`` holding uint64 values.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import _build

PULSE_OK = 0
PULSE_ERR_INVALID = 1
PULSE_ERR_RANGE = 2
PULSE_ERR_CUDA = 3
PULSE_ERR_TIMEOUT = 4
PULSE_ERR_INDEX = 5
PULSE_ERR_NOMEM = 6

_U16 = (torch.bfloat16, torch.int16, torch.uint16)
_lib = None


class PulseError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {error_string(status)}")


class PulseTensor(ctypes.Structure):
    _fields_ = [
        ("master", ctypes.c_void_p),
        ("prev", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("n", ctypes.c_uint64),
        ("idx", ctypes.c_void_p),
        ("val", ctypes.c_void_p),
        ("mask", ctypes.c_void_p),
    ]


class PulseMxTensor(ctypes.Structure):
    _fields_ = [
        ("master", ctypes.c_void_p),
        ("prev_codes", ctypes.c_void_p),
        ("prev_scales", ctypes.c_void_p),
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("n", ctypes.c_uint64),
        ("idx", ctypes.c_void_p),
        ("val", ctypes.c_void_p),
        ("sidx", ctypes.c_void_p),
        ("sval", ctypes.c_void_p),
    ]


MX_BLOCK = 32
MX_E4M3 = 0  # MXFP8 view: one E4M3 code per byte
MX_E2M1 = 1  # MXFP4 view: two E2M1 codes per byte, element 2j in the low nibble
MX_NVFP4 = 2  # NVFP4 view: E2M1 codes as MXFP4, E4M3 scale per 16, FP32 scale per tensor
_U8 = (torch.uint8, torch.int8)


def mx_blocks(n: int) -> int:
    """Scale bytes of an n-element MX view."""
    return (int(n) + MX_BLOCK - 1) // MX_BLOCK


def mx_code_bytes(n: int, fmt: int = MX_E4M3) -> int:
    """Code bytes of an n-element MX view of format ``fmt``."""
    if fmt not in (MX_E4M3, MX_E2M1, MX_NVFP4):
        raise ValueError(f"unknown MX format {fmt}")
    return int(n) if fmt == MX_E4M3 else (int(n) + 1) // 2


def mx_scale_count(n: int, fmt: int = MX_E4M3) -> int:
    """Block scales of an n-element view of format ``fmt`` (16 elements per
    scale for NVFP4, 32 for the MX formats)."""
    mx_code_bytes(n, fmt)  # checks the format
    block = 16 if fmt == MX_NVFP4 else MX_BLOCK
    return (int(n) + block - 1) // block


class PulseComposeSegment(ctypes.Structure):
    _fields_ = [
        ("idx_a", ctypes.c_void_p),
        ("val_a", ctypes.c_void_p),
        ("count_a", ctypes.c_uint64),
        ("idx_b", ctypes.c_void_p),
        ("val_b", ctypes.c_void_p),
        ("count_b", ctypes.c_uint64),
        ("idx_out", ctypes.c_void_p),
        ("val_out", ctypes.c_void_p),
    ]


class PulsePatchRef(ctypes.Structure):
    _fields_ = [
        ("idx", ctypes.c_void_p),
        ("val", ctypes.c_void_p),
        ("count", ctypes.c_uint64),
    ]


class PulsePackSegment(ctypes.Structure):
    _fields_ = [
        ("idx", ctypes.c_void_p),
        ("count", ctypes.c_uint64),
        ("firsts", ctypes.c_void_p),
        ("widths", ctypes.c_void_p),
        ("chunk_off", ctypes.c_void_p),
        ("payload", ctypes.c_void_p),
    ]


class PulsePatchOut(ctypes.Structure):
    _fields_ = [
        ("idx", ctypes.c_void_p),
        ("val", ctypes.c_void_p),
        ("room", ctypes.c_uint64),
    ]


class PulseLocoTensor(ctypes.Structure):
    _fields_ = [
        ("global_w", ctypes.c_void_p),
        ("local_w", ctypes.c_void_p),
        ("err", ctypes.c_void_p),
        ("n", ctypes.c_uint64),
        ("idx", ctypes.c_void_p),
        ("val", ctypes.c_void_p),
        ("acc", ctypes.c_void_p),
    ]


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libpulse.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        P, U64, I = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int
        sigs = {
            "pulse_error_string": ([I], ctypes.c_char_p),
            "pulse_encode_tile_elems": ([], ctypes.c_uint32),
            "pulse_encode": ([P, P, U64, P, P, P, P], I),
            "pulse_apply": ([P, P, P, U64, P], I),
            "pulse_apply_checked": ([P, U64, P, P, U64, P], I),
            "pulse_xor_mask": ([P, P, U64, P, P], I),
            "pulse_xor_apply": ([P, P, U64, P], I),
            "pulse_get_error": ([P], I),
            "pulse_plan_create": ([ctypes.POINTER(PulseTensor), I, ctypes.POINTER(P)], I),
            "pulse_plan_destroy": ([P], I),
            "pulse_plan_num_tensors": ([P], I),
            "pulse_plan_num_tiles": ([P], U64),
            "pulse_encode_multi": ([P, P, P], I),
            "pulse_apply_multi": ([P, P, P], I),
            "pulse_apply_multi_device": ([P, P, P], I),
            "pulse_apply_chain_multi": ([P, ctypes.POINTER(PulsePatchRef), I, P], I),
            "pulse_compose_chain_multi": ([P, ctypes.POINTER(PulsePatchRef), I,
                                           ctypes.POINTER(PulsePatchOut), P, P], I),
            "pulse_xor_mask_multi": ([P, P], I),
            "pulse_xor_apply_multi": ([P, P], I),
            "pulse_plan_get_error": ([P], I),
            "pulse_debug_encode_orphan_tile": ([P, P, U64, P, P, P, U64, P], I),
            "pulse_encode_noalloc": ([P, P, U64, P, P, P, P], I),
            "pulse_compose": ([P, P, U64, P, P, U64, P, P, P, P], I),
            "pulse_compose_u8": ([P, P, U64, P, P, U64, P, P, P, P], I),
            "pulse_compose_multi": ([ctypes.POINTER(PulseComposeSegment), I, I, P, P], I),
            "pulse_loco_gate": ([P, P, P, U64, P, P, P, P], I),
            "pulse_loco_accumulate": ([P, U64, P, P, U64, P], I),
            "pulse_loco_plan_create": ([ctypes.POINTER(PulseLocoTensor), I, ctypes.POINTER(P)], I),
            "pulse_loco_plan_destroy": ([P], I),
            "pulse_loco_gate_multi": ([P, P, P], I),
            "pulse_loco_accumulate_multi": ([P, P, P], I),
            "pulse_loco_plan_get_error": ([P], I),
            "pulse_pack_indices": ([P, U64, P, P, P, P, P, P], I),
            "pulse_unpack_indices": ([P, P, P, P, U64, P, P], I),
            "pulse_pack_indices_multi": ([ctypes.POINTER(PulsePackSegment), I, P, P], I),
            "pulse_unpack_indices_multi": ([ctypes.POINTER(PulsePackSegment), I, P], I),
            "pulse_mx_quantize": ([P, U64, P, P, P], I),
            "pulse_mx_encode": ([P, P, P, U64, P, P, P, P, P, P], I),
            "pulse_mx_apply": ([P, P, U64, P, P, U64, P, P, U64, P], I),
            "pulse_mx_plan_create": ([ctypes.POINTER(PulseMxTensor), I, ctypes.POINTER(P)], I),
            "pulse_mx_plan_destroy": ([P], I),
            "pulse_mx_plan_num_tensors": ([P], I),
            "pulse_mx_encode_multi": ([P, P, P], I),
            "pulse_mx_apply_multi": ([P, P, P], I),
            "pulse_mx_apply_multi_device": ([P, P, P], I),
            "pulse_mx_plan_get_error": ([P], I),
            "pulse_mx_quantize_fmt": ([I, P, U64, P, P, P], I),
            "pulse_mx_encode_fmt": ([I, P, P, P, U64, P, P, P, P, P, P], I),
            "pulse_mx_apply_fmt": ([I, P, P, U64, P, P, U64, P, P, U64, P], I),
            "pulse_mx_plan_create_fmt": ([ctypes.POINTER(PulseMxTensor), I, I, ctypes.POINTER(P)], I),
            "pulse_nvfp4_quantize": ([P, U64, P, P, P, P], I),
            "pulse_nvfp4_encode": ([P, P, P, U64, P, P, P, P, P, P, P], I),
            "pulse_nvfp4_encode_multi": ([P, P, P, P], I),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def error_string(status: int) -> str:
    return lib().pulse_error_string(int(status)).decode()


def _raise(status: int, where: str):
    if status != PULSE_OK:
        raise PulseError(status, where)


def tile_elems() -> int:
    return int(lib().pulse_encode_tile_elems())


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtypes, device=None, numel=None, min_numel=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise TypeError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise TypeError(f"{name}: must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name}: {t.numel()} elements, need at least {min_numel}")


# ------------------------------------------------------------ single tensor

def encode(master: torch.Tensor, prev: torch.Tensor, idx_out: Optional[torch.Tensor] = None,
           val_out: Optional[torch.Tensor] = None, count_out: Optional[torch.Tensor] = None):
    """pulse_encode: returns (idx, val, count); refreshes ``prev`` in place.

    ``idx``/``val`` have room for n entries; the patch is their first
    ``count`` entries (``count`` is a 1-element device int64 tensor).
    """
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    _need(prev, "prev", _U16, dev, n)
    if idx_out is None:
        idx_out = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
    if val_out is None:
        val_out = torch.empty(max(n, 1), dtype=torch.int16, device=dev)
    if count_out is None:
        count_out = torch.empty(1, dtype=torch.int64, device=dev)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=n)
    _need(val_out, "val_out", _U16, dev, min_numel=n)
    _need(count_out, "count_out", (torch.int64, torch.uint64), dev, min_numel=1)
    with torch.cuda.device(dev):
        st = lib().pulse_encode(_ptr(master), _ptr(prev), n, _ptr(idx_out), _ptr(val_out),
                                _ptr(count_out), _stream(dev))
    _raise(st, "pulse_encode")
    return idx_out, val_out, count_out


def encode_noalloc(master: torch.Tensor, prev: torch.Tensor, idx_out: torch.Tensor,
                   val_out: torch.Tensor, count_out: torch.Tensor):
    """pulse_encode_noalloc: as encode, for callers that must not allocate device
    memory (the library uses a fixed internal scratch array instead of a
    cudaMalloc'd workspace). The caller passes every output buffer; n is at most
    2^28. A count of 2^64 - 1 means a device wait gave up."""
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    _need(prev, "prev", _U16, dev, n)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=n)
    _need(val_out, "val_out", _U16, dev, min_numel=n)
    _need(count_out, "count_out", (torch.int64, torch.uint64), dev, min_numel=1)
    with torch.cuda.device(dev):
        st = lib().pulse_encode_noalloc(_ptr(master), _ptr(prev), n, _ptr(idx_out), _ptr(val_out),
                                        _ptr(count_out), _stream(dev))
    _raise(st, "pulse_encode_noalloc")
    return idx_out, val_out, count_out


def apply(w: torch.Tensor, idx: torch.Tensor, val: torch.Tensor, count: int, checked: bool = False):
    """pulse_apply / pulse_apply_checked: w[idx[j]] = val[j] for j < count."""
    _need(w, "w", _U16)
    dev = w.device
    count = int(count)
    _need(idx, "idx", (torch.int32, torch.uint32), dev, min_numel=count)
    _need(val, "val", _U16, dev, min_numel=count)
    with torch.cuda.device(dev):
        if checked:
            st = lib().pulse_apply_checked(_ptr(w), w.numel(), _ptr(idx), _ptr(val), count, _stream(dev))
        else:
            st = lib().pulse_apply(_ptr(w), _ptr(idx), _ptr(val), count, _stream(dev))
    _raise(st, "pulse_apply")
    return w


def xor_mask(master: torch.Tensor, prev: torch.Tensor, mask_out: Optional[torch.Tensor] = None):
    """pulse_xor_mask: returns the mask; refreshes ``prev`` in place."""
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    _need(prev, "prev", _U16, dev, n)
    if mask_out is None:
        mask_out = torch.empty(n, dtype=torch.int16, device=dev)
    _need(mask_out, "mask_out", _U16, dev, n)
    with torch.cuda.device(dev):
        st = lib().pulse_xor_mask(_ptr(master), _ptr(prev), n, _ptr(mask_out), _stream(dev))
    _raise(st, "pulse_xor_mask")
    return mask_out


def xor_apply(w: torch.Tensor, mask: torch.Tensor):
    """pulse_xor_apply: w ^= mask in place."""
    _need(w, "w", _U16)
    _need(mask, "mask", _U16, w.device, w.numel())
    with torch.cuda.device(w.device):
        st = lib().pulse_xor_apply(_ptr(w), _ptr(mask), w.numel(), _stream(w.device))
    _raise(st, "pulse_xor_apply")
    return w


def get_error(device: Optional[torch.device] = None) -> int:
    """pulse_get_error on torch's current stream: syncs it, returns and clears the code."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        return int(lib().pulse_get_error(_stream(dev)))


def debug_encode_orphan_tile(master, prev, idx_out, val_out, count_out, wait_limit_ns: int) -> int:
    """Test hook for the look-back watchdog (see include/pulse.h). Returns the status."""
    dev = master.device
    with torch.cuda.device(dev):
        return int(lib().pulse_debug_encode_orphan_tile(
            _ptr(master), _ptr(prev), master.numel(), _ptr(idx_out), _ptr(val_out),
            _ptr(count_out), int(wait_limit_ns), _stream(dev)))


# ------------------------------------------------------------- multi-tensor

class TensorSlot:
    """Buffers of one model tensor for a Plan (any field may be None)."""

    def __init__(self, n: int, master=None, prev=None, w=None, idx=None, val=None, mask=None):
        self.n = int(n)
        self.master, self.prev, self.w = master, prev, w
        self.idx, self.val, self.mask = idx, val, mask


class PreparedChain:
    """A chain of patch versions checked and marshalled for one Plan."""

    def __init__(self, plan, refs, nversions: int, keep, counts):
        self.plan, self.refs, self.nversions = plan, refs, int(nversions)
        self._keep = keep  # the patch tensors stay alive with the references
        self.counts = counts  # counts[v][t], clamped to each tensor's size


class PreparedCompose:
    """A chain and its output segments marshalled for Plan.compose_chain."""

    def __init__(self, chain: PreparedChain, outs, arr):
        self.chain, self.outs, self.arr = chain, outs, arr


class Plan:
    """pulse_plan: tile tables of a fixed tensor list, built once, replayed per step."""

    def __init__(self, slots: Sequence[TensorSlot], device: Optional[torch.device] = None):
        if len(slots) == 0:
            raise ValueError("a plan needs at least one tensor")
        self.slots = list(slots)  # keeps the buffers alive while the plan exists
        dev = device
        arr = (PulseTensor * len(slots))()
        for i, s in enumerate(slots):
            for name, t in (("master", s.master), ("prev", s.prev), ("w", s.w), ("idx", s.idx),
                            ("val", s.val), ("mask", s.mask)):
                if t is None:
                    continue
                if dev is None:
                    dev = t.device
                # patch segments need room for n entries where encode writes
                # them; an apply-only segment needs room for the counts applied
                room = s.n if s.master is not None else None
                if name == "master":
                    _need(t, name, (torch.float32,), dev, s.n)
                elif name == "idx":
                    _need(t, name, (torch.int32, torch.uint32), dev, min_numel=room)
                elif name == "val":
                    _need(t, name, _U16, dev, min_numel=room)
                else:
                    _need(t, name, _U16, dev, s.n)
            arr[i] = PulseTensor(_ptr(s.master), _ptr(s.prev), _ptr(s.w), s.n, _ptr(s.idx),
                                 _ptr(s.val), _ptr(s.mask))
        if dev is None:
            raise ValueError("a plan needs at least one device buffer")
        self.device = dev
        self.ntensors = len(slots)
        self._room = [min(s.idx.numel(), s.val.numel()) if s.idx is not None and s.val is not None
                      else 0 for s in slots]
        handle = ctypes.c_void_p()
        with torch.cuda.device(dev):
            st = lib().pulse_plan_create(arr, len(slots), ctypes.byref(handle))
        _raise(st, "pulse_plan_create")
        self._h = handle

    @property
    def num_tiles(self) -> int:
        return int(lib().pulse_plan_num_tiles(self._h))

    def encode(self, counts_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        if counts_out is None:
            counts_out = torch.empty(self.ntensors, dtype=torch.int64, device=self.device)
        _need(counts_out, "counts_out", (torch.int64, torch.uint64), self.device, min_numel=self.ntensors)
        with torch.cuda.device(self.device):
            st = lib().pulse_encode_multi(self._h, _ptr(counts_out), _stream(self.device))
        _raise(st, "pulse_encode_multi")
        return counts_out

    def apply(self, counts):
        """counts: a device int64 tensor (no host round trip) or host integers."""
        with torch.cuda.device(self.device):
            if isinstance(counts, torch.Tensor) and counts.is_cuda:
                _need(counts, "counts", (torch.int64, torch.uint64), self.device, min_numel=self.ntensors)
                if any(r < s.n for r, s in zip(self._room, self.slots)):
                    raise ValueError("device counts need patch segments with room for n entries")
                st = lib().pulse_apply_multi_device(self._h, _ptr(counts), _stream(self.device))
            else:
                vals = [int(c) for c in counts]
                # the library reads min(count, n) entries (a larger count is
                # clamped and reported as PULSE_ERR_INDEX)
                for t, (c, r) in enumerate(zip(vals, self._room)):
                    if min(c, self.slots[t].n) > r:
                        raise ValueError(f"tensor {t}: count {c} exceeds its patch segment ({r})")
                host = (ctypes.c_uint64 * self.ntensors)(*vals)
                st = lib().pulse_apply_multi(self._h, host, _stream(self.device))
        _raise(st, "pulse_apply_multi")

    def prepare_chain(self, patches) -> "PreparedChain":
        """Check and marshal a chain once: patches[v][t] = (idx, val, count)
        of tensor t in the v-th version to apply (oldest first); counts are
        host integers. The result can be passed to apply_chain any number of
        times while the patch buffers stay alive."""
        nv = len(patches)
        if nv < 1:
            raise ValueError("a chain needs at least one version")
        arr = (PulsePatchRef * (nv * self.ntensors))()
        keep = []
        for v, row in enumerate(patches):
            if len(row) != self.ntensors:
                raise ValueError(f"version {v}: {len(row)} segments for {self.ntensors} tensors")
            for t, (idx, val, count) in enumerate(row):
                c = int(count)
                use = min(c, self.slots[t].n)
                if use > 0:
                    _need(idx, "idx", (torch.int32, torch.uint32), self.device, min_numel=use)
                    _need(val, "val", _U16, self.device, min_numel=use)
                    keep.append((idx, val))
                arr[v * self.ntensors + t] = PulsePatchRef(_ptr(idx) if c > 0 else None,
                                                           _ptr(val) if c > 0 else None, c)
        counts = [[min(int(c), s.n) for (_, _, c), s in zip(row, self.slots)] for row in patches]
        return PreparedChain(self, arr, nv, keep, counts)

    def apply_chain(self, patches):
        """pulse_apply_chain_multi: bring w forward by every version of the
        chain (a PreparedChain, or the nested list prepare_chain takes) in
        one pass; equals apply() of each version in turn."""
        prep = patches if isinstance(patches, PreparedChain) else self.prepare_chain(patches)
        if prep.plan is not self:
            raise ValueError("the chain was prepared for another plan")
        with torch.cuda.device(self.device):
            st = lib().pulse_apply_chain_multi(self._h, prep.refs, prep.nversions,
                                               _stream(self.device))
        _raise(st, "pulse_apply_chain_multi")

    def prepare_compose(self, patches, outs=None) -> "PreparedCompose":
        """Check and marshal a k-way composition once: the chain (a
        PreparedChain or the nested list prepare_chain takes) and per tensor
        (idx, val) device output buffers with room for min(n, sum of the
        versions' counts) entries (allocated when ``outs`` is None)."""
        prep = patches if isinstance(patches, PreparedChain) else self.prepare_chain(patches)
        if prep.plan is not self:
            raise ValueError("the chain was prepared for another plan")
        if prep.nversions > 16:
            raise ValueError("a composition takes at most 16 versions")
        need = [min(s.n, sum(prep.counts[v][t] for v in range(prep.nversions)))
                for t, s in enumerate(self.slots)]
        if outs is None:
            outs = [(torch.empty(max(r, 1), dtype=torch.int32, device=self.device),
                     torch.empty(max(r, 1), dtype=torch.int16, device=self.device)) for r in need]
        if len(outs) != self.ntensors:
            raise ValueError(f"{len(outs)} output segments for {self.ntensors} tensors")
        arr = (PulsePatchOut * self.ntensors)()
        for t, ((oi, ov), r) in enumerate(zip(outs, need)):
            _need(oi, "idx_out", (torch.int32, torch.uint32), self.device, min_numel=r)
            _need(ov, "val_out", _U16, self.device, min_numel=r)
            arr[t] = PulsePatchOut(_ptr(oi), _ptr(ov), min(oi.numel(), ov.numel()))
        return PreparedCompose(prep, outs, arr)

    def compose_chain(self, patches, outs=None, counts_out: Optional[torch.Tensor] = None):
        """pulse_compose_chain_multi: one composed patch per tensor for a chain
        of 1..16 versions (a PreparedCompose, or what prepare_compose takes).
        Returns (outs, counts): per tensor (idx, val) buffers whose first
        counts[t] entries are the composed segment (counts: device int64)."""
        pc = patches if isinstance(patches, PreparedCompose) else self.prepare_compose(patches, outs)
        if pc.chain.plan is not self:
            raise ValueError("the composition was prepared for another plan")
        if counts_out is None:
            counts_out = torch.empty(self.ntensors, dtype=torch.int64, device=self.device)
        _need(counts_out, "counts_out", (torch.int64, torch.uint64), self.device,
              min_numel=self.ntensors)
        with torch.cuda.device(self.device):
            st = lib().pulse_compose_chain_multi(self._h, pc.chain.refs, pc.chain.nversions, pc.arr,
                                                 _ptr(counts_out), _stream(self.device))
        _raise(st, "pulse_compose_chain_multi")
        return pc.outs, counts_out

    def xor_mask(self):
        with torch.cuda.device(self.device):
            st = lib().pulse_xor_mask_multi(self._h, _stream(self.device))
        _raise(st, "pulse_xor_mask_multi")

    def xor_apply(self):
        with torch.cuda.device(self.device):
            st = lib().pulse_xor_apply_multi(self._h, _stream(self.device))
        _raise(st, "pulse_xor_apply_multi")

    def get_error(self) -> int:
        with torch.cuda.device(self.device):
            return int(lib().pulse_plan_get_error(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            with torch.cuda.device(self.device):
                lib().pulse_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


# ------------------------------------------------------------ MXFP8 view

def mx_quantize(master: torch.Tensor, codes_out: Optional[torch.Tensor] = None,
                scales_out: Optional[torch.Tensor] = None, fmt: int = MX_E4M3):
    """pulse_mx_quantize_fmt: returns the MX view of format ``fmt`` (codes
    uint8[mx_code_bytes(n, fmt)], scales uint8[ceil(n/32)])."""
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    ncb = mx_code_bytes(n, fmt)
    if codes_out is None:
        codes_out = torch.empty(ncb, dtype=torch.uint8, device=dev)
    if scales_out is None:
        scales_out = torch.empty(mx_blocks(n), dtype=torch.uint8, device=dev)
    _need(codes_out, "codes_out", _U8, dev, ncb)
    _need(scales_out, "scales_out", _U8, dev, mx_blocks(n))
    with torch.cuda.device(dev):
        st = lib().pulse_mx_quantize_fmt(fmt, _ptr(master), n, _ptr(codes_out), _ptr(scales_out),
                                         _stream(dev))
    _raise(st, "pulse_mx_quantize_fmt")
    return codes_out, scales_out


def mx_encode(master: torch.Tensor, prev_codes: torch.Tensor, prev_scales: torch.Tensor,
              idx_out=None, val_out=None, sidx_out=None, sval_out=None, counts_out=None,
              fmt: int = MX_E4M3):
    """pulse_mx_encode_fmt: returns (idx, val, sidx, sval, counts); refreshes
    the previous view in place. ``counts`` is a 2-element device int64 tensor
    {changed code bytes, changed scales}; each segment is the first count
    entries of its buffers."""
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    nb = mx_blocks(n)
    ncb = mx_code_bytes(n, fmt)
    _need(prev_codes, "prev_codes", _U8, dev, ncb)
    _need(prev_scales, "prev_scales", _U8, dev, nb)
    if idx_out is None:
        idx_out = torch.empty(max(ncb, 1), dtype=torch.int32, device=dev)
    if val_out is None:
        val_out = torch.empty(max(ncb, 1), dtype=torch.uint8, device=dev)
    if sidx_out is None:
        sidx_out = torch.empty(max(nb, 1), dtype=torch.int32, device=dev)
    if sval_out is None:
        sval_out = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    if counts_out is None:
        counts_out = torch.empty(2, dtype=torch.int64, device=dev)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=ncb)
    _need(val_out, "val_out", _U8, dev, min_numel=ncb)
    _need(sidx_out, "sidx_out", (torch.int32, torch.uint32), dev, min_numel=nb)
    _need(sval_out, "sval_out", _U8, dev, min_numel=nb)
    _need(counts_out, "counts_out", (torch.int64, torch.uint64), dev, min_numel=2)
    with torch.cuda.device(dev):
        st = lib().pulse_mx_encode_fmt(fmt, _ptr(master), _ptr(prev_codes), _ptr(prev_scales), n,
                                       _ptr(idx_out), _ptr(val_out), _ptr(sidx_out), _ptr(sval_out),
                                       _ptr(counts_out), _stream(dev))
    _raise(st, "pulse_mx_encode_fmt")
    return idx_out, val_out, sidx_out, sval_out, counts_out


def mx_apply(codes: torch.Tensor, scales: torch.Tensor, idx, val, count: int, sidx, sval,
             scount: int, fmt: int = MX_E4M3, n: Optional[int] = None):
    """pulse_mx_apply_fmt: codes[idx[j]] = val[j] (j < count), scales[sidx[j]] = sval[j]
    (j < scount), on a view of ``n`` elements (default: every code byte full)."""
    _need(codes, "codes", _U8)
    dev = codes.device
    if n is None:
        n = codes.numel() * (1 if fmt == MX_E4M3 else 2)
    n = int(n)
    _need(codes, "codes", _U8, dev, mx_code_bytes(n, fmt))
    _need(scales, "scales", _U8, dev, mx_scale_count(n, fmt))
    count, scount = int(count), int(scount)
    _need(idx, "idx", (torch.int32, torch.uint32), dev, min_numel=count)
    _need(val, "val", _U8, dev, min_numel=count)
    _need(sidx, "sidx", (torch.int32, torch.uint32), dev, min_numel=scount)
    _need(sval, "sval", _U8, dev, min_numel=scount)
    with torch.cuda.device(dev):
        st = lib().pulse_mx_apply_fmt(fmt, _ptr(codes), _ptr(scales), n, _ptr(idx), _ptr(val), count,
                                      _ptr(sidx), _ptr(sval), scount, _stream(dev))
    _raise(st, "pulse_mx_apply_fmt")


def nvfp4_quantize(master: torch.Tensor):
    """pulse_nvfp4_quantize: the NVFP4 view (codes uint8[ceil(n/2)], block
    scales uint8[ceil(n/16)], tensor scale: a 1-element device float32)."""
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    codes = torch.empty(max(mx_code_bytes(n, MX_NVFP4), 1), dtype=torch.uint8, device=dev)
    scales = torch.empty(max(mx_scale_count(n, MX_NVFP4), 1), dtype=torch.uint8, device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().pulse_nvfp4_quantize(_ptr(master), n, _ptr(codes), _ptr(scales), _ptr(ts),
                                        _stream(dev))
    _raise(st, "pulse_nvfp4_quantize")
    return codes[:mx_code_bytes(n, MX_NVFP4)], scales[:mx_scale_count(n, MX_NVFP4)], ts


def nvfp4_encode(master: torch.Tensor, prev_codes: torch.Tensor, prev_scales: torch.Tensor,
                 idx_out=None, val_out=None, sidx_out=None, sval_out=None, counts_out=None,
                 tscale_out=None):
    """pulse_nvfp4_encode: returns (idx, val, sidx, sval, counts, tscale);
    refreshes the previous codes and block scales in place."""
    _need(master, "master", (torch.float32,))
    dev = master.device
    n = master.numel()
    nb, ncb = mx_scale_count(n, MX_NVFP4), mx_code_bytes(n, MX_NVFP4)
    _need(prev_codes, "prev_codes", _U8, dev, ncb)
    _need(prev_scales, "prev_scales", _U8, dev, nb)
    if idx_out is None:
        idx_out = torch.empty(max(ncb, 1), dtype=torch.int32, device=dev)
    if val_out is None:
        val_out = torch.empty(max(ncb, 1), dtype=torch.uint8, device=dev)
    if sidx_out is None:
        sidx_out = torch.empty(max(nb, 1), dtype=torch.int32, device=dev)
    if sval_out is None:
        sval_out = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    if counts_out is None:
        counts_out = torch.empty(2, dtype=torch.int64, device=dev)
    if tscale_out is None:
        tscale_out = torch.empty(1, dtype=torch.float32, device=dev)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=ncb)
    _need(val_out, "val_out", _U8, dev, min_numel=ncb)
    _need(sidx_out, "sidx_out", (torch.int32, torch.uint32), dev, min_numel=nb)
    _need(sval_out, "sval_out", _U8, dev, min_numel=nb)
    _need(counts_out, "counts_out", (torch.int64, torch.uint64), dev, min_numel=2)
    _need(tscale_out, "tscale_out", (torch.float32,), dev, min_numel=1)
    with torch.cuda.device(dev):
        st = lib().pulse_nvfp4_encode(_ptr(master), _ptr(prev_codes), _ptr(prev_scales), n,
                                      _ptr(idx_out), _ptr(val_out), _ptr(sidx_out), _ptr(sval_out),
                                      _ptr(counts_out), _ptr(tscale_out), _stream(dev))
    _raise(st, "pulse_nvfp4_encode")
    return idx_out, val_out, sidx_out, sval_out, counts_out, tscale_out


class MxTensorSlot:
    """Buffers of one model tensor for an MxPlan (any field may be None)."""

    def __init__(self, n: int, master=None, prev_codes=None, prev_scales=None, codes=None,
                 scales=None, idx=None, val=None, sidx=None, sval=None):
        self.n = int(n)
        self.master, self.prev_codes, self.prev_scales = master, prev_codes, prev_scales
        self.codes, self.scales = codes, scales
        self.idx, self.val, self.sidx, self.sval = idx, val, sidx, sval


class MxPlan:
    """pulse_mx_plan: the MX view (format ``fmt``) of a fixed tensor list, one
    launch per step.

    Counts are 2 x ntensors int64 in list order: {codes_0, scales_0, codes_1, ...}."""

    def __init__(self, slots: Sequence[MxTensorSlot], device: Optional[torch.device] = None,
                 fmt: int = MX_E4M3):
        if len(slots) == 0:
            raise ValueError("a plan needs at least one tensor")
        self.slots = list(slots)
        self.fmt = fmt
        dev = device
        arr = (PulseMxTensor * len(slots))()
        for i, s in enumerate(slots):
            nb = mx_scale_count(s.n, fmt)
            ncb = mx_code_bytes(s.n, fmt)
            checks = (("master", s.master, (torch.float32,), s.n, None),
                      ("prev_codes", s.prev_codes, _U8, ncb, None),
                      ("prev_scales", s.prev_scales, _U8, nb, None),
                      ("codes", s.codes, _U8, ncb, None),
                      ("scales", s.scales, _U8, nb, None),
                      ("idx", s.idx, (torch.int32, torch.uint32), None, ncb),
                      ("val", s.val, _U8, None, ncb),
                      ("sidx", s.sidx, (torch.int32, torch.uint32), None, nb),
                      ("sval", s.sval, _U8, None, nb))
            for name, t, dtypes, numel, min_numel in checks:
                if t is None:
                    continue
                if dev is None:
                    dev = t.device
                _need(t, name, dtypes, dev, numel, min_numel)
            arr[i] = PulseMxTensor(_ptr(s.master), _ptr(s.prev_codes), _ptr(s.prev_scales),
                                   _ptr(s.codes), _ptr(s.scales), s.n, _ptr(s.idx), _ptr(s.val),
                                   _ptr(s.sidx), _ptr(s.sval))
        if dev is None:
            raise ValueError("a plan needs at least one device buffer")
        self.device = dev
        self.ntensors = len(slots)
        handle = ctypes.c_void_p()
        with torch.cuda.device(dev):
            st = lib().pulse_mx_plan_create_fmt(arr, len(slots), fmt, ctypes.byref(handle))
        _raise(st, "pulse_mx_plan_create_fmt")
        self._h = handle

    def encode(self, counts_out: Optional[torch.Tensor] = None,
               tscales_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Whole-model encode; for an NVFP4 plan the new tensor scales go to
        ``tscales_out`` (device float32, ntensors; kept as ``self.tscales``)."""
        if counts_out is None:
            counts_out = torch.empty(2 * self.ntensors, dtype=torch.int64, device=self.device)
        _need(counts_out, "counts_out", (torch.int64, torch.uint64), self.device,
              min_numel=2 * self.ntensors)
        with torch.cuda.device(self.device):
            if self.fmt == MX_NVFP4:
                if tscales_out is None:
                    tscales_out = torch.empty(self.ntensors, dtype=torch.float32, device=self.device)
                _need(tscales_out, "tscales_out", (torch.float32,), self.device,
                      min_numel=self.ntensors)
                self.tscales = tscales_out
                st = lib().pulse_nvfp4_encode_multi(self._h, _ptr(counts_out), _ptr(tscales_out),
                                                    _stream(self.device))
            else:
                st = lib().pulse_mx_encode_multi(self._h, _ptr(counts_out), _stream(self.device))
        _raise(st, "pulse_mx_encode_multi")
        return counts_out

    def apply(self, counts):
        """counts: a device int64 tensor (no host round trip) or 2 x ntensors host integers."""
        with torch.cuda.device(self.device):
            if isinstance(counts, torch.Tensor) and counts.is_cuda:
                _need(counts, "counts", (torch.int64, torch.uint64), self.device,
                      min_numel=2 * self.ntensors)
                st = lib().pulse_mx_apply_multi_device(self._h, _ptr(counts), _stream(self.device))
            else:
                vals = [int(c) for c in counts]
                if len(vals) != 2 * self.ntensors:
                    raise ValueError(f"expected {2 * self.ntensors} counts, got {len(vals)}")
                host = (ctypes.c_uint64 * len(vals))(*vals)
                st = lib().pulse_mx_apply_multi(self._h, host, _stream(self.device))
        _raise(st, "pulse_mx_apply_multi")

    def get_error(self) -> int:
        with torch.cuda.device(self.device):
            return int(lib().pulse_mx_plan_get_error(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            with torch.cuda.device(self.device):
                lib().pulse_mx_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


# ------------------------------------------------------- patch composition

def _value_kind(t: torch.Tensor) -> int:
    if t.dtype in _U16:
        return 2
    if t.dtype in _U8:
        return 1
    raise TypeError(f"patch values must be 16-bit or 8-bit, not {t.dtype}")


def compose(idx_a: torch.Tensor, val_a: torch.Tensor, count_a: int,
            idx_b: torch.Tensor, val_b: torch.Tensor, count_b: int,
            idx_out: Optional[torch.Tensor] = None, val_out: Optional[torch.Tensor] = None,
            count_out: Optional[torch.Tensor] = None):
    """pulse_compose / pulse_compose_u8: one patch equal to patch A (the first
    count_a entries of idx_a/val_a) followed by patch B. Returns (idx, val,
    count); the result is the first ``count`` entries (device int64)."""
    _need(idx_a, "idx_a", (torch.int32, torch.uint32))
    dev = idx_a.device
    count_a, count_b = int(count_a), int(count_b)
    vb = _value_kind(val_a)
    if _value_kind(val_b) != vb:
        raise TypeError("val_a and val_b differ in width")
    _need(idx_a, "idx_a", (torch.int32, torch.uint32), dev, min_numel=count_a)
    _need(val_a, "val_a", (val_a.dtype,), dev, min_numel=count_a)
    _need(idx_b, "idx_b", (torch.int32, torch.uint32), dev, min_numel=count_b)
    _need(val_b, "val_b", (val_b.dtype,), dev, min_numel=count_b)
    cap = max(count_a + count_b, 1)
    if idx_out is None:
        idx_out = torch.empty(cap, dtype=torch.int32, device=dev)
    if val_out is None:
        val_out = torch.empty(cap, dtype=val_a.dtype, device=dev)
    if count_out is None:
        count_out = torch.empty(1, dtype=torch.int64, device=dev)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=count_a + count_b)
    _need(val_out, "val_out", _U16 if vb == 2 else _U8, dev, min_numel=count_a + count_b)
    _need(count_out, "count_out", (torch.int64, torch.uint64), dev, min_numel=1)
    fn = lib().pulse_compose if vb == 2 else lib().pulse_compose_u8
    with torch.cuda.device(dev):
        st = fn(_ptr(idx_a), _ptr(val_a), count_a, _ptr(idx_b), _ptr(val_b), count_b,
                _ptr(idx_out), _ptr(val_out), _ptr(count_out), _stream(dev))
    _raise(st, "pulse_compose")
    return idx_out, val_out, count_out


def compose_multi(segments, counts_out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pulse_compose_multi. ``segments``: a list of (idx_a, val_a, count_a,
    idx_b, val_b, count_b, idx_out, val_out) with host counts; all values of
    one width. Returns counts_out (device int64, one per segment)."""
    if not segments:
        raise ValueError("no segments")
    dev = segments[0][0].device
    vb = _value_kind(segments[0][1])
    arr = (PulseComposeSegment * len(segments))()
    for i, (ia, va, ka, ib, vbv, kb, io, vo) in enumerate(segments):
        ka, kb = int(ka), int(kb)
        for name, t in (("val_a", va), ("val_b", vbv), ("val_out", vo)):
            if _value_kind(t) != vb:
                raise TypeError(f"segment {i}: {name} differs in width")
        _need(ia, "idx_a", (torch.int32, torch.uint32), dev, min_numel=ka)
        _need(va, "val_a", (va.dtype,), dev, min_numel=ka)
        _need(ib, "idx_b", (torch.int32, torch.uint32), dev, min_numel=kb)
        _need(vbv, "val_b", (vbv.dtype,), dev, min_numel=kb)
        _need(io, "idx_out", (torch.int32, torch.uint32), dev, min_numel=ka + kb)
        _need(vo, "val_out", (vo.dtype,), dev, min_numel=ka + kb)
        arr[i] = PulseComposeSegment(_ptr(ia), _ptr(va), ka, _ptr(ib), _ptr(vbv), kb,
                                     _ptr(io), _ptr(vo))
    if counts_out is None:
        counts_out = torch.empty(len(segments), dtype=torch.int64, device=dev)
    _need(counts_out, "counts_out", (torch.int64, torch.uint64), dev, min_numel=len(segments))
    with torch.cuda.device(dev):
        st = lib().pulse_compose_multi(arr, len(segments), vb, _ptr(counts_out), _stream(dev))
    _raise(st, "pulse_compose_multi")
    return counts_out


# ------------------------------------------------------------- PULSELoCo

def loco_gate(global_w: torch.Tensor, local_w: torch.Tensor, err: torch.Tensor,
              idx_out: Optional[torch.Tensor] = None, val_out: Optional[torch.Tensor] = None,
              count_out: Optional[torch.Tensor] = None):
    """pulse_loco_gate: returns (idx, val, count) of the entries sent; updates
    ``err`` (the FP32 error-feedback buffer) in place."""
    _need(global_w, "global_w", (torch.float32,))
    dev = global_w.device
    n = global_w.numel()
    _need(local_w, "local_w", (torch.float32,), dev, n)
    _need(err, "err", (torch.float32,), dev, n)
    if idx_out is None:
        idx_out = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
    if val_out is None:
        val_out = torch.empty(max(n, 1), dtype=torch.float32, device=dev)
    if count_out is None:
        count_out = torch.empty(1, dtype=torch.int64, device=dev)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=n)
    _need(val_out, "val_out", (torch.float32,), dev, min_numel=n)
    _need(count_out, "count_out", (torch.int64, torch.uint64), dev, min_numel=1)
    with torch.cuda.device(dev):
        st = lib().pulse_loco_gate(_ptr(global_w), _ptr(local_w), _ptr(err), n, _ptr(idx_out),
                                   _ptr(val_out), _ptr(count_out), _stream(dev))
    _raise(st, "pulse_loco_gate")
    return idx_out, val_out, count_out


def loco_accumulate(acc: torch.Tensor, idx: torch.Tensor, val: torch.Tensor, count: int):
    """pulse_loco_accumulate: acc[idx[j]] += val[j] for j < count (FP32)."""
    _need(acc, "acc", (torch.float32,))
    dev = acc.device
    count = int(count)
    _need(idx, "idx", (torch.int32, torch.uint32), dev, min_numel=count)
    _need(val, "val", (torch.float32,), dev, min_numel=count)
    with torch.cuda.device(dev):
        st = lib().pulse_loco_accumulate(_ptr(acc), acc.numel(), _ptr(idx), _ptr(val), count,
                                         _stream(dev))
    _raise(st, "pulse_loco_accumulate")
    return acc


class LocoTensorSlot:
    """Buffers of one model tensor for a LocoPlan (any field may be None)."""

    def __init__(self, n: int, global_w=None, local_w=None, err=None, idx=None, val=None, acc=None):
        self.n = int(n)
        self.global_w, self.local_w, self.err = global_w, local_w, err
        self.idx, self.val, self.acc = idx, val, acc


class LocoPlan:
    """pulse_loco_plan: the gate / accumulation of a whole model, one launch each."""

    def __init__(self, slots: Sequence[LocoTensorSlot], device: Optional[torch.device] = None):
        if len(slots) == 0:
            raise ValueError("a plan needs at least one tensor")
        self.slots = list(slots)
        dev = device
        arr = (PulseLocoTensor * len(slots))()
        for i, s in enumerate(slots):
            for name, t, dtypes, numel, room in (
                    ("global_w", s.global_w, (torch.float32,), s.n, None),
                    ("local_w", s.local_w, (torch.float32,), s.n, None),
                    ("err", s.err, (torch.float32,), s.n, None),
                    ("idx", s.idx, (torch.int32, torch.uint32), None, s.n),
                    ("val", s.val, (torch.float32,), None, s.n),
                    ("acc", s.acc, (torch.float32,), s.n, None)):
                if t is None:
                    continue
                if dev is None:
                    dev = t.device
                _need(t, name, dtypes, dev, numel, room)
            arr[i] = PulseLocoTensor(_ptr(s.global_w), _ptr(s.local_w), _ptr(s.err), s.n,
                                     _ptr(s.idx), _ptr(s.val), _ptr(s.acc))
        if dev is None:
            raise ValueError("a plan needs at least one device buffer")
        self.device = dev
        self.ntensors = len(slots)
        handle = ctypes.c_void_p()
        with torch.cuda.device(dev):
            st = lib().pulse_loco_plan_create(arr, len(slots), ctypes.byref(handle))
        _raise(st, "pulse_loco_plan_create")
        self._h = handle

    def gate(self, counts_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        if counts_out is None:
            counts_out = torch.empty(self.ntensors, dtype=torch.int64, device=self.device)
        _need(counts_out, "counts_out", (torch.int64, torch.uint64), self.device, min_numel=self.ntensors)
        with torch.cuda.device(self.device):
            st = lib().pulse_loco_gate_multi(self._h, _ptr(counts_out), _stream(self.device))
        _raise(st, "pulse_loco_gate_multi")
        return counts_out

    def accumulate(self, counts: torch.Tensor):
        _need(counts, "counts", (torch.int64, torch.uint64), self.device, min_numel=self.ntensors)
        with torch.cuda.device(self.device):
            st = lib().pulse_loco_accumulate_multi(self._h, _ptr(counts), _stream(self.device))
        _raise(st, "pulse_loco_accumulate_multi")

    def get_error(self) -> int:
        with torch.cuda.device(self.device):
            return int(lib().pulse_loco_plan_get_error(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            with torch.cuda.device(self.device):
                lib().pulse_loco_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


# ------------------------------------------------------------ index packing

PACK_BLOCK = 128
PACK_CHUNK = 4096


def pack_sizes(count: int):
    """Elements of (firsts, widths, chunk_off, payload) that a packed segment of
    ``count`` indices needs."""
    nb = (count + PACK_BLOCK - 1) // PACK_BLOCK
    nc = (count + PACK_CHUNK - 1) // PACK_CHUNK
    return max(nb, 1), max(nb, 1), max(nc, 1), max(512 * nb, 16)


def pack_indices(idx: torch.Tensor, count: int, alloc=None):
    """pulse_pack_indices on the first ``count`` entries of ``idx``. Returns
    (firsts, widths, chunk_off, payload, payload_bytes); the packed payload is
    the first ``payload_bytes`` bytes (device int64 tensor) of ``payload``.
    ``alloc(numel, dtype, device)`` makes the output buffers (default
    torch.empty)."""
    _need(idx, "idx", (torch.int32, torch.uint32))
    dev = idx.device
    count = int(count)
    _need(idx, "idx", (torch.int32, torch.uint32), dev, min_numel=count)
    alloc = alloc or (lambda numel, dtype, device: torch.empty(numel, dtype=dtype, device=device))
    nf, nw, nc, npay = pack_sizes(count)
    firsts = alloc(nf, torch.int32, dev)
    widths = alloc(nw, torch.uint8, dev)
    chunk_off = alloc(nc, torch.int64, dev)
    payload = alloc(npay, torch.uint8, dev)
    payload_bytes = alloc(1, torch.int64, dev)
    with torch.cuda.device(dev):
        st = lib().pulse_pack_indices(_ptr(idx), count, _ptr(firsts), _ptr(widths), _ptr(chunk_off),
                                      _ptr(payload), _ptr(payload_bytes), _stream(dev))
    _raise(st, "pulse_pack_indices")
    return firsts, widths, chunk_off, payload, payload_bytes


def unpack_indices(firsts: torch.Tensor, widths: torch.Tensor, chunk_off: torch.Tensor,
                   payload: torch.Tensor, count: int, idx_out: Optional[torch.Tensor] = None):
    """pulse_unpack_indices: the ``count`` indices of a packed segment."""
    dev = firsts.device
    count = int(count)
    nb = (count + PACK_BLOCK - 1) // PACK_BLOCK
    nc = (count + PACK_CHUNK - 1) // PACK_CHUNK
    _need(firsts, "firsts", (torch.int32, torch.uint32), dev, min_numel=nb)
    _need(widths, "widths", _U8, dev, min_numel=nb)
    _need(chunk_off, "chunk_off", (torch.int64, torch.uint64), dev, min_numel=nc)
    _need(payload, "payload", _U8, dev)
    if idx_out is None:
        idx_out = torch.empty(max(count, 1), dtype=torch.int32, device=dev)
    _need(idx_out, "idx_out", (torch.int32, torch.uint32), dev, min_numel=count)
    with torch.cuda.device(dev):
        st = lib().pulse_unpack_indices(_ptr(firsts), _ptr(widths), _ptr(chunk_off), _ptr(payload),
                                        count, _ptr(idx_out), _stream(dev))
    _raise(st, "pulse_unpack_indices")
    return idx_out


class PackJob:
    """pulse_pack_indices_multi / pulse_unpack_indices_multi over a fixed list
    of index segments: the output buffers and both segment tables are built
    once; pack() and unpack() are one launch each for the whole list.

    segments: list of (idx tensor, count) with strictly ascending indices.
    After pack(): packed[s] = (firsts, widths, chunk_off, payload) of segment
    s, payload_bytes[s] (device int64) its payload size. unpack() rebuilds
    every segment into unpacked[s] (first count entries)."""

    def __init__(self, segments, alloc=None):
        """``alloc(numel, dtype, device)`` makes the output buffers (default
        torch.empty)."""
        alloc = alloc or (lambda numel, dtype, device: torch.empty(numel, dtype=dtype, device=device))
        if len(segments) == 0:
            raise ValueError("a pack job needs at least one segment")
        dev = None
        self.counts, self.packed, self.unpacked, keep = [], [], [], []
        n = len(segments)
        self._pack_arr = (PulsePackSegment * n)()
        self._unpack_arr = (PulsePackSegment * n)()
        for i, (idx, count) in enumerate(segments):
            count = int(count)
            if dev is None:
                dev = idx.device
            _need(idx, "idx", (torch.int32, torch.uint32), dev, min_numel=count)
            nf, nw, nc, npay = pack_sizes(count)
            firsts = alloc(nf, torch.int32, dev)
            widths = alloc(nw, torch.uint8, dev)
            chunk_off = alloc(nc, torch.int64, dev)
            payload = alloc(npay, torch.uint8, dev)
            out = alloc(max(count, 1), torch.int32, dev)
            self.counts.append(count)
            self.packed.append((firsts, widths, chunk_off, payload))
            self.unpacked.append(out)
            keep.append(idx)
            self._pack_arr[i] = PulsePackSegment(_ptr(idx), count, _ptr(firsts), _ptr(widths),
                                                 _ptr(chunk_off), _ptr(payload))
            self._unpack_arr[i] = PulsePackSegment(_ptr(out), count, _ptr(firsts), _ptr(widths),
                                                   _ptr(chunk_off), _ptr(payload))
        self.device = dev
        self.nsegs = n
        self._keep = keep
        self.payload_bytes = torch.zeros(n, dtype=torch.int64, device=dev)

    def pack(self) -> torch.Tensor:
        with torch.cuda.device(self.device):
            st = lib().pulse_pack_indices_multi(self._pack_arr, self.nsegs, _ptr(self.payload_bytes),
                                                _stream(self.device))
        _raise(st, "pulse_pack_indices_multi")
        return self.payload_bytes

    def unpack(self):
        with torch.cuda.device(self.device):
            st = lib().pulse_unpack_indices_multi(self._unpack_arr, self.nsegs, _stream(self.device))
        _raise(st, "pulse_unpack_indices_multi")
        return self.unpacked
