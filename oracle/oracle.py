"""numpy wrapper around the plain-C oracle (``pulse_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).

All arrays are numpy: FP32 master weights as ``float32``, BF16 weights,
patch values and masks as ``uint16`` bit patterns, patch indices as
``uint32``. Functions that update ``prev`` or ``w`` do so in place, like the
CUDA entry points they check.

Multi-tensor forms run the single-tensor definition over the tensors in list
order; each tensor has its own patch segment with tensor-local indices (the
whole-model, single-launch form described in the humansand.ai summary,
section "Pipeline'i GPU'lara tasimak", computes exactly this).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("pulse_oracle.c", "mx_oracle.c", "mxfp4_oracle.c",
                                          "nvfp4_oracle.c", "compose_oracle.c", "loco_oracle.c",
                                          "pack_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library with gcc -O2 (no CUDA)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(s) for s in _SRCS))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        # -ffp-contract=off: every FP32 operation rounds on its own (no FMA)
        subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror",
                        "-ffp-contract=off", "-shared", "-fPIC", "-o", tmp, *_SRCS, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            U64 = ctypes.c_uint64
            lib.oracle_bf16_rne.argtypes = [ctypes.c_uint32]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_bf16_rne_array.argtypes = [P, P, U64]
            lib.oracle_bf16_rne_array.restype = None
            lib.oracle_encode.argtypes = [P, P, U64, P, P]
            lib.oracle_encode.restype = U64
            lib.oracle_count_changed.argtypes = [P, P, U64]
            lib.oracle_count_changed.restype = U64
            lib.oracle_apply.argtypes = [P, P, P, U64]
            lib.oracle_apply.restype = None
            lib.oracle_xor_mask.argtypes = [P, P, U64, P]
            lib.oracle_xor_mask.restype = None
            lib.oracle_xor_apply.argtypes = [P, P, U64]
            lib.oracle_xor_apply.restype = None
            lib.oracle_e4m3_rne.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_rne.restype = ctypes.c_uint8
            lib.oracle_mx_block_scale.argtypes = [P, U64]
            lib.oracle_mx_block_scale.restype = ctypes.c_uint8
            lib.oracle_mxfp8_quantize.argtypes = [P, U64, P, P]
            lib.oracle_mxfp8_quantize.restype = None
            lib.oracle_mxfp8_encode.argtypes = [P, P, P, U64, P, P, P, P, P]
            lib.oracle_mxfp8_encode.restype = None
            lib.oracle_e2m1_rne.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_rne.restype = ctypes.c_uint8
            lib.oracle_mxfp4_block_scale.argtypes = [P, U64]
            lib.oracle_mxfp4_block_scale.restype = ctypes.c_uint8
            lib.oracle_mxfp4_quantize.argtypes = [P, U64, P, P]
            lib.oracle_mxfp4_quantize.restype = None
            lib.oracle_mxfp4_encode.argtypes = [P, P, P, U64, P, P, P, P, P]
            lib.oracle_mxfp4_encode.restype = None
            lib.oracle_nvfp4_tensor_scale.argtypes = [P, U64]
            lib.oracle_nvfp4_tensor_scale.restype = ctypes.c_float
            lib.oracle_nvfp4_quantize.argtypes = [P, U64, P, P]
            lib.oracle_nvfp4_quantize.restype = ctypes.c_float
            lib.oracle_nvfp4_encode.argtypes = [P, P, P, U64, P, P, P, P, P]
            lib.oracle_nvfp4_encode.restype = ctypes.c_float
            lib.oracle_apply_u8.argtypes = [P, P, P, U64]
            lib.oracle_apply_u8.restype = None
            lib.oracle_compose.argtypes = [P, P, U64, P, P, U64, P, P]
            lib.oracle_compose.restype = U64
            lib.oracle_compose_u8.argtypes = [P, P, U64, P, P, U64, P, P]
            lib.oracle_compose_u8.restype = U64
            lib.oracle_loco_gate.argtypes = [P, P, P, U64, P, P]
            lib.oracle_loco_gate.restype = U64
            lib.oracle_loco_accumulate.argtypes = [P, P, P, U64]
            lib.oracle_loco_accumulate.restype = None
            lib.oracle_pack_indices.argtypes = [P, U64, P, P, P, P]
            lib.oracle_pack_indices.restype = U64
            lib.oracle_unpack_indices.argtypes = [P, P, P, P, U64, P]
            lib.oracle_unpack_indices.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _check(a: np.ndarray, dtype, name: str, writable: bool = False):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or a.ndim != 1:
        raise TypeError(f"{name}: expected a 1-D numpy {np.dtype(dtype).name} array")
    if not a.flags.c_contiguous:
        raise TypeError(f"{name}: must be contiguous")
    if writable and not a.flags.writeable:
        raise TypeError(f"{name}: must be writable")


def bf16_rne(bits) -> np.ndarray | int:
    """RNE cast of FP32 bit patterns (uint32 array or int) to BF16 bits."""
    lib = _load()
    if isinstance(bits, (int, np.integer)):
        return int(lib.oracle_bf16_rne(int(bits) & 0xFFFFFFFF))
    a = np.ascontiguousarray(bits, dtype=np.uint32).reshape(-1)
    out = np.empty(a.size, dtype=np.uint16)
    lib.oracle_bf16_rne_array(_ptr(a), _ptr(out), a.size)
    return out


def encode(master: np.ndarray, prev: np.ndarray):
    """Returns (idx[k] uint32, val[k] uint16); refreshes ``prev`` in place."""
    _check(master, np.float32, "master")
    _check(prev, np.uint16, "prev", writable=True)
    if master.size != prev.size:
        raise ValueError("master and prev differ in length")
    n = master.size
    idx = np.empty(max(n, 1), dtype=np.uint32)
    val = np.empty(max(n, 1), dtype=np.uint16)
    k = _load().oracle_encode(_ptr(master), _ptr(prev), n, _ptr(idx), _ptr(val))
    return idx[:k].copy(), val[:k].copy()


def count_changed(master: np.ndarray, prev: np.ndarray) -> int:
    _check(master, np.float32, "master")
    _check(prev, np.uint16, "prev")
    return int(_load().oracle_count_changed(_ptr(master), _ptr(prev), master.size))


def apply(w: np.ndarray, idx: np.ndarray, val: np.ndarray) -> None:
    """w[idx[j]] = val[j] for j in order, in place."""
    _check(w, np.uint16, "w", writable=True)
    _check(idx, np.uint32, "idx")
    _check(val, np.uint16, "val")
    if idx.size != val.size:
        raise ValueError("idx and val differ in length")
    if idx.size and int(idx.max()) >= w.size:
        raise IndexError("patch index out of range")
    _load().oracle_apply(_ptr(w), _ptr(idx), _ptr(val), idx.size)


def xor_mask(master: np.ndarray, prev: np.ndarray) -> np.ndarray:
    """Returns mask = rne(master) ^ prev; refreshes ``prev`` in place."""
    _check(master, np.float32, "master")
    _check(prev, np.uint16, "prev", writable=True)
    if master.size != prev.size:
        raise ValueError("master and prev differ in length")
    mask = np.empty(master.size, dtype=np.uint16)
    _load().oracle_xor_mask(_ptr(master), _ptr(prev), master.size, _ptr(mask))
    return mask


def xor_apply(w: np.ndarray, mask: np.ndarray) -> None:
    """w ^= mask, in place."""
    _check(w, np.uint16, "w", writable=True)
    _check(mask, np.uint16, "mask")
    if w.size != mask.size:
        raise ValueError("w and mask differ in length")
    _load().oracle_xor_apply(_ptr(w), _ptr(mask), w.size)


# ------------------------------------------------------------ multi-tensor

def encode_multi(masters, prevs):
    """List-order encode; returns a list of (idx, val) segments."""
    return [encode(m, p) for m, p in zip(masters, prevs)]


def apply_multi(ws, patches) -> None:
    for w, (idx, val) in zip(ws, patches):
        apply(w, idx, val)


def xor_mask_multi(masters, prevs):
    return [xor_mask(m, p) for m, p in zip(masters, prevs)]


# ------------------------------------------- the same code on many host cores

def _chunks(n: int, parts: int):
    step = -(-n // max(1, parts))
    return [(c0, min(n, c0 + step)) for c0 in range(0, n, max(1, step))]


def encode_chunked(master: np.ndarray, prev: np.ndarray, pool, parts: int):
    """The scalar encode spread over host threads, for timing the oracle on
    every core (not a second definition: it calls the same C loops).

    Count pass: each of ``parts`` contiguous chunks counts its changed
    elements (``oracle_count_changed``). An exclusive scan of those counts
    gives each chunk's first patch slot. Emit pass: each chunk runs
    ``oracle_encode`` on its slice into its slots and shifts the slice-local
    indices by the chunk's start. Concatenated in chunk order the result is
    the single-threaded patch. ``pool`` is a thread pool (ctypes releases the
    interpreter lock during the C calls). Returns (idx, val); refreshes
    ``prev``."""
    _check(master, np.float32, "master")
    _check(prev, np.uint16, "prev", writable=True)
    if master.size != prev.size:
        raise ValueError("master and prev differ in length")
    lib = _load()
    spans = _chunks(master.size, parts)
    counts = list(pool.map(
        lambda s: int(lib.oracle_count_changed(_ptr(master[s[0]:]), _ptr(prev[s[0]:]),
                                               s[1] - s[0])), spans))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    k = int(offs[-1])
    idx = np.empty(max(k, 1), dtype=np.uint32)
    val = np.empty(max(k, 1), dtype=np.uint16)

    def emit(i):
        c0, c1 = spans[i]
        o = int(offs[i])
        got = lib.oracle_encode(_ptr(master[c0:]), _ptr(prev[c0:]), c1 - c0,
                                _ptr(idx[o:]), _ptr(val[o:]))
        if got != counts[i]:
            raise RuntimeError("emit pass disagrees with the count pass")
        idx[o:o + got] += np.uint32(c0)

    list(pool.map(emit, range(len(spans))))
    return idx[:k], val[:k]


def apply_chunked(w: np.ndarray, idx: np.ndarray, val: np.ndarray, pool, parts: int) -> None:
    """``oracle_apply`` over contiguous ranges of the patch on host threads.
    Patch indices are distinct (an encode patch is strictly ascending), so the
    ranges write disjoint elements and the order between them is immaterial."""
    _check(w, np.uint16, "w", writable=True)
    _check(idx, np.uint32, "idx")
    _check(val, np.uint16, "val")
    if idx.size != val.size:
        raise ValueError("idx and val differ in length")
    if idx.size and int(idx.max()) >= w.size:
        raise IndexError("patch index out of range")
    lib = _load()
    list(pool.map(lambda s: lib.oracle_apply(_ptr(w), _ptr(idx[s[0]:]), _ptr(val[s[0]:]),
                                             s[1] - s[0]), _chunks(idx.size, parts)))


def xor_apply_multi(ws, masks) -> None:
    for w, m in zip(ws, masks):
        xor_apply(w, m)


# ------------------------------------------------- MXFP8 serving view

MX_BLOCK = 32


def e4m3_rne(y) -> int:
    """E4M3 code of one finite value y (a Python float), RNE, clamped to 448."""
    return int(_load().oracle_e4m3_rne(float(y)))


def mx_block_scale(block: np.ndarray) -> int:
    """E8M0 scale byte of one block of 1..32 FP32 values."""
    _check(block, np.float32, "block")
    if not 1 <= block.size <= MX_BLOCK:
        raise ValueError("a block holds 1..32 values")
    return int(_load().oracle_mx_block_scale(_ptr(block), block.size))


def mx_blocks(n: int) -> int:
    return (n + MX_BLOCK - 1) // MX_BLOCK


def mxfp8_quantize(master: np.ndarray):
    """Returns the MXFP8 view (codes uint8[n], scales uint8[ceil(n/32)])."""
    _check(master, np.float32, "master")
    n = master.size
    codes = np.empty(n, dtype=np.uint8)
    scales = np.empty(mx_blocks(n), dtype=np.uint8)
    _load().oracle_mxfp8_quantize(_ptr(master), n, _ptr(codes), _ptr(scales))
    return codes, scales


def mxfp8_encode(master: np.ndarray, prev_codes: np.ndarray, prev_scales: np.ndarray):
    """Returns (idx uint32, val uint8, sidx uint32, sval uint8); refreshes
    ``prev_codes`` and ``prev_scales`` in place."""
    _check(master, np.float32, "master")
    _check(prev_codes, np.uint8, "prev_codes", writable=True)
    _check(prev_scales, np.uint8, "prev_scales", writable=True)
    n = master.size
    if prev_codes.size != n or prev_scales.size != mx_blocks(n):
        raise ValueError("view arrays do not match the master's length")
    nb = mx_blocks(n)
    idx = np.empty(max(n, 1), dtype=np.uint32)
    val = np.empty(max(n, 1), dtype=np.uint8)
    sidx = np.empty(max(nb, 1), dtype=np.uint32)
    sval = np.empty(max(nb, 1), dtype=np.uint8)
    counts = np.zeros(2, dtype=np.uint64)
    _load().oracle_mxfp8_encode(_ptr(master), _ptr(prev_codes), _ptr(prev_scales), n,
                                _ptr(idx), _ptr(val), _ptr(sidx), _ptr(sval), _ptr(counts))
    k, ks = int(counts[0]), int(counts[1])
    return idx[:k].copy(), val[:k].copy(), sidx[:ks].copy(), sval[:ks].copy()


def apply_u8(w: np.ndarray, idx: np.ndarray, val: np.ndarray) -> None:
    """w[idx[j]] = val[j] for j in order, in place (one byte segment)."""
    _check(w, np.uint8, "w", writable=True)
    _check(idx, np.uint32, "idx")
    _check(val, np.uint8, "val")
    if idx.size != val.size:
        raise ValueError("idx and val differ in length")
    if idx.size and int(idx.max()) >= w.size:
        raise IndexError("patch index out of range")
    _load().oracle_apply_u8(_ptr(w), _ptr(idx), _ptr(val), idx.size)


def mxfp8_apply(codes: np.ndarray, scales: np.ndarray, patch) -> None:
    """Apply both segments of an MXFP8 patch (idx, val, sidx, sval) in place."""
    idx, val, sidx, sval = patch
    apply_u8(codes, idx, val)
    apply_u8(scales, sidx, sval)


# ------------------------------------------------------------- MXFP4 view

def e2m1_rne(y) -> int:
    """E2M1 code (4 bits, bit 3 = sign) of one finite value y, RNE, clamped to 6."""
    return int(_load().oracle_e2m1_rne(float(y)))


def mxfp4_block_scale(block: np.ndarray) -> int:
    """E8M0 scale byte of one MXFP4 block of 1..32 FP32 values."""
    _check(block, np.float32, "block")
    if not 1 <= block.size <= MX_BLOCK:
        raise ValueError("a block holds 1..32 values")
    return int(_load().oracle_mxfp4_block_scale(_ptr(block), block.size))


def mxfp4_code_bytes(n: int) -> int:
    """Bytes of an n-element MXFP4 code array (two codes per byte)."""
    return (n + 1) // 2


def mxfp4_quantize(master: np.ndarray):
    """Returns the MXFP4 view (codes uint8[ceil(n/2)], element 2j in the low
    nibble of byte j; scales uint8[ceil(n/32)])."""
    _check(master, np.float32, "master")
    n = master.size
    codes = np.empty(mxfp4_code_bytes(n), dtype=np.uint8)
    scales = np.empty(mx_blocks(n), dtype=np.uint8)
    _load().oracle_mxfp4_quantize(_ptr(master), n, _ptr(codes), _ptr(scales))
    return codes, scales


def mxfp4_encode(master: np.ndarray, prev_codes: np.ndarray, prev_scales: np.ndarray):
    """Returns (idx uint32, val uint8, sidx uint32, sval uint8): changed code
    BYTES and changed scales; refreshes ``prev_codes`` and ``prev_scales``."""
    _check(master, np.float32, "master")
    _check(prev_codes, np.uint8, "prev_codes", writable=True)
    _check(prev_scales, np.uint8, "prev_scales", writable=True)
    n = master.size
    if prev_codes.size != mxfp4_code_bytes(n) or prev_scales.size != mx_blocks(n):
        raise ValueError("view arrays do not match the master's length")
    nb, ncb = mx_blocks(n), mxfp4_code_bytes(n)
    idx = np.empty(max(ncb, 1), dtype=np.uint32)
    val = np.empty(max(ncb, 1), dtype=np.uint8)
    sidx = np.empty(max(nb, 1), dtype=np.uint32)
    sval = np.empty(max(nb, 1), dtype=np.uint8)
    counts = np.zeros(2, dtype=np.uint64)
    _load().oracle_mxfp4_encode(_ptr(master), _ptr(prev_codes), _ptr(prev_scales), n,
                                _ptr(idx), _ptr(val), _ptr(sidx), _ptr(sval), _ptr(counts))
    k, ks = int(counts[0]), int(counts[1])
    return idx[:k].copy(), val[:k].copy(), sidx[:ks].copy(), sval[:ks].copy()


def mxfp4_apply(codes: np.ndarray, scales: np.ndarray, patch) -> None:
    """Apply both segments of an MXFP4 patch (byte idx, val, sidx, sval) in place."""
    idx, val, sidx, sval = patch
    apply_u8(codes, idx, val)
    apply_u8(scales, sidx, sval)


# ------------------------------------------------------------- NVFP4 view

NV_BLOCK = 16


def nv_blocks(n: int) -> int:
    return (n + NV_BLOCK - 1) // NV_BLOCK


def nvfp4_tensor_scale(master: np.ndarray) -> float:
    """S = (largest finite magnitude) / 2688, in FP32."""
    _check(master, np.float32, "master")
    return float(np.float32(_load().oracle_nvfp4_tensor_scale(_ptr(master), master.size)))


def nvfp4_quantize(master: np.ndarray):
    """Returns the NVFP4 view: (codes uint8[ceil(n/2)], block scales
    uint8[ceil(n/16)] (E4M3), tensor scale as a numpy float32)."""
    _check(master, np.float32, "master")
    n = master.size
    codes = np.empty(mxfp4_code_bytes(n), dtype=np.uint8)
    scales = np.empty(nv_blocks(n), dtype=np.uint8)
    S = _load().oracle_nvfp4_quantize(_ptr(master), n, _ptr(codes), _ptr(scales))
    return codes, scales, np.float32(S)


def nvfp4_encode(master: np.ndarray, prev_codes: np.ndarray, prev_scales: np.ndarray):
    """Returns (idx, val, sidx, sval, tensor scale): changed code bytes,
    changed block scales and the new tensor scale; refreshes the previous
    view in place."""
    _check(master, np.float32, "master")
    _check(prev_codes, np.uint8, "prev_codes", writable=True)
    _check(prev_scales, np.uint8, "prev_scales", writable=True)
    n = master.size
    if prev_codes.size != mxfp4_code_bytes(n) or prev_scales.size != nv_blocks(n):
        raise ValueError("view arrays do not match the master's length")
    nb, ncb = nv_blocks(n), mxfp4_code_bytes(n)
    idx = np.empty(max(ncb, 1), dtype=np.uint32)
    val = np.empty(max(ncb, 1), dtype=np.uint8)
    sidx = np.empty(max(nb, 1), dtype=np.uint32)
    sval = np.empty(max(nb, 1), dtype=np.uint8)
    counts = np.zeros(2, dtype=np.uint64)
    S = _load().oracle_nvfp4_encode(_ptr(master), _ptr(prev_codes), _ptr(prev_scales), n,
                                    _ptr(idx), _ptr(val), _ptr(sidx), _ptr(sval), _ptr(counts))
    k, ks = int(counts[0]), int(counts[1])
    return idx[:k].copy(), val[:k].copy(), sidx[:ks].copy(), sval[:ks].copy(), np.float32(S)


# ---------------------------------------------------- patch-chain composition

def compose(a, b):
    """One patch equal to patch ``a`` followed by patch ``b`` (each an (idx,
    val) pair with strictly ascending idx): the union of the indices, the
    later value on a shared index. Values uint16 or uint8 (both the same)."""
    ia, va = a
    ib, vb = b
    _check(ia, np.uint32, "idx_a")
    _check(ib, np.uint32, "idx_b")
    if va.dtype != vb.dtype or va.dtype not in (np.uint16, np.uint8):
        raise TypeError("values must both be uint16 or both uint8")
    _check(va, va.dtype, "val_a")
    _check(vb, vb.dtype, "val_b")
    if ia.size != va.size or ib.size != vb.size:
        raise ValueError("idx and val differ in length")
    cap = max(ia.size + ib.size, 1)
    idx = np.empty(cap, dtype=np.uint32)
    val = np.empty(cap, dtype=va.dtype)
    fn = _load().oracle_compose if va.dtype == np.uint16 else _load().oracle_compose_u8
    k = fn(_ptr(ia), _ptr(va), ia.size, _ptr(ib), _ptr(vb), ib.size, _ptr(idx), _ptr(val))
    return idx[:k].copy(), val[:k].copy()


def compose_chain(patches):
    """Left fold of compose over a list of patches (oldest first)."""
    if not patches:
        raise ValueError("empty chain")
    out = patches[0]
    for p in patches[1:]:
        out = compose(out, p)
    return out


# ------------------------------------------------- PULSELoCo gate (sender)

def loco_gate(global_w: np.ndarray, local_w: np.ndarray, err: np.ndarray):
    """Returns (idx uint32, val float32) of the entries that pass the
    visibility gate; updates ``err`` (float32) in place."""
    _check(global_w, np.float32, "global")
    _check(local_w, np.float32, "local")
    _check(err, np.float32, "err", writable=True)
    n = global_w.size
    if local_w.size != n or err.size != n:
        raise ValueError("global, local and err differ in length")
    idx = np.empty(max(n, 1), dtype=np.uint32)
    val = np.empty(max(n, 1), dtype=np.float32)
    k = _load().oracle_loco_gate(_ptr(global_w), _ptr(local_w), _ptr(err), n, _ptr(idx), _ptr(val))
    return idx[:k].copy(), val[:k].copy()


def loco_accumulate(acc: np.ndarray, idx: np.ndarray, val: np.ndarray) -> None:
    """acc[idx[j]] += val[j] in order, FP32, in place."""
    _check(acc, np.float32, "acc", writable=True)
    _check(idx, np.uint32, "idx")
    _check(val, np.float32, "val")
    if idx.size != val.size:
        raise ValueError("idx and val differ in length")
    if idx.size and int(idx.max()) >= acc.size:
        raise IndexError("index out of range")
    _load().oracle_loco_accumulate(_ptr(acc), _ptr(idx), _ptr(val), idx.size)


# ------------------------------------------------------ index packing

PACK_BLOCK = 128
PACK_CHUNK = 4096   # entries per independently decodable chunk (32 blocks)


def pack_indices(idx: np.ndarray):
    """Returns (firsts uint32[B], widths uint8[B], chunk_off uint64[C],
    payload uint8[...]) for strictly ascending uint32 indices."""
    _check(idx, np.uint32, "idx")
    k = idx.size
    nb = (k + PACK_BLOCK - 1) // PACK_BLOCK
    nc = (k + PACK_CHUNK - 1) // PACK_CHUNK
    firsts = np.zeros(max(nb, 1), dtype=np.uint32)
    widths = np.zeros(max(nb, 1), dtype=np.uint8)
    chunk_off = np.zeros(max(nc, 1), dtype=np.uint64)
    payload = np.zeros(max(nb * 512, 1), dtype=np.uint8)
    size = _load().oracle_pack_indices(_ptr(idx), k, _ptr(firsts), _ptr(widths), _ptr(chunk_off),
                                       _ptr(payload))
    return firsts[:nb].copy(), widths[:nb].copy(), chunk_off[:nc].copy(), payload[:size].copy()


def unpack_indices(firsts, widths, chunk_off, payload, k: int) -> np.ndarray:
    _check(firsts, np.uint32, "firsts")
    _check(widths, np.uint8, "widths")
    _check(chunk_off, np.uint64, "chunk_off")
    _check(payload, np.uint8, "payload")
    out = np.empty(max(int(k), 1), dtype=np.uint32)
    pl = payload if payload.size else np.zeros(1, np.uint8)
    _load().oracle_unpack_indices(_ptr(firsts), _ptr(widths), _ptr(chunk_off), _ptr(pl), int(k),
                                  _ptr(out))
    return out[:int(k)].copy()
