"""Helpers shared by the tests: device<->numpy moves of bit patterns and
oracle-side expectations. Bit patterns travel as int16/int32 tensors on the
device and as uint16/uint32 numpy arrays on the host."""
from __future__ import annotations

import re
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pulse.h")


def header_functions(path: str = HEADER):
    """Names of every function declared in the public header."""
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pulse_[a-z0-9_]+)\s*\(", text)))


def dev_f32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def dev_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(device)


def dev_u32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(device)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def host_u32(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def patch_of(idx_t: torch.Tensor, val_t: torch.Tensor, count_t) -> tuple:
    k = int(count_t.item()) if isinstance(count_t, torch.Tensor) else int(count_t)
    return host_u32(idx_t[:k]), host_u16(val_t[:k]), k


# ------------------------------------------------------------- guard zones
# compute-sanitizer is not available where the GPU tests run, so every output
# buffer a kernel writes is allocated with a guard zone on both sides, filled
# with a fixed byte, and the zones are checked after the call: a write past
# either end of a buffer fails the test.
GUARD_BYTES = 4096
GUARD_FILL = 0xA5


class Guarded:
    """``numel`` elements of ``dtype`` on ``device`` between two guard zones of
    GUARD_BYTES bytes. ``t`` is the usable view; it starts GUARD_BYTES after the
    allocation, so it keeps the alignment of a fresh allocation. ``init``
    (a tensor or numpy array) fills ``t``; otherwise ``t`` holds the fill byte."""

    def __init__(self, numel: int, dtype, device="cuda", init=None):
        es = torch.empty(0, dtype=dtype).element_size()
        self.g = GUARD_BYTES // es
        self.numel = int(numel)
        self.raw = torch.empty(self.numel + 2 * self.g, dtype=dtype, device=device)
        self.raw.view(torch.uint8).fill_(GUARD_FILL)
        self.t = self.raw[self.g:self.g + self.numel]
        if init is not None:
            src = init if isinstance(init, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(init))
            self.t.copy_(src.view(dtype) if src.dtype.itemsize == es else src.to(dtype))

    def intact(self) -> bool:
        b = self.raw.view(torch.uint8)
        gb = self.g * self.raw.element_size()
        return bool((b[:gb] == GUARD_FILL).all()) and bool((b[b.numel() - gb:] == GUARD_FILL).all())

    def check(self, name: str = "buffer"):
        assert self.intact(), f"{name}: a write landed in a guard zone (out of bounds)"


def guarded_u16(a: np.ndarray, device="cuda") -> Guarded:
    """Guarded int16 device copy of a uint16 array (BF16 bit patterns)."""
    return Guarded(a.size, torch.int16, device,
                   init=torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)))


def guarded_u8(a: np.ndarray, device="cuda") -> Guarded:
    return Guarded(a.size, torch.uint8, device,
                   init=torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)))


def check_all(**bufs):
    for name, b in bufs.items():
        b.check(name)
