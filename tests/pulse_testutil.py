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
