"""Seeded synthetic inputs for the weight-delta encode/apply path.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds none of the method's arithmetic (no rounding, no
comparison, no compaction): it only names tensor sets and draws random
numbers. The one cast it performs, the initial BF16 view ``prev0``, is
torch's own ``.to(torch.bfloat16)``; any uint16 array is a valid ``prev``, so
parity never depends on how it was produced.

Tensor sets (shapes follow the model families the PULSE technical summary,
arXiv 2602.03839, evaluates on, section "Significato e Affermazioni":
Qwen / Llama families):

* ``single``      one flat tensor (2^20 elements, or 2^28 for the density sweep)
* ``llama_layer`` one Llama-style decoder layer, 9 tensors, 218,112,000 params
* ``llama3_8b``   a Llama-3-8B-shaped model, 291 tensors, 8,030,261,248 params
* ``qwen2_5_1_5b`` a Qwen2.5-1.5B-shaped model with q/k/v biases and tied
  embedding, 338 tensors, 1,543,714,304 params

Distributions: weights and biases ~ N(0, 0.02); RMSNorm vectors ~ 1 + N(0, 0.01);
update ``master = w0 + eta * z`` with z ~ N(0, 1) i.i.d. FP32 and eta = 3e-6
(the RL learning rate named in the PULSE technical summary, section
"Osservazione Centrale: Sparsità Visibile al Calcolo").
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence

import numpy as np

ETA_DEFAULT = 3e-6
ETA_SWEEP = (1e-7, 3e-7, 1e-6, 3e-6, 1e-5, 3e-5, 1e-4)
WEIGHT_STD = 0.02
NORM_STD = 0.01


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    kind: str  # "weight" | "norm" | "bias"

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def _llama_layer(prefix: str, hidden: int, q_heads: int, kv_heads: int,
                 head_dim: int, mlp: int, qkv_bias: bool) -> List[TensorSpec]:
    q = q_heads * head_dim
    kv = kv_heads * head_dim
    out = [TensorSpec(f"{prefix}self_attn.q_proj.weight", (q, hidden), "weight")]
    if qkv_bias:
        out.append(TensorSpec(f"{prefix}self_attn.q_proj.bias", (q,), "bias"))
    out.append(TensorSpec(f"{prefix}self_attn.k_proj.weight", (kv, hidden), "weight"))
    if qkv_bias:
        out.append(TensorSpec(f"{prefix}self_attn.k_proj.bias", (kv,), "bias"))
    out.append(TensorSpec(f"{prefix}self_attn.v_proj.weight", (kv, hidden), "weight"))
    if qkv_bias:
        out.append(TensorSpec(f"{prefix}self_attn.v_proj.bias", (kv,), "bias"))
    out += [
        TensorSpec(f"{prefix}self_attn.o_proj.weight", (hidden, q), "weight"),
        TensorSpec(f"{prefix}mlp.gate_proj.weight", (mlp, hidden), "weight"),
        TensorSpec(f"{prefix}mlp.up_proj.weight", (mlp, hidden), "weight"),
        TensorSpec(f"{prefix}mlp.down_proj.weight", (hidden, mlp), "weight"),
        TensorSpec(f"{prefix}input_layernorm.weight", (hidden,), "norm"),
        TensorSpec(f"{prefix}post_attention_layernorm.weight", (hidden,), "norm"),
    ]
    return out


def llama_layer() -> List[TensorSpec]:
    """One Llama-3-8B decoder layer: hidden 4096, 32 q / 8 kv heads x 128, MLP 14336."""
    return _llama_layer("model.layers.0.", 4096, 32, 8, 128, 14336, False)


def llama3_8b() -> List[TensorSpec]:
    """Llama-3-8B-shaped set: embed, 32 layers, final norm, untied lm_head (vocab 128256)."""
    out = [TensorSpec("model.embed_tokens.weight", (128256, 4096), "weight")]
    for i in range(32):
        out += _llama_layer(f"model.layers.{i}.", 4096, 32, 8, 128, 14336, False)
    out.append(TensorSpec("model.norm.weight", (4096,), "norm"))
    out.append(TensorSpec("lm_head.weight", (128256, 4096), "weight"))
    return out


def qwen2_5_1_5b() -> List[TensorSpec]:
    """Qwen2.5-1.5B-shaped set: hidden 1536, 12 q / 2 kv heads x 128, MLP 8960,
    vocab 151936, q/k/v biases, tied embedding (no separate lm_head)."""
    out = [TensorSpec("model.embed_tokens.weight", (151936, 1536), "weight")]
    for i in range(28):
        out += _llama_layer(f"model.layers.{i}.", 1536, 12, 2, 128, 8960, True)
    out.append(TensorSpec("model.norm.weight", (1536,), "norm"))
    return out


def single(n: int) -> List[TensorSpec]:
    return [TensorSpec("flat", (n,), "weight")]


# The five workloads. Sizes and seeds are fixed here so tests and bench agree.
CONFIGS = {
    1: dict(name="single_2^20", specs=lambda: single(1 << 20), seed=0, eta=ETA_DEFAULT),
    2: dict(name="llama_layer_218M", specs=llama_layer, seed=1, eta=ETA_DEFAULT),
    3: dict(name="llama3_8b_8.03B", specs=llama3_8b, seed=2, eta=ETA_DEFAULT),
    4: dict(name="flat_2^28_eta_sweep", specs=lambda: single(1 << 28), seed=3, eta=None),
    5: dict(name="qwen2.5_1.5b_20step_chain", specs=qwen2_5_1_5b, seed=4, eta=ETA_DEFAULT),
}

CHAIN_STEPS = 20
CHAIN_SEED_BASE = 10000


def sweep_seed(i: int) -> int:
    """Seed of the update draw for the i-th eta of the density sweep."""
    return 3 + 100 * i


def total_params(specs: Sequence[TensorSpec]) -> int:
    return sum(s.numel for s in specs)


# ---------------------------------------------------------------- numpy (CPU)

def np_init(spec: TensorSpec, rng: np.random.Generator) -> np.ndarray:
    """FP32 initial master weights for one tensor (flattened)."""
    z = rng.standard_normal(spec.numel, dtype=np.float32)
    if spec.kind == "norm":
        return (np.float32(1.0) + np.float32(NORM_STD) * z).astype(np.float32)
    return (np.float32(WEIGHT_STD) * z).astype(np.float32)


def np_update(w: np.ndarray, eta: float, rng: np.random.Generator) -> np.ndarray:
    """One Adam-like step of size eta: w + eta * z (FP32)."""
    z = rng.standard_normal(w.size, dtype=np.float32)
    return (w + np.float32(eta) * z).astype(np.float32)


def np_bf16_view_torch(w: np.ndarray) -> np.ndarray:
    """Initial BF16 view as uint16 bit patterns, produced by torch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(w)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def np_pair(n: int, seed: int, eta: float = ETA_DEFAULT, kind: str = "weight"):
    """(master_new f32, prev u16) for one tensor of n elements, drawn on the CPU."""
    rng = np.random.default_rng(seed)
    w0 = np_init(TensorSpec("t", (n,), kind), rng)
    prev = np_bf16_view_torch(w0)
    master = np_update(w0, eta, rng)
    return master, prev


# -------------------------------------------------------------- torch (device)

def torch_generator(device, seed: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def torch_init_(out, spec: TensorSpec, gen):
    """Fill ``out`` (FP32, flat, on device) with the initial master weights."""
    import torch
    torch.randn(out.shape, generator=gen, dtype=torch.float32, device=out.device, out=out)
    if spec.kind == "norm":
        out.mul_(NORM_STD).add_(1.0)
    else:
        out.mul_(WEIGHT_STD)
    return out


def torch_update_(master, eta: float, gen, chunk: int = 1 << 26):
    """master += eta * z, z ~ N(0,1) drawn in chunks to bound scratch memory."""
    import torch
    n = master.numel()
    z = torch.empty(min(chunk, n), dtype=torch.float32, device=master.device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        zz = z[: e - s]
        torch.randn(zz.shape, generator=gen, dtype=torch.float32, device=master.device, out=zz)
        master[s:e].add_(zz, alpha=eta)
    return master


def torch_bf16_view_(prev_u16, master_f32):
    """prev <- torch's BF16 cast of master (bit patterns stored as int16)."""
    import torch
    prev_u16.copy_(master_f32.to(torch.bfloat16).view(torch.int16))
    return prev_u16


def torch_model(specs: Sequence[TensorSpec], seed: int, eta: float, device,
                chunk: int = 1 << 26):
    """Draws one training step on the device for every tensor, in list order.

    Per tensor: w0 (initial master, FP32) then z; returns a list of
    (master = w0 + eta * z, prev0 = torch's BF16 cast of w0) pairs, flat,
    one allocation each (int16 holds the BF16 bit patterns of prev0).
    """
    import torch
    gen = torch_generator(device, seed)
    out = []
    for spec in specs:
        m = torch.empty(spec.numel, dtype=torch.float32, device=device)
        torch_init_(m, spec, gen)
        p = torch.empty(spec.numel, dtype=torch.int16, device=device)
        torch_bf16_view_(p, m)
        torch_update_(m, eta, gen, chunk)
        out.append((m, p))
    return out


def torch_model_states(specs: Sequence[TensorSpec], seed: int, eta: float, device,
                       chunk: int = 1 << 26):
    """The same draws as ``torch_model`` (per tensor: w0, then z), returned as
    (w0, master = w0 + eta * z) pairs of FP32 tensors, for views other than
    BF16 that are built from w0 by the code under test."""
    import torch
    gen = torch_generator(device, seed)
    out = []
    for spec in specs:
        w0 = torch.empty(spec.numel, dtype=torch.float32, device=device)
        torch_init_(w0, spec, gen)
        m = w0.clone()
        torch_update_(m, eta, gen, chunk)
        out.append((w0, m))
    return out


def torch_step_(masters, step: int, eta: float = ETA_DEFAULT, chunk: int = 1 << 26):
    """One more Adam-sized step of a chain: master += eta * z, z drawn from
    seed CHAIN_SEED_BASE + step, tensors in list order."""
    if not masters:
        return
    gen = torch_generator(masters[0].device, CHAIN_SEED_BASE + step)
    for m in masters:
        torch_update_(m, eta, gen, chunk)
