"""Seeded synthetic inputs: model shapes, weights, KV caches, token ids, positions.

This module only draws random numbers and names shapes.  It holds none of the
forward pass's arithmetic, so the CPU oracle and the CUDA path can both be fed
from it without sharing any computation.

Workloads are the dense Llama-3 / Qwen3 decoder shapes that the MegaOps paper
evaluates on ("MegaOps: A Kernel Overlapping Framework with PyTorch-like
Modularity and Megakernel Performance", Abstract: dense Llama3 and Qwen3
models).  No checkpoint is used: every weight is drawn from a seeded normal.

Distributions:
  * embedding / projection / LM-head matrices: N(0, 0.02), rounded to bf16;
  * RMSNorm gains (attention, FFN, final, per-head q/k): 1 + N(0, 0.02) in bf16,
    so normalised activations keep unit scale while the gain multiply is still
    exercised;
  * KV cache contents: N(0, 1) in bf16 (read as post-RoPE keys and values);
  * token ids: uniform over the vocabulary; ragged contexts: uniform integers.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class ModelCfg:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float
    rope_theta: float
    qk_norm: bool = False
    tied_embeddings: bool = False

    def replace(self, **kw) -> "ModelCfg":
        return dataclasses.replace(self, **kw)


# Workload shapes.  Names say what they are; sizes are the public model shapes.
TOY_1L = ModelCfg(n_layers=1, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                  ffn=688, vocab=1024, rms_eps=1e-5, rope_theta=1e4)
LLAMA32_1B = ModelCfg(n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
                      ffn=8192, vocab=128256, rms_eps=1e-5, rope_theta=5e5,
                      tied_embeddings=True)
LLAMA3_8B = ModelCfg(n_layers=32, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                     ffn=14336, vocab=128256, rms_eps=1e-5, rope_theta=5e5)
QWEN3_8B = ModelCfg(n_layers=36, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                    ffn=12288, vocab=151936, rms_eps=1e-6, rope_theta=1e6, qk_norm=True)

# Seeds of the input recipe.
SEED_WEIGHTS = 0
SEED_KV = 1
SEED_TOKENS = 2
SEED_CONTEXTS = 3


def _sub_seed(base: int, name: str) -> int:
    return (base * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, mean: float, std: float, seed: int, device) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    g = _gen(seed, device)
    # draw in row chunks so that an fp32 temporary never exceeds ~256 MB
    rows = shape[0] if len(shape) > 1 else 1
    per_row = 1
    for s in shape[1:]:
        per_row *= s
    chunk = max(1, (1 << 26) // max(per_row, 1))
    flat = out.view(rows, per_row) if len(shape) > 1 else out.view(1, -1)
    for r0 in range(0, flat.shape[0], chunk):
        r1 = min(flat.shape[0], r0 + chunk)
        t = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                        dtype=torch.float32)
        t.mul_(std).add_(mean)
        flat[r0:r1].copy_(t)
    return out


def weight_shapes(cfg: ModelCfg) -> Dict[str, tuple]:
    H, d, F = cfg.hidden, cfg.head_dim, cfg.ffn
    shapes = {"embed": (cfg.vocab, H), "final_norm": (H,)}
    if not cfg.tied_embeddings:
        shapes["lm_head"] = (cfg.vocab, H)
    for l in range(cfg.n_layers):
        p = f"layers.{l}."
        shapes[p + "attn_norm"] = (H,)
        shapes[p + "wq"] = (cfg.n_q_heads * d, H)
        shapes[p + "wk"] = (cfg.n_kv_heads * d, H)
        shapes[p + "wv"] = (cfg.n_kv_heads * d, H)
        shapes[p + "wo"] = (H, cfg.n_q_heads * d)
        if cfg.qk_norm:
            shapes[p + "q_norm"] = (d,)
            shapes[p + "k_norm"] = (d,)
        shapes[p + "ffn_norm"] = (H,)
        shapes[p + "w_gate"] = (F, H)
        shapes[p + "w_up"] = (F, H)
        shapes[p + "w_down"] = (H, F)
    return shapes


def is_norm(name: str) -> bool:
    return name.endswith("norm")


def make_weights(cfg: ModelCfg, seed: int = SEED_WEIGHTS, device="cpu",
                 std: float = 0.02) -> Dict[str, torch.Tensor]:
    """All weights as bf16 tensors on `device`, [out, in] row-major."""
    out = {}
    for name, shape in weight_shapes(cfg).items():
        if is_norm(name):
            out[name] = _normal_bf16(shape, 1.0, std, _sub_seed(seed, name), device)
        else:
            out[name] = _normal_bf16(shape, 0.0, std, _sub_seed(seed, name), device)
    return out


def kv_cache_shape(cfg: ModelCfg, max_batch: int, max_ctx: int) -> tuple:
    """[layer][k|v][sequence][kv head][position][head_dim], bf16."""
    return (cfg.n_layers, 2, max_batch, cfg.n_kv_heads, max_ctx, cfg.head_dim)


def make_kv_cache(cfg: ModelCfg, max_batch: int, max_ctx: int, seed: int = SEED_KV,
                  device="cpu") -> torch.Tensor:
    shape = kv_cache_shape(cfg, max_batch, max_ctx)
    flat = (cfg.n_layers * 2 * max_batch * cfg.n_kv_heads, max_ctx * cfg.head_dim)
    return _normal_bf16(flat, 0.0, 1.0, seed, device).view(shape)


def make_tokens(n: int, vocab: int, seed: int = SEED_TOKENS) -> torch.Tensor:
    g = _gen(seed, "cpu")
    return torch.randint(0, vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def make_contexts(n: int, lo: int, hi: int, seed: int = SEED_CONTEXTS) -> torch.Tensor:
    """Ragged cached lengths, uniform integers in [lo, hi] inclusive."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's raw bits as a numpy uint16 array (CPU copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def weights_as_bits(w: Dict[str, torch.Tensor]) -> Dict[str, "object"]:
    return {k: bf16_bits(v) for k, v in w.items()}


class LazyBits:
    """Mapping name -> uint16 bits, copying each device tensor to the host on use."""

    def __init__(self, w: Dict[str, torch.Tensor]):
        self._w = w

    def __getitem__(self, name):
        return bf16_bits(self._w[name])

    def __contains__(self, name):
        return name in self._w

    def get(self, name, default: Optional[object] = None):
        return self[name] if name in self._w else default
