"""Plain CPU forward pass of a dense Llama-3 / Qwen3-style decoder (NumPy).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may call this module; the library never does, and this module
imports nothing from the library.  It is written for a reader to check by eye:
no tiling, no fusion, no reordering beyond the definitions below.

What it computes
----------------
The MegaOps paper ("MegaOps: A Kernel Overlapping Framework with PyTorch-like
Modularity and Megakernel Performance", Abstract) evaluates dense Llama3 and
Qwen3 models, decode and prefill.  Tile-level dependencies (same Abstract) and
the on-device interpreter with barriers held as tensors ("Lecture 112:
Production Megakernels for Real-World Inference", Key takeaways and Technical
details) only change the *order* in which independent work runs, so the result
the GPU path must reproduce is the plain forward pass of that model family,
written out here.

Readings where the pages say nothing (each is a parameter of the workload, not
code shared with the GPU path):
  * RoPE pairs element i with i + d/2 ("rotate half"); angle p * theta^(-2i/d),
    computed in float64; no frequency scaling.
  * GQA: query head h reads kv head h // (n_q / n_kv).
  * Softmax over scores q.k / sqrt(d), max-subtracted, no mask in decode beyond
    the cached length, causal in prefill.
  * RMSNorm: x / sqrt(mean(x^2) + eps) * w.  Qwen3-style per-head q/k RMSNorm
    (same eps) is applied before RoPE.
  * FFN: SwiGLU, down(silu(gate(h)) * up(h)), silu(z) = z / (1 + exp(-z)).
  * Decode: sequence b holds positions[b] cached tokens; the new token sits at
    index positions[b] and attends over positions[b] + 1 keys.  Cached slots are
    read as post-RoPE keys.
  * Prefill: one sequence at positions 0..S-1, causal; returns the last token's
    logits (or all of them) and the K/V it produced.

Precision: every step runs in `dtype` (float32 by default, float64 for the
pins); weights and the cache arrive as bf16 bit patterns and are widened
exactly.  The KV cache stores bf16, so the keys and values a step produces
enter attention rounded to bf16 (nearest, ties to even), exactly as a later
step reads them back from the cache; kv_bf16=False keeps them in `dtype`.

Parity: pinned (closed forms, invariants, library special cases and brute
force on tiny inputs) by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# element-wise pieces
# ---------------------------------------------------------------------------

def widen_bf16(a) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exactly; float input passes through."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


def _f(a, dtype):
    return np.asarray(widen_bf16(a), dtype=dtype)


def round_bf16(x, dtype=np.float32) -> np.ndarray:
    """Nearest bf16 value of x (ties to the even significand), returned in dtype.

    bf16 keeps 8 significant bits over float32's exponent range: writing
    x = m * 2^e with 0.5 <= |m| < 1, the representable neighbours are multiples
    of 2^(e - 8); below the smallest normal (2^-126) the spacing stays 2^-133.
    np.rint rounds halves to even, which is IEEE round-to-nearest-even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    return (np.rint(x / q) * q).astype(dtype)


def rmsnorm(x, w, eps, dtype=np.float32) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    x = _f(x, dtype)
    w = _f(w, dtype)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + dtype(eps)) * w


def rope_angles(pos, d, theta) -> np.ndarray:
    """Angles p * theta^(-2i/d) for i < d/2, float64; shape pos.shape + (d/2,)."""
    i = np.arange(d // 2, dtype=np.float64)
    inv_freq = np.float64(theta) ** (-2.0 * i / d)
    return np.multiply.outer(np.asarray(pos, dtype=np.float64), inv_freq)


def rope_rotate_half(u, pos, theta, dtype=np.float32) -> np.ndarray:
    """Rotate pairs (u_i, u_{i+d/2}) by angle p*theta_i.

    `pos` must broadcast against u.shape[:-1] (e.g. a scalar, or positions with
    trailing singleton axes for the head axis).
    """
    u = _f(u, dtype)
    d = u.shape[-1]
    a = rope_angles(pos, d, theta)
    c = np.cos(a).astype(dtype)
    s = np.sin(a).astype(dtype)
    u1 = u[..., : d // 2]
    u2 = u[..., d // 2:]
    return np.concatenate([u1 * c - u2 * s, u2 * c + u1 * s], axis=-1)


def silu(z, dtype=np.float32) -> np.ndarray:
    z = _f(z, dtype)
    return z / (dtype(1) + np.exp(-z))


def linear(W, x, dtype=np.float32, row_chunk: int = 16384) -> np.ndarray:
    """y = x @ W^T for W [out, in] (bf16 bits or float), x [..., in]."""
    x = _f(x, dtype)
    W = np.asarray(W)
    out = np.empty(x.shape[:-1] + (W.shape[0],), dtype=dtype)
    for r0 in range(0, W.shape[0], row_chunk):
        r1 = min(W.shape[0], r0 + row_chunk)
        out[..., r0:r1] = x @ _f(W[r0:r1], dtype).T
    return out


def gqa_attention(q, K, V, dtype=np.float32) -> np.ndarray:
    """Grouped-query attention of one token.

    q [n_q, d]; K, V [n_kv, n, d] (all n keys visible) -> o [n_q, d].
    """
    q = _f(q, dtype)
    K = _f(K, dtype)
    V = _f(V, dtype)
    n_q, d = q.shape
    n_kv = K.shape[0]
    group = n_q // n_kv
    scale = dtype(1.0 / np.sqrt(d))
    o = np.empty((n_q, d), dtype=dtype)
    for h in range(n_q):
        g = h // group
        s = (K[g] @ q[h]) * scale
        s = s - s.max()
        p = np.exp(s)
        p = p / p.sum()
        o[h] = p @ V[g]
    return o


def causal_gqa_attention(q, K, V, dtype=np.float32) -> np.ndarray:
    """Causal grouped-query attention over one sequence.

    q [S, n_q, d]; K, V [n_kv, S, d] -> o [S, n_q, d]; query i sees keys 0..i.
    """
    q = _f(q, dtype)
    K = _f(K, dtype)
    V = _f(V, dtype)
    S, n_q, d = q.shape
    n_kv = K.shape[0]
    group = n_q // n_kv
    scale = dtype(1.0 / np.sqrt(d))
    future = np.triu(np.ones((S, S), dtype=bool), k=1)
    o = np.empty((S, n_q, d), dtype=dtype)
    for h in range(n_q):
        g = h // group
        s = (q[:, h, :] @ K[g].T) * scale
        s[future] = -np.inf
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        o[:, h, :] = p @ V[g]
    return o


# ---------------------------------------------------------------------------
# whole model
# ---------------------------------------------------------------------------

def _cfg(cfg, key):
    return cfg[key] if isinstance(cfg, dict) else getattr(cfg, key)


def _lm_weight(cfg, w):
    return w["embed"] if _cfg(cfg, "tied_embeddings") else w["lm_head"]


def decode_step(cfg, w, tokens, positions, kv, dtype=np.float32, kv_bf16: bool = True):
    """One decode step for B sequences.

    cfg: model shape (attributes or dict keys n_layers, hidden, n_q_heads,
         n_kv_heads, head_dim, ffn, vocab, rms_eps, rope_theta, qk_norm,
         tied_embeddings).
    w:   name -> weight (bf16 bits as uint16, or float), [out, in].
    tokens, positions: [B] ints; sequence b sits in cache slot b.
    kv:  [n_layers][2][max_batch][n_kv][max_ctx][d] (bf16 bits or float); only
         positions < positions[b] of slot b are read.
    kv_bf16: the new token's key and value enter attention as the bf16 cache
         stores them (round_bf16); False keeps them in dtype.
    Returns (logits [B, vocab], k_new [L, B, n_kv, d], v_new [L, B, n_kv, d]).
    """
    L = _cfg(cfg, "n_layers")
    nq, nkv, d = _cfg(cfg, "n_q_heads"), _cfg(cfg, "n_kv_heads"), _cfg(cfg, "head_dim")
    eps, theta = _cfg(cfg, "rms_eps"), _cfg(cfg, "rope_theta")
    qk_norm = _cfg(cfg, "qk_norm")
    tokens = np.asarray(tokens, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    B = tokens.shape[0]

    x = _f(np.asarray(w["embed"])[tokens], dtype)               # [B, H]
    k_new = np.zeros((L, B, nkv, d), dtype=dtype)
    v_new = np.zeros((L, B, nkv, d), dtype=dtype)
    for l in range(L):
        p = f"layers.{l}."
        h = rmsnorm(x, w[p + "attn_norm"], eps, dtype)
        q = linear(w[p + "wq"], h, dtype)
        k = linear(w[p + "wk"], h, dtype)
        v = linear(w[p + "wv"], h, dtype)
        o = np.empty((B, nq * d), dtype=dtype)
        for b in range(B):
            pos = int(positions[b])
            qb = q[b].reshape(nq, d)
            kb = k[b].reshape(nkv, d)
            vb = v[b].reshape(nkv, d)
            if qk_norm:
                qb = rmsnorm(qb, w[p + "q_norm"], eps, dtype)
                kb = rmsnorm(kb, w[p + "k_norm"], eps, dtype)
            qb = rope_rotate_half(qb, pos, theta, dtype)
            kb = rope_rotate_half(kb, pos, theta, dtype)
            if kv_bf16:
                kb, vb = round_bf16(kb, dtype), round_bf16(vb, dtype)
            Kb = np.concatenate([_f(kv[l, 0, b, :, :pos, :], dtype), kb[:, None, :]], axis=1)
            Vb = np.concatenate([_f(kv[l, 1, b, :, :pos, :], dtype), vb[:, None, :]], axis=1)
            o[b] = gqa_attention(qb, Kb, Vb, dtype).reshape(-1)
            k_new[l, b] = kb
            v_new[l, b] = vb
        x = x + linear(w[p + "wo"], o, dtype)
        h2 = rmsnorm(x, w[p + "ffn_norm"], eps, dtype)
        a = silu(linear(w[p + "w_gate"], h2, dtype), dtype) * linear(w[p + "w_up"], h2, dtype)
        x = x + linear(w[p + "w_down"], a, dtype)
    hf = rmsnorm(x, w["final_norm"], eps, dtype)
    logits = linear(_lm_weight(cfg, w), hf, dtype)
    return logits, k_new, v_new


def prefill(cfg, w, tokens, dtype=np.float32, all_logits: bool = False,
            kv_bf16: bool = True):
    """Causal forward of one prompt at positions 0..S-1.

    Returns (logits, K, V): logits [vocab] of the last token (or [S, vocab] when
    all_logits), K and V [L, n_kv, S, d] (post-RoPE keys, values).  With
    kv_bf16 the keys and values are rounded to bf16 (round_bf16) before the
    attention reads them, as a bf16 KV cache holds them.
    """
    L = _cfg(cfg, "n_layers")
    nq, nkv, d = _cfg(cfg, "n_q_heads"), _cfg(cfg, "n_kv_heads"), _cfg(cfg, "head_dim")
    eps, theta = _cfg(cfg, "rms_eps"), _cfg(cfg, "rope_theta")
    qk_norm = _cfg(cfg, "qk_norm")
    tokens = np.asarray(tokens, dtype=np.int64)
    S = tokens.shape[0]
    pos = np.arange(S)

    x = _f(np.asarray(w["embed"])[tokens], dtype)               # [S, H]
    K_all = np.zeros((L, nkv, S, d), dtype=dtype)
    V_all = np.zeros((L, nkv, S, d), dtype=dtype)
    for l in range(L):
        p = f"layers.{l}."
        h = rmsnorm(x, w[p + "attn_norm"], eps, dtype)
        q = linear(w[p + "wq"], h, dtype).reshape(S, nq, d)
        k = linear(w[p + "wk"], h, dtype).reshape(S, nkv, d)
        v = linear(w[p + "wv"], h, dtype).reshape(S, nkv, d)
        if qk_norm:
            q = rmsnorm(q, w[p + "q_norm"], eps, dtype)
            k = rmsnorm(k, w[p + "k_norm"], eps, dtype)
        q = rope_rotate_half(q, pos[:, None], theta, dtype)
        k = rope_rotate_half(k, pos[:, None], theta, dtype)
        if kv_bf16:
            k, v = round_bf16(k, dtype), round_bf16(v, dtype)
        Kl = np.ascontiguousarray(k.transpose(1, 0, 2))         # [n_kv, S, d]
        Vl = np.ascontiguousarray(v.transpose(1, 0, 2))
        K_all[l] = Kl
        V_all[l] = Vl
        o = causal_gqa_attention(q, Kl, Vl, dtype).reshape(S, nq * d)
        x = x + linear(w[p + "wo"], o, dtype)
        h2 = rmsnorm(x, w[p + "ffn_norm"], eps, dtype)
        a = silu(linear(w[p + "w_gate"], h2, dtype), dtype) * linear(w[p + "w_up"], h2, dtype)
        x = x + linear(w[p + "w_down"], a, dtype)
    rows = x if all_logits else x[-1:]
    hf = rmsnorm(rows, w["final_norm"], eps, dtype)
    logits = linear(_lm_weight(cfg, w), hf, dtype)
    return (logits if all_logits else logits[0]), K_all, V_all
