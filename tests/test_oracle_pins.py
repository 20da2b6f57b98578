"""Pins for the CPU oracle: closed forms, invariants, library special cases,
brute force on tiny inputs.  Each test is chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign, index or pairing, a transposed operand)
fails at least one of them.  CPU only."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import model as om
from tile_level_overlap_gb300 import synth

F64 = np.float64


def _golden(golden_dir, name):
    rows = []
    with open(f"{golden_dir}/closed_forms.txt") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            n, inp, exp = [s.strip() for s in line.split("|")]
            if n == name:
                rows.append((inp, [float(eval(e, {"math": math})) for e in _split(exp)]))
    assert rows, name
    return rows


def _split(expr):
    # split a comma list at top level (expressions may contain commas in calls)
    out, depth, cur = [], 0, ""
    for ch in expr:
        if ch == "(":
            depth += 1
        elif ch == ")":
            depth -= 1
        if ch == "," and depth == 0:
            out.append(cur)
            cur = ""
        else:
            cur += ch
    out.append(cur)
    return out


# ---------------------------------------------------------------- bf16 widening

def test_widen_bf16_exact():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x3E4D], dtype=np.uint16)
    got = oracle.widen_bf16(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 0.0
    assert np.signbit(got[3]) and np.isinf(got[4])
    t = torch.randn(1000).to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.widen_bf16(synth.bf16_bits(t)), t.float().numpy())


def test_round_bf16_closed_forms():
    r = lambda v: float(oracle.round_bf16(np.float64(v), F64))
    u = 2.0 ** -7                          # bf16 spacing in [1, 2)
    assert r(1.0) == 1.0 and r(0.0) == 0.0 and r(-3.0) == -3.0
    assert r(1 + u / 2) == 1.0             # tie -> even significand (1.0)
    assert r(1 + 3 * u / 2) == 1 + 2 * u   # tie -> even significand (1 + 2u)
    assert r(1 + u / 2 + 2 ** -30) == 1 + u
    assert r(-(1 + u / 2 + 2 ** -30)) == -(1 + u)
    assert r(255.9) == 256.0               # carries into the next binade
    assert r(2.0 ** -130) == 2.0 ** -130   # subnormal range, multiple of 2^-133
    assert r(3 * 2.0 ** -134) == 2 * 2.0 ** -133   # 1.5 quanta -> tie -> even (2)
    assert np.isinf(r(np.inf)) and np.isnan(r(np.nan))


def test_round_bf16_vs_torch_conversion():
    # torch's float32 -> bfloat16 cast is round-to-nearest-even
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.randn(20000, generator=g) * 10.0 ** torch.randint(-30, 30, (20000,), generator=g),
                   torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], dtype=torch.float32)])
    want = x.to(torch.bfloat16).float().numpy()
    got = oracle.round_bf16(x.numpy(), np.float32)
    np.testing.assert_array_equal(got, want)
    assert np.all((got.view(np.uint32) & 0xFFFF) == 0)   # representable in bf16


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    rng = np.random.default_rng(0)
    for c, eps in [(3.0, 0.5), (-0.25, 1e-5), (7.0, 2.0)]:
        x = np.full(16, c)
        w = rng.normal(size=16)
        got = oracle.rmsnorm(x, w, eps, F64)
        np.testing.assert_allclose(got, c / math.sqrt(c * c + eps) * w, rtol=1e-14)


def test_rmsnorm_golden(golden_dir):
    (inp, exp), = _golden(golden_dir, "rmsnorm_eps0_w21")
    x = np.array([float(v) for v in inp.split(",")])
    np.testing.assert_allclose(oracle.rmsnorm(x, np.array([2.0, 1.0]), 0.0, F64), exp, rtol=1e-14)


def test_rmsnorm_scale_invariant_and_vs_torch():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 64))
    w = rng.normal(size=64)
    a = oracle.rmsnorm(x, w, 0.0, F64)
    b = oracle.rmsnorm(3.7 * x, w, 0.0, F64)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 1e-5, F64), ref, rtol=1e-13)


# ---------------------------------------------------------------- RoPE

def test_rope_golden(golden_dir):
    for name, p in [("rope_d4_t100_p1", 1), ("rope_d4_t100_p3", 3)]:
        for inp, exp in _golden(golden_dir, name):
            u = np.array([float(v) for v in inp.split(",")])
            got = oracle.rope_rotate_half(u, p, 100.0, F64)
            np.testing.assert_allclose(got, exp, atol=1e-15)


def test_rope_position_zero_is_identity_and_norm_preserved():
    rng = np.random.default_rng(2)
    u = rng.normal(size=(6, 128))
    np.testing.assert_array_equal(oracle.rope_rotate_half(u, 0, 5e5, F64), u)
    for p in [1, 17, 4095, 123456]:
        r = oracle.rope_rotate_half(u, p, 5e5, F64)
        np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(u, axis=-1),
                                   rtol=1e-13)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=64), rng.normal(size=64)
    def dot(m, n):
        return float(oracle.rope_rotate_half(q, m, 1e4, F64) @ oracle.rope_rotate_half(k, n, 1e4, F64))
    base = dot(10, 3)
    for t in [1, 50, 1000]:
        assert abs(dot(10 + t, 3 + t) - base) < 1e-10
    assert abs(dot(3, 10) - base) > 1e-3   # depends on the sign of m - n


def test_rope_matches_complex_rotation():
    # (u_i + i u_{i+d/2}) * exp(i p theta^(-2i/d)), computed by torch.polar
    rng = np.random.default_rng(4)
    d, theta = 64, 1e6
    u = rng.normal(size=(3, d))
    pos = np.array([0, 5, 777])
    inv = torch.tensor(theta, dtype=torch.float64) ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    ang = torch.from_numpy(pos).double()[:, None] * inv[None, :]
    z = torch.complex(torch.from_numpy(u[:, : d // 2]), torch.from_numpy(u[:, d // 2:]))
    zr = z * torch.polar(torch.ones_like(ang), ang)
    ref = torch.cat([zr.real, zr.imag], dim=-1).numpy()
    got = oracle.rope_rotate_half(u, pos, theta, F64)
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_qknorm_then_rope_golden(golden_dir):
    (inp, exp), = _golden(golden_dir, "qknorm_then_rope_d2_p1")
    x = np.array([float(v) for v in inp.split(",")])
    n = oracle.rmsnorm(x, np.array([2.0, 1.0]), 0.0, F64)
    got = oracle.rope_rotate_half(n, 1, 10.0, F64)
    np.testing.assert_allclose(got, exp, rtol=1e-14)


# ---------------------------------------------------------------- SiLU / SwiGLU

def test_silu_closed_forms_and_torch():
    assert oracle.silu(np.array([0.0]), F64)[0] == 0.0
    np.testing.assert_allclose(oracle.silu(np.array([40.0]), F64), [40.0], rtol=1e-15)
    z = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(oracle.silu(z, F64) - oracle.silu(-z, F64), z, atol=1e-14)
    np.testing.assert_allclose(oracle.silu(z, F64), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14)


def test_swiglu_golden(golden_dir):
    for inp, exp in _golden(golden_dir, "swiglu"):
        g, u = [float(s.split("=")[1]) for s in inp.split(",")]
        got = oracle.silu(np.array([g]), F64)[0] * u
        assert abs(got - exp[0]) < 1e-15


# ---------------------------------------------------------------- linear

def test_linear_vs_triple_loop():
    rng = np.random.default_rng(5)
    W = rng.normal(size=(3, 5))
    x = rng.normal(size=(2, 5))
    ref = np.zeros((2, 3))
    for b in range(2):
        for r in range(3):
            for c in range(5):
                ref[b, r] += W[r, c] * x[b, c]
    np.testing.assert_allclose(oracle.linear(W, x, F64), ref, rtol=1e-14)
    # row chunking does not change the result
    np.testing.assert_allclose(oracle.linear(W, x, F64, row_chunk=2), oracle.linear(W, x, F64),
                               rtol=1e-14)


def test_linear_bf16_bits_widened():
    t = (torch.randn(7, 9) * 0.02).to(torch.bfloat16)
    x = np.random.default_rng(6).normal(size=9)
    np.testing.assert_allclose(oracle.linear(synth.bf16_bits(t), x, F64),
                               t.double().numpy() @ x, rtol=1e-12)


# ---------------------------------------------------------------- attention

def test_attention_one_key_returns_v():
    rng = np.random.default_rng(7)
    q = rng.normal(size=(4, 16))
    K = rng.normal(size=(2, 1, 16))
    V = rng.normal(size=(2, 1, 16))
    o = oracle.gqa_attention(q, K, V, F64)
    np.testing.assert_array_equal(o[:2], np.repeat(V[0], 2, 0))
    np.testing.assert_array_equal(o[2:], np.repeat(V[1], 2, 0))


def test_attention_equal_keys_gives_mean_v():
    rng = np.random.default_rng(8)
    q = rng.normal(size=(2, 8))
    K = np.repeat(rng.normal(size=(1, 1, 8)), 9, axis=1)
    V = rng.normal(size=(1, 9, 8))
    o = oracle.gqa_attention(q, K, V, F64)
    np.testing.assert_allclose(o, np.repeat(V[0].mean(0, keepdims=True), 2, 0), rtol=1e-13)


def test_attention_two_keys_golden(golden_dir):
    (inp, exp), = _golden(golden_dir, "attn_two_keys_d4")
    q = np.array([[2.0, 0, 0, 0]])
    K = np.array([[[1.0, 0, 0, 0], [0, 1.0, 0, 0]]])
    V = np.array([[[1.0, 0, 0, 0], [0, 0, 0, 4.0]]])
    np.testing.assert_allclose(oracle.gqa_attention(q, K, V, F64)[0], exp, rtol=1e-14)


def test_gqa_head_mapping_consecutive_groups():
    n_q, n_kv, n, d = 8, 2, 5, 4
    q = np.random.default_rng(9).normal(size=(n_q, d))
    K = np.random.default_rng(10).normal(size=(n_kv, n, d))
    V = np.stack([np.full((n, d), float(g)) for g in range(n_kv)])
    o = oracle.gqa_attention(q, K, V, F64)
    for h in range(n_q):
        np.testing.assert_allclose(o[h], h // (n_q // n_kv), rtol=1e-14)


def test_attention_vs_torch_sdpa():
    rng = np.random.default_rng(11)
    n_q, n_kv, n, d = 8, 2, 33, 32
    q = rng.normal(size=(n_q, d))
    K = rng.normal(size=(n_kv, n, d))
    V = rng.normal(size=(n_kv, n, d))
    rep = n_q // n_kv
    Kt = torch.from_numpy(K).repeat_interleave(rep, 0)
    Vt = torch.from_numpy(V).repeat_interleave(rep, 0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], Kt, Vt)[:, 0, :].numpy()
    np.testing.assert_allclose(oracle.gqa_attention(q, K, V, F64), ref, rtol=1e-12, atol=1e-13)
    # grouped == multi-head on repeat-interleaved K/V
    np.testing.assert_allclose(oracle.gqa_attention(q, K, V, F64),
                               oracle.gqa_attention(q, Kt.numpy(), Vt.numpy(), F64), rtol=1e-14)


def test_causal_attention_vs_torch_and_rows():
    rng = np.random.default_rng(12)
    S, n_q, n_kv, d = 13, 4, 2, 16
    q = rng.normal(size=(S, n_q, d))
    K = rng.normal(size=(n_kv, S, d))
    V = rng.normal(size=(n_kv, S, d))
    o = om.causal_gqa_attention(q, K, V, F64)
    np.testing.assert_array_equal(o[0], np.repeat(V[:, 0, :], 2, 0))    # row 0 sees key 0 only
    for i in [1, 6, 12]:
        np.testing.assert_allclose(o[i], oracle.gqa_attention(q[i], K[:, : i + 1], V[:, : i + 1], F64),
                                   rtol=1e-12)
    Kt = torch.from_numpy(K).repeat_interleave(2, 0)
    Vt = torch.from_numpy(V).repeat_interleave(2, 0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q).transpose(0, 1), Kt, Vt, is_causal=True)
    np.testing.assert_allclose(o, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- whole model

TINY = synth.ModelCfg(n_layers=2, hidden=32, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=48,
                      vocab=50, rms_eps=1e-5, rope_theta=1e4)


def _w(cfg, seed=0):
    return synth.weights_as_bits(synth.make_weights(cfg, seed=seed, std=0.2))


def _f64(w):
    return {k: oracle.widen_bf16(v).astype(np.float64) for k, v in w.items()}


def _zero_layer_logits(cfg, w, tokens):
    x = torch.from_numpy(oracle.widen_bf16(w["embed"])[np.asarray(tokens)]).double()
    h = F.rms_norm(x, (cfg.hidden,), torch.from_numpy(oracle.widen_bf16(w["final_norm"])).double(),
                   eps=cfg.rms_eps)
    lm = w["embed"] if cfg.tied_embeddings else w["lm_head"]
    return (h @ torch.from_numpy(oracle.widen_bf16(lm)).double().T).numpy()


@pytest.mark.parametrize("tied", [False, True])
def test_zero_layers_closed_form(tied):
    cfg = TINY.replace(n_layers=0, tied_embeddings=tied)
    w = _w(cfg)
    toks = [3, 17]
    kv = np.zeros((0, 2, 2, 2, 4, 8), dtype=np.uint16)
    logits, _, _ = oracle.decode_step(cfg, w, toks, [0, 0], kv, F64)
    np.testing.assert_allclose(logits, _zero_layer_logits(cfg, w, toks), rtol=1e-12)


def test_zeroed_output_projections_make_layers_identity():
    cfg = TINY
    w = _f64(_w(cfg))
    for l in range(cfg.n_layers):
        w[f"layers.{l}.wo"][:] = 0
        w[f"layers.{l}.w_down"][:] = 0
    toks = np.array([5, 9, 44])
    kv = np.random.default_rng(0).normal(size=(cfg.n_layers, 2, 3, 2, 10, 8))
    logits, _, _ = oracle.decode_step(cfg, w, toks, [4, 0, 9], kv, F64)
    ref = _zero_layer_logits(cfg.replace(n_layers=0), {k: v for k, v in _w(cfg).items()}, toks)
    np.testing.assert_allclose(logits, ref, rtol=1e-12)


def _torch_prefill(cfg, w, tokens, kv_bf16=False):
    """Independent float64 forward from torch library ops (F.rms_norm, complex
    RoPE via torch.polar, F.scaled_dot_product_attention, F.silu); with kv_bf16
    the keys and values pass through torch's bfloat16 cast first."""
    T = {k: torch.from_numpy(oracle.widen_bf16(v)).double() for k, v in w.items()}
    S, d = len(tokens), cfg.head_dim
    x = T["embed"][torch.as_tensor(tokens)]
    inv = torch.tensor(cfg.rope_theta, dtype=torch.float64) ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(S, d // 2, dtype=torch.float64), torch.arange(S, dtype=torch.float64)[:, None] * inv)

    def rope(u):  # [heads, S, d]
        z = torch.complex(u[..., : d // 2], u[..., d // 2:]) * rot
        return torch.cat([z.real, z.imag], -1)

    for l in range(cfg.n_layers):
        p = f"layers.{l}."
        h = F.rms_norm(x, (cfg.hidden,), T[p + "attn_norm"], eps=cfg.rms_eps)
        q = (h @ T[p + "wq"].T).view(S, cfg.n_q_heads, d).transpose(0, 1)
        k = (h @ T[p + "wk"].T).view(S, cfg.n_kv_heads, d).transpose(0, 1)
        v = (h @ T[p + "wv"].T).view(S, cfg.n_kv_heads, d).transpose(0, 1)
        if cfg.qk_norm:
            q = F.rms_norm(q, (d,), T[p + "q_norm"], eps=cfg.rms_eps)
            k = F.rms_norm(k, (d,), T[p + "k_norm"], eps=cfg.rms_eps)
        q, k = rope(q), rope(k)
        if kv_bf16:
            k = k.float().to(torch.bfloat16).double()
            v = v.float().to(torch.bfloat16).double()
        rep = cfg.n_q_heads // cfg.n_kv_heads
        o = F.scaled_dot_product_attention(q, k.repeat_interleave(rep, 0), v.repeat_interleave(rep, 0),
                                           is_causal=True)
        x = x + o.transpose(0, 1).reshape(S, -1) @ T[p + "wo"].T
        h2 = F.rms_norm(x, (cfg.hidden,), T[p + "ffn_norm"], eps=cfg.rms_eps)
        x = x + (F.silu(h2 @ T[p + "w_gate"].T) * (h2 @ T[p + "w_up"].T)) @ T[p + "w_down"].T
    hf = F.rms_norm(x, (cfg.hidden,), T["final_norm"], eps=cfg.rms_eps)
    lm = T["embed"] if cfg.tied_embeddings else T["lm_head"]
    return (hf @ lm.T).numpy()


@pytest.mark.parametrize("qk_norm,tied", [(False, False), (True, False), (False, True)])
def test_prefill_vs_torch_library_forward(qk_norm, tied):
    cfg = TINY.replace(qk_norm=qk_norm, tied_embeddings=tied)
    w = _w(cfg, seed=1)
    toks = synth.make_tokens(11, cfg.vocab).numpy()
    got, _, _ = oracle.prefill(cfg, w, toks, F64, all_logits=True, kv_bf16=False)
    np.testing.assert_allclose(got, _torch_prefill(cfg, w, toks), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("qk_norm", [False, True])
def test_prefill_bf16_cache_vs_torch_library_forward(qk_norm):
    cfg = TINY.replace(qk_norm=qk_norm)
    w = _w(cfg, seed=1)
    toks = synth.make_tokens(11, cfg.vocab).numpy()
    got, K, V = oracle.prefill(cfg, w, toks, F64, all_logits=True)
    np.testing.assert_allclose(got, _torch_prefill(cfg, w, toks, kv_bf16=True), rtol=1e-10, atol=1e-12)
    # the K/V handed back are the stored (bf16) values
    assert np.all((K.astype(np.float32).view(np.uint32) & 0xFFFF) == 0)
    assert np.all((V.astype(np.float32).view(np.uint32) & 0xFFFF) == 0)
    plain, _, _ = oracle.prefill(cfg, w, toks, F64, all_logits=True, kv_bf16=False)
    assert np.abs(plain - got).max() > 1e-6          # the rounding is not a no-op


@pytest.mark.parametrize("qk_norm", [False, True])
def test_prefill_then_decode_equals_longer_prefill(qk_norm):
    cfg = TINY.replace(qk_norm=qk_norm)
    w = _w(cfg, seed=2)
    toks = synth.make_tokens(10, cfg.vocab, seed=5).numpy()
    S = 9
    _, K, V = oracle.prefill(cfg, w, toks[:S], F64)
    kv = np.zeros((cfg.n_layers, 2, 1, cfg.n_kv_heads, 16, cfg.head_dim))
    kv[:, 0, 0, :, :S] = K
    kv[:, 1, 0, :, :S] = V
    dec, knew, vnew = oracle.decode_step(cfg, w, toks[S:S + 1], [S], kv, F64)
    full, K2, V2 = oracle.prefill(cfg, w, toks, F64)
    np.testing.assert_allclose(dec[0], full, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(knew[:, 0], K2[:, :, S], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(vnew[:, 0], V2[:, :, S], rtol=1e-11, atol=1e-12)


def test_prefill_causality():
    cfg = TINY
    w = _w(cfg, seed=3)
    toks = synth.make_tokens(8, cfg.vocab, seed=6).numpy()
    full, _, _ = oracle.prefill(cfg, w, toks, F64, all_logits=True)
    toks2 = toks.copy()
    toks2[5:] = (toks2[5:] + 7) % cfg.vocab
    other, _, _ = oracle.prefill(cfg, w, toks2, F64, all_logits=True)
    np.testing.assert_array_equal(full[:5], other[:5])
    assert np.abs(full[5:] - other[5:]).max() > 1e-6


def test_decode_batch_rows_independent():
    cfg = TINY.replace(qk_norm=True)
    w = _w(cfg, seed=4)
    rng = np.random.default_rng(13)
    kv = rng.normal(size=(cfg.n_layers, 2, 3, cfg.n_kv_heads, 12, cfg.head_dim))
    toks, pos = np.array([1, 2, 3]), np.array([0, 11, 5])
    full, kn, vn = oracle.decode_step(cfg, w, toks, pos, kv, F64)
    for b in range(3):
        one, k1, v1 = oracle.decode_step(cfg, w, toks[b:b + 1], pos[b:b + 1], kv[:, :, b:b + 1], F64)
        np.testing.assert_allclose(full[b], one[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(kn[:, b], k1[:, 0], rtol=1e-12, atol=1e-13)


def test_qk_norm_makes_q_and_k_scale_invariant():
    cfg = TINY.replace(qk_norm=True, rms_eps=1e-30)
    w = _f64(_w(cfg, seed=5))
    rng = np.random.default_rng(14)
    kv = rng.normal(size=(cfg.n_layers, 2, 1, cfg.n_kv_heads, 6, cfg.head_dim))
    base, _, _ = oracle.decode_step(cfg, w, [7], [5], kv, F64)
    w2 = dict(w)
    for l in range(cfg.n_layers):
        w2[f"layers.{l}.wq"] = 3.0 * w[f"layers.{l}.wq"]
        w2[f"layers.{l}.wk"] = 0.5 * w[f"layers.{l}.wk"]
    scaled, _, _ = oracle.decode_step(cfg, w2, [7], [5], kv, F64)
    np.testing.assert_allclose(scaled, base, rtol=1e-11)
    plain = cfg.replace(qk_norm=False)
    a, _, _ = oracle.decode_step(plain, w, [7], [5], kv, F64)
    b, _, _ = oracle.decode_step(plain, w2, [7], [5], kv, F64)
    assert np.abs(a - b).max() > 1e-6


def test_float32_close_to_float64():
    cfg = TINY.replace(qk_norm=True)
    w = _w(cfg, seed=6)
    kv = synth.bf16_bits(synth.make_kv_cache(cfg, 2, 20))
    a, _, _ = oracle.decode_step(cfg, w, [4, 8], [19, 3], kv, np.float32)
    b, _, _ = oracle.decode_step(cfg, w, [4, 8], [19, 3], kv, F64)
    assert np.abs(a - b).max() <= 1e-4 * np.sqrt((b ** 2).mean())


def test_decode_new_kv_is_the_rounded_value():
    cfg = TINY.replace(qk_norm=True)
    w = _w(cfg, seed=8)
    kv = synth.bf16_bits(synth.make_kv_cache(cfg, 2, 12))
    _, kn, vn = oracle.decode_step(cfg, w, [3, 9], [11, 0], kv, F64)
    _, kp, vp = oracle.decode_step(cfg, w, [3, 9], [11, 0], kv, F64, kv_bf16=False)
    # layer 0 computes the same k, v either way; later layers see the rounding
    np.testing.assert_array_equal(kn[0], oracle.round_bf16(kp[0], F64))
    np.testing.assert_array_equal(vn[0], oracle.round_bf16(vp[0], F64))
    assert np.all((kn.astype(np.float32).view(np.uint32) & 0xFFFF) == 0)
    assert np.abs(kn[0] - kp[0]).max() > 0
