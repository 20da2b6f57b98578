"""Thin Python binding of libmk's C ABI (include/mk.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of libmk.  Tensors are passed as raw device pointers; PyTorch is used
for device memory and streams.  There is no fallback: if libmk.so is missing
or no GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmk.so")

MK_OK = 0
MK_ERR_INVALID_ARG = 1
MK_ERR_CUDA = 2
MK_ERR_TIMEOUT = 3
MK_ERR_BOUNDS = 4
MK_ERR_UNSUPPORTED = 5
MK_ERR_NO_DEVICE = 6
MK_DECODE = 0
MK_PREFILL = 1
MK_LM_FUSED, MK_LM_SEPARATE = 0, 1
TRACE_WORDS = 16  # u64 words per trace record (mk_trace_copy)
MK_NOALLOC_SCRATCH_BYTES = 16 << 20  # static device scratch of mk_decode_step_noalloc

EXPORTED = [
    "mk_plan_create", "mk_plan_destroy", "mk_kv_cache_bytes", "mk_decode_step",
    "mk_decode_step_host", "mk_prefill", "mk_run_per_op", "mk_status", "mk_plan_reset",
    "mk_status_string", "mk_plan_get_stats", "mk_plan_check", "mk_plan_set_debug",
    "mk_trace_copy", "mk_plan_debug_drop_release", "mk_debug_gemm_bf16", "mk_decode_step_noalloc",
    "mk_plan_set_lm_mode", "mk_decode_steps", "mk_prefill_logits", "mk_prefill_batch",
    "mk_decode_step_slots", "mk_plan_create_for_sms", "mk_prefill_chunks",
]


class mk_model_cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("qk_norm", ctypes.c_int), ("tied_embeddings", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class mk_weight_ptrs(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p)] + [(n, _PP) for n in (
                    "attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "ffn_norm",
                    "w_gate", "w_up", "w_down")]


class mk_plan_stats(ctypes.Structure):
    _fields_ = [("n_instr_decode", ctypes.c_uint32), ("n_instr_prefill", ctypes.c_uint32),
                ("n_barriers", ctypes.c_uint32), ("n_launches_per_op_decode", ctypes.c_uint32),
                ("n_ctas", ctypes.c_uint32), ("n_splits", ctypes.c_uint32),
                ("weight_bytes", ctypes.c_uint64), ("scratch_bytes", ctypes.c_uint64),
                ("decode_path", ctypes.c_uint32), ("queue_hash", ctypes.c_uint64)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmk.so (built by tile_level_overlap_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with tile_level_overlap_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    L.mk_plan_create.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.POINTER(mk_weight_ptrs),
                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)]
    L.mk_plan_create_for_sms.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.POINTER(mk_weight_ptrs),
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)]
    L.mk_plan_destroy.argtypes = [vp]
    L.mk_plan_destroy.restype = None
    L.mk_kv_cache_bytes.argtypes = [vp]
    L.mk_kv_cache_bytes.restype = ctypes.c_size_t
    L.mk_decode_step.argtypes = [vp, i32p, i32p, ctypes.c_int, vp, f32p, vp]
    L.mk_decode_step_host.argtypes = [vp, i32p, i32p, ctypes.c_int, vp, f32p, vp]
    L.mk_prefill.argtypes = [vp, i32p, ctypes.c_int, vp, f32p, vp]
    L.mk_run_per_op.argtypes = [vp, ctypes.c_int, ctypes.c_int, i32p, i32p, ctypes.c_int, vp, f32p, vp]
    L.mk_status.argtypes = [vp, vp]
    L.mk_plan_reset.argtypes = [vp, vp]
    L.mk_status_string.argtypes = [ctypes.c_int]
    L.mk_status_string.restype = ctypes.c_char_p
    L.mk_plan_get_stats.argtypes = [vp, ctypes.POINTER(mk_plan_stats)]
    L.mk_plan_check.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.c_int, ctypes.c_int,
                                ctypes.c_uint64, ctypes.POINTER(mk_plan_stats)]
    L.mk_plan_set_debug.argtypes = [vp, ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64]
    L.mk_plan_set_lm_mode.argtypes = [vp, ctypes.c_int]
    L.mk_decode_steps.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, vp, vp]
    L.mk_prefill_logits.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp]
    L.mk_decode_step_slots.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp, vp]
    L.mk_prefill_batch.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int,
                                   vp, vp, vp]
    L.mk_prefill_chunks.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, vp, vp, vp]
    L.mk_trace_copy.argtypes = [vp, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
    L.mk_plan_debug_drop_release.argtypes = [vp, ctypes.c_uint32]
    L.mk_debug_gemm_bf16.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, vp]
    L.mk_decode_step_noalloc.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.POINTER(mk_weight_ptrs),
                                         ctypes.c_int, ctypes.c_int, i32p, i32p, ctypes.c_int, vp,
                                         f32p, vp]
    _lib = L
    return L


class MkError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {lib().mk_status_string(code).decode()} (code {code})")


def _check(code: int, what: str) -> None:
    if code != MK_OK:
        raise MkError(code, what)


def model_cfg(cfg) -> mk_model_cfg:
    return mk_model_cfg(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                        cfg.ffn, cfg.vocab, float(cfg.rms_eps), float(cfg.rope_theta),
                        int(bool(cfg.qk_norm)), int(bool(cfg.tied_embeddings)))


def plan_check(cfg, max_batch: int, max_ctx: int, seed: int = 0):
    """Host-only plan build + simulation; returns (status, stats)."""
    st = mk_plan_stats()
    rc = lib().mk_plan_check(ctypes.byref(model_cfg(cfg)), max_batch, max_ctx, seed, ctypes.byref(st))
    return rc, st


def weight_ptrs(cfg, weights):
    """mk_weight_ptrs over name -> torch bf16 CUDA tensor; returns (struct,
    keep-alive list of the pointer arrays it references)."""
    n = cfg.n_layers
    keep = []
    wp = mk_weight_ptrs()
    wp.embed = _ptr(weights["embed"])
    wp.final_norm = _ptr(weights["final_norm"])
    wp.lm_head = _ptr(weights["lm_head"]) if "lm_head" in weights else None
    for k in ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "ffn_norm", "w_gate", "w_up",
              "w_down"):
        if all(f"layers.{l}.{k}" in weights for l in range(n)):
            a = (ctypes.c_void_p * n)(*[_ptr(weights[f"layers.{l}.{k}"]) for l in range(n)])
            keep.append(a)
            setattr(wp, k, ctypes.cast(a, _PP))
    return wp, keep


def decode_step_noalloc(cfg, weights, max_batch: int, max_ctx: int, tokens, positions, kv, logits,
                        stream=None) -> int:
    """mk_decode_step_noalloc: one decode step using only the library's static
    device scratch (no device allocation).  Returns the C status code."""
    wp, keep = weight_ptrs(cfg, weights)
    rc = lib().mk_decode_step_noalloc(ctypes.byref(model_cfg(cfg)), ctypes.byref(wp), max_batch,
                                      max_ctx, _ptr(tokens), _ptr(positions), int(tokens.numel()),
                                      _ptr(kv), _ptr(logits), _stream_ptr(stream))
    del keep
    return rc


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t) -> int:
    return int(t.data_ptr())


class Plan:
    """A plan over weights held as torch bf16 CUDA tensors (name -> tensor, as
    produced by synth.make_weights).  Keeps references so the weights outlive
    the plan."""

    def __init__(self, cfg, weights: Dict[str, "object"], max_batch: int, max_ctx: int,
                 n_sms: int = 0):
        """n_sms > 0 (test-only): tile and launch the plan as on a device with
        that many SMs (mk_plan_create_for_sms)."""
        L = lib()
        self.cfg = cfg
        self.max_batch = max_batch
        self.max_ctx = max_ctx
        self._w = weights
        n = cfg.n_layers

        def arr(key):
            if not all(f"layers.{l}.{key}" in weights for l in range(n)):
                return None
            a = (ctypes.c_void_p * n)(*[_ptr(weights[f"layers.{l}.{key}"]) for l in range(n)])
            return a

        self._arrays = {k: arr(k) for k in ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm",
                                            "ffn_norm", "w_gate", "w_up", "w_down")}
        wp = mk_weight_ptrs()
        wp.embed = _ptr(weights["embed"])
        wp.final_norm = _ptr(weights["final_norm"])
        wp.lm_head = _ptr(weights["lm_head"]) if "lm_head" in weights else None
        for k, a in self._arrays.items():
            setattr(wp, k, ctypes.cast(a, _PP) if a is not None else None)
        h = ctypes.c_void_p()
        _check(L.mk_plan_create_for_sms(ctypes.byref(model_cfg(cfg)), ctypes.byref(wp), max_batch,
                                        max_ctx, int(n_sms), ctypes.byref(h)), "mk_plan_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().mk_plan_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- sizes
    def kv_cache_bytes(self) -> int:
        return int(lib().mk_kv_cache_bytes(self.h))

    def stats(self) -> mk_plan_stats:
        st = mk_plan_stats()
        _check(lib().mk_plan_get_stats(self.h, ctypes.byref(st)), "mk_plan_get_stats")
        return st

    # ---- steps (device tensors)
    def decode_step(self, tokens, positions, kv, logits, stream=None) -> None:
        _check(lib().mk_decode_step(self.h, _ptr(tokens), _ptr(positions), int(tokens.numel()),
                                    _ptr(kv), _ptr(logits), _stream_ptr(stream)), "mk_decode_step")

    def decode_steps(self, token, position, n_steps: int, kv, out_tokens, logits, stream=None) -> None:
        """mk_decode_steps: n_steps greedy decode steps of one sequence in one
        launch (device tensors: token [1], position [1], out_tokens [n_steps],
        logits [V])."""
        _check(lib().mk_decode_steps(self.h, _ptr(token), _ptr(position), int(n_steps), _ptr(kv),
                                     _ptr(out_tokens), _ptr(logits), _stream_ptr(stream)),
               "mk_decode_steps")

    def decode_step_slots(self, tokens, positions, slots, kv, logits, stream=None) -> None:
        """mk_decode_step_slots: column c is tokens[c] of cache slot slots[c] at
        positions[c] (a prompt chunk = several columns of one slot)."""
        _check(lib().mk_decode_step_slots(self.h, _ptr(tokens), _ptr(positions), _ptr(slots),
                                          int(tokens.numel()), _ptr(kv), _ptr(logits),
                                          _stream_ptr(stream)), "mk_decode_step_slots")

    def decode_step_host(self, tokens, positions, kv, logits, stream=None) -> int:
        """tokens/positions/logits are CPU tensors (pinned for speed)."""
        return lib().mk_decode_step_host(self.h, _ptr(tokens), _ptr(positions), int(tokens.numel()),
                                         _ptr(kv), _ptr(logits), _stream_ptr(stream))

    def prefill(self, tokens, kv, logits, stream=None) -> None:
        _check(lib().mk_prefill(self.h, _ptr(tokens), int(tokens.numel()), _ptr(kv), _ptr(logits),
                                _stream_ptr(stream)), "mk_prefill")

    def prefill_batch(self, tokens, lens, kv, logits, stream=None) -> None:
        """mk_prefill_batch: tokens device [batch, stride], lens a list of
        prompt lengths, logits device [batch, V]; prompt b to cache slot b."""
        n = len(lens)
        arr = (ctypes.c_int32 * n)(*[int(v) for v in lens])
        _check(lib().mk_prefill_batch(self.h, _ptr(tokens), arr, n, int(tokens.shape[1]), _ptr(kv),
                                      _ptr(logits), _stream_ptr(stream)), "mk_prefill_batch")

    def prefill_chunks(self, tokens, chunks, kv, logits, stream=None) -> None:
        """mk_prefill_chunks: tokens device int32 [*], chunks a list of (slot,
        pos0, len, token offset), logits device [n, V]."""
        n = len(chunks)
        flat = [int(v) for c in chunks for v in c]
        arr = (ctypes.c_int32 * (4 * n))(*flat)
        _check(lib().mk_prefill_chunks(self.h, _ptr(tokens), arr, n, _ptr(kv), _ptr(logits),
                                       _stream_ptr(stream)), "mk_prefill_chunks")

    def prefill_logits(self, tokens, kv, logits, stream=None) -> None:
        """mk_prefill_logits: the prompt's logits for every token, [len, V]."""
        _check(lib().mk_prefill_logits(self.h, _ptr(tokens), int(tokens.numel()), _ptr(kv),
                                       _ptr(logits), _stream_ptr(stream)), "mk_prefill_logits")

    def run_per_op(self, mode: int, tokens, positions, kv, logits, use_graph: bool = False,
                   stream=None) -> None:
        n = int(tokens.numel())
        _check(lib().mk_run_per_op(self.h, mode, int(use_graph), _ptr(tokens),
                                   _ptr(positions) if positions is not None else None, n,
                                   _ptr(kv), _ptr(logits), _stream_ptr(stream)), "mk_run_per_op")

    def status(self, stream=None) -> int:
        return lib().mk_status(self.h, _stream_ptr(stream))

    def reset(self, stream=None) -> None:
        _check(lib().mk_plan_reset(self.h, _stream_ptr(stream)), "mk_plan_reset")

    def set_debug(self, force_ctas: int = 0, queue_perm_seed: int = 0, trace: bool = False,
                  wait_limit_ns: int = 0) -> None:
        _check(lib().mk_plan_set_debug(self.h, force_ctas, queue_perm_seed, int(trace), wait_limit_ns),
               "mk_plan_set_debug")

    def set_lm_mode(self, mode: int) -> None:
        """MK_LM_FUSED: the LM head inside the persistent step; MK_LM_SEPARATE:
        the layers persistent, then the LM head as a kernel-per-operator launch."""
        _check(lib().mk_plan_set_lm_mode(self.h, mode), "mk_plan_set_lm_mode")

    def debug_drop_release(self, index: int) -> None:
        _check(lib().mk_plan_debug_drop_release(self.h, index), "mk_plan_debug_drop_release")

    def trace(self):
        """Trace records of the last traced launch as a numpy structured array."""
        import numpy as np
        n = self.stats().n_instr_decode
        buf = np.zeros(n * TRACE_WORDS, dtype=np.uint64)
        got = ctypes.c_size_t()
        _check(lib().mk_trace_copy(self.h, buf.ctypes.data, buf.nbytes, ctypes.byref(got)), "mk_trace_copy")
        rec = buf[: got.value * TRACE_WORDS].reshape(-1, TRACE_WORDS)
        return rec
