"""mk_decode_step_noalloc: the decode step for callers that cannot allocate
device memory when they run it (their device memory is already owned by their
own pool or by an external memory manager).  Its scratch is the library's
static device array, so it is checked against the plan-based entry point,
mk_decode_step, on the same inputs: logits per row within
2e-2 * RMS(reference row), the tolerance of the other decode tests, and
bit-identical (the same plan, kernel and queue run in both), on two calls in a
row (the second finds the first call's leftovers in the array).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import time

import numpy as np
import pytest
import torch

from tile_level_overlap_gb300 import build, mk, synth

pytestmark = pytest.mark.gpu

TOL = 2e-2

# A second shape for the interleaving test: head_dim 128 with q/k norm.
D128_QK = synth.ModelCfg(n_layers=2, hidden=512, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=768,
                         vocab=1000, rms_eps=1e-6, rope_theta=1e6, qk_norm=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    mk.lib()


def _close(got, ref):
    for b in range(ref.shape[0]):
        rms = np.sqrt((ref[b] ** 2).mean())
        assert np.abs(got[b] - ref[b]).max() <= TOL * rms


@pytest.mark.parametrize("cfg,max_batch,max_ctx,positions", [
    (synth.TOY_1L, 4, 129, [128, 0, 77]),
    (synth.LLAMA32_1B, 1, 1025, [1024]),
])
def test_noalloc_matches_plan_entry_point(cfg, max_batch, max_ctx, positions):
    dev = torch.device("cuda:0")
    w = synth.make_weights(cfg, device=dev)
    kv = synth.make_kv_cache(cfg, max_batch, max_ctx, device=dev)
    B = len(positions)
    tokens = synth.make_tokens(B, cfg.vocab).to(dev)
    pos = torch.tensor(positions, dtype=torch.int32, device=dev)
    plan = mk.Plan(cfg, w, max_batch, max_ctx)
    ref = torch.empty((B, cfg.vocab), device=dev)
    plan.decode_step(tokens, pos, kv, ref)
    assert plan.status() == mk.MK_OK
    ref = ref.cpu().numpy()
    plan.close()
    for _ in range(2):
        got = torch.full((B, cfg.vocab), float("nan"), device=dev)
        rc = mk.decode_step_noalloc(cfg, w, max_batch, max_ctx, tokens, pos, kv, got)
        assert rc == mk.MK_OK
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        _close(got, ref)
        np.testing.assert_array_equal(got, ref)
    del w, kv
    torch.cuda.empty_cache()


def test_noalloc_rejects_shapes_beyond_its_static_scratch():
    # A 65536-token cache at head_dim 128: its RoPE table alone (one (cos, sin)
    # float pair per position and rotation pair) is larger than the static
    # array, whatever the SM count or the tiling, so the call is refused before
    # any device work and every weight pointer may alias one small tensor.
    cfg = synth.LLAMA3_8B
    max_ctx = 1 << 16
    rope_bytes = max_ctx * (cfg.head_dim // 2) * 8
    assert rope_bytes > mk.MK_NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    x = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    w = {name: x for name in synth.weight_shapes(cfg)}
    t = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty((1, 8), device=dev)
    assert mk.decode_step_noalloc(cfg, w, 1, max_ctx, t, t, x, logits) == mk.MK_ERR_UNSUPPORTED


def _plan_logits(cfg, w, max_batch, max_ctx, tokens, pos, kv):
    plan = mk.Plan(cfg, w, max_batch, max_ctx)
    try:
        out = torch.empty((tokens.numel(), cfg.vocab), device=tokens.device)
        plan.decode_step(tokens, pos, kv, out)
        assert plan.status() == mk.MK_OK
        return out.cpu().numpy()
    finally:
        plan.close()


def test_noalloc_interleaved_shapes_and_moved_weights():
    """Calls that alternate between two shapes, and a call whose weights moved
    (same shape, other tensors): each is bit-identical to the plan entry point,
    so the array's queue, RoPE table and layer table are re-copied whenever the
    previous call left another shape's or other weights' in it.  Also prints
    the host time of a repeated call (plan and tables kept)."""
    dev = torch.device("cuda:0")
    cases = []
    for cfg, mb, mc, positions, seed in ((synth.TOY_1L, 4, 129, [128, 0, 77], 0),
                                         (D128_QK, 2, 300, [299, 5], 0)):
        w = synth.make_weights(cfg, seed=seed, device=dev)
        kv = synth.make_kv_cache(cfg, mb, mc, device=dev)
        t = synth.make_tokens(len(positions), cfg.vocab).to(dev)
        p = torch.tensor(positions, dtype=torch.int32, device=dev)
        cases.append((cfg, w, mb, mc, t, p, kv, _plan_logits(cfg, w, mb, mc, t, p, kv)))
    # the first shape with other weights (same shape, new tensors)
    cfg, _, mb, mc, t, p, kv, _ = cases[0]
    w2 = synth.make_weights(cfg, seed=5, device=dev)
    cases.append((cfg, w2, mb, mc, t, p, kv, _plan_logits(cfg, w2, mb, mc, t, p, kv)))
    for i in (0, 1, 0, 2, 0, 1, 1):
        cfg, w, mb, mc, t, p, kv, ref = cases[i]
        got = torch.full((t.numel(), cfg.vocab), float("nan"), device=dev)
        assert mk.decode_step_noalloc(cfg, w, mb, mc, t, p, kv, got) == mk.MK_OK
        np.testing.assert_array_equal(got.cpu().numpy(), ref)
    cfg, w, mb, mc, t, p, kv, _ = cases[1]
    got = torch.empty((t.numel(), cfg.vocab), device=dev)
    torch.cuda.synchronize()
    n = 20
    t0 = time.perf_counter()
    for _ in range(n):
        mk.decode_step_noalloc(cfg, w, mb, mc, t, p, kv, got)
    host_us = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize()
    print(f"NOALLOC host time per repeated call: {host_us:.1f} us")


def test_noalloc_refuses_a_capturing_stream():
    cfg = synth.TOY_1L
    dev = torch.device("cuda:0")
    w = synth.make_weights(cfg, device=dev)
    kv = synth.make_kv_cache(cfg, 1, 129, device=dev)
    t = synth.make_tokens(1, cfg.vocab).to(dev)
    p = torch.tensor([3], dtype=torch.int32, device=dev)
    out = torch.empty((1, cfg.vocab), device=dev)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    rc = None
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            out.zero_()
            rc = mk.decode_step_noalloc(cfg, w, 1, 129, t, p, kv, out, stream=s)
    assert rc == mk.MK_ERR_INVALID_ARG
