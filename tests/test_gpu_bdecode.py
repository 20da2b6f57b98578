"""Batched decode on the tensor cores (plans whose batch the CUDA-core decode
path does not take), through the C ABI, against the CPU oracle.

Tolerances (written here): per logits row b,
    max_v |gpu[b, v] - oracle[b, v]| <= 2e-2 * RMS_v(oracle[b, :]);
the key and value written to slot positions[b] are bf16 like the oracle's
(rounded the same way), so each element is within two bf16 spacings plus
2e-2 * RMS of the oracle's.  Exact bit-identity across runs, persistent-CTA
counts, random topological queue orders and the kernel-per-operator runner.
"""
import numpy as np
import pytest
import torch

import oracle
from tile_level_overlap_gb300 import build, mk, synth

pytestmark = pytest.mark.gpu

TOL = 2e-2

# small shapes that exercise: one K chunk (head_dim 64), q/k norm with
# head_dim 128, and split-K over 2..4 chunks
BD_SMALL = synth.ModelCfg(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512,
                          vocab=1000, rms_eps=1e-5, rope_theta=1e4)
BD_D128_QK = synth.ModelCfg(n_layers=2, hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, ffn=768,
                            vocab=700, rms_eps=1e-6, rope_theta=1e6, qk_norm=True)
BD_SPLITK = synth.ModelCfg(n_layers=2, hidden=2048, n_q_heads=16, n_kv_heads=4, head_dim=128,
                           ffn=4096, vocab=3000, rms_eps=1e-5, rope_theta=5e5)


def _rows_close(got, ref, tol=TOL):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    for b in range(ref.shape[0]):
        rms = np.sqrt((ref[b] ** 2).mean())
        err = np.abs(got[b] - ref[b]).max()
        assert err <= tol * rms, f"row {b}: max |delta| {err:.4e} > {tol} * rms {rms:.4e}"


def _kv_close(name, gpu, orc):
    gpu = np.asarray(gpu, np.float64)
    orc = np.asarray(orc, np.float64)
    rms = np.sqrt((orc ** 2).mean())
    bad = np.abs(gpu - orc) > 2.0 ** -6 * np.abs(orc) + 2e-2 * rms
    assert not bad.any(), f"{name}: {bad.sum()} elements off by more than two bf16 spacings"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    mk.lib()


class BModel:
    def __init__(self, cfg, max_batch, max_ctx, seed=0):
        self.cfg = cfg
        self.dev = torch.device("cuda:0")
        self.w = synth.make_weights(cfg, seed=seed, device=self.dev)
        self.kv = synth.make_kv_cache(cfg, max_batch, max_ctx, device=self.dev)
        self.plan = mk.Plan(cfg, self.w, max_batch, max_ctx)
        self.max_batch = max_batch
        assert self.plan.kv_cache_bytes() == self.kv.numel() * 2
        # the batch exceeds what the CUDA-core path takes: tensor-core plan
        assert self.plan.stats().decode_path == 1

    def step(self, tokens, positions, per_op=False, graph=False):
        t = torch.as_tensor(tokens, dtype=torch.int32).to(self.dev)
        p = torch.as_tensor(positions, dtype=torch.int32).to(self.dev)
        logits = torch.full((len(tokens), self.cfg.vocab), float("nan"), device=self.dev)
        if per_op:
            self.plan.run_per_op(mk.MK_DECODE, t, p, self.kv, logits, use_graph=graph)
        else:
            self.plan.decode_step(t, p, self.kv, logits)
        rc = self.plan.status()
        assert rc == mk.MK_OK, mk.lib().mk_status_string(rc)
        return logits.cpu().numpy()

    def check(self, tokens, positions):
        kv_before = synth.bf16_bits(self.kv)
        got = self.step(tokens, positions)
        ref, knew, vnew = oracle.decode_step(self.cfg, synth.LazyBits(self.w), tokens, positions,
                                             kv_before)
        _rows_close(got, ref)
        kv_after = oracle.widen_bf16(synth.bf16_bits(self.kv))
        for b, pb in enumerate(positions):
            _kv_close(f"k[{b}]", kv_after[:, 0, b, :, pb, :], knew[:, b])
            _kv_close(f"v[{b}]", kv_after[:, 1, b, :, pb, :], vnew[:, b])
        # nothing else of the cache moved
        before = oracle.widen_bf16(kv_before)
        mask = np.ones(before.shape[:5], dtype=bool)
        for b, pb in enumerate(positions):
            mask[:, :, b, :, pb] = False
        np.testing.assert_array_equal(kv_after[mask], before[mask])
        return got

    def close(self):
        self.plan.close()
        del self.w, self.kv
        torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def small():
    m = BModel(BD_SMALL, max_batch=12, max_ctx=300)
    yield m
    m.close()


@pytest.mark.parametrize("batch", [12, 9, 1])
def test_small_batched_matches_oracle(small, batch):
    tokens = synth.make_tokens(batch, small.cfg.vocab, seed=batch).numpy()
    positions = synth.make_contexts(batch, 0, 299, seed=batch).numpy()
    small.check(tokens, positions)


def test_small_edge_positions(small):
    # a fresh sequence (nothing cached), short contexts fewer than the splits,
    # and the last slot of the cache
    positions = np.array([0, 1, 2, 3, 4, 63, 64, 65, 127, 128, 200, 299], dtype=np.int32)
    tokens = synth.make_tokens(12, small.cfg.vocab, seed=77).numpy()
    small.check(tokens, positions)


def test_small_bit_identical_runs_ctas_orders_and_per_op(small):
    tokens = synth.make_tokens(12, small.cfg.vocab, seed=5).numpy()
    positions = synth.make_contexts(12, 10, 290, seed=5).numpy()
    ref = small.step(tokens, positions)
    np.testing.assert_array_equal(small.step(tokens, positions), ref)
    n = small.plan.stats().n_ctas
    try:
        for ctas in [1, 7, n // 2]:
            small.plan.set_debug(force_ctas=ctas)
            np.testing.assert_array_equal(small.step(tokens, positions), ref)
        for seed in [3, 11]:
            small.plan.set_debug(queue_perm_seed=seed)
            np.testing.assert_array_equal(small.step(tokens, positions), ref)
    finally:
        small.plan.set_debug()
    np.testing.assert_array_equal(small.step(tokens, positions, per_op=True), ref)
    np.testing.assert_array_equal(small.step(tokens, positions, per_op=True, graph=True), ref)
    try:
        small.plan.set_lm_mode(mk.MK_LM_SEPARATE)
        np.testing.assert_array_equal(small.step(tokens, positions), ref)
    finally:
        small.plan.set_lm_mode(mk.MK_LM_FUSED)


def test_head_dim_128_qk_norm_batched():
    m = BModel(BD_D128_QK, max_batch=16, max_ctx=200, seed=3)
    try:
        tokens = synth.make_tokens(16, m.cfg.vocab, seed=9).numpy()
        positions = synth.make_contexts(16, 0, 199, seed=9).numpy()
        m.check(tokens, positions)
    finally:
        m.close()


def test_split_k_batched():
    m = BModel(BD_SPLITK, max_batch=20, max_ctx=160, seed=4)
    try:
        tokens = synth.make_tokens(20, m.cfg.vocab, seed=13).numpy()
        positions = synth.make_contexts(20, 5, 159, seed=13).numpy()
        m.check(tokens, positions)
    finally:
        m.close()


def test_llama3_8b_width_batch8_context4096():
    """Llama-3-8B widths (2 of 32 layers), 8 sequences at context 4096: the
    batch-8 decode workload."""
    cfg = synth.LLAMA3_8B.replace(n_layers=2)
    m = BModel(cfg, max_batch=8, max_ctx=4097)
    try:
        tokens = synth.make_tokens(8, cfg.vocab, seed=21).numpy()
        m.check(tokens, np.full(8, 4096, dtype=np.int32))
    finally:
        m.close()


def test_qwen3_8b_width_batch32_ragged():
    """Qwen3-8B widths (q/k norm; 2 of 36 layers), 32 sequences with cached
    lengths uniform in [512, 2048]: the ragged batch-32 decode workload."""
    cfg = synth.QWEN3_8B.replace(n_layers=2)
    m = BModel(cfg, max_batch=32, max_ctx=2049)
    try:
        tokens = synth.make_tokens(32, cfg.vocab, seed=22).numpy()
        positions = synth.make_contexts(32, 512, 2048).numpy()
        m.check(tokens, positions)
    finally:
        m.close()


def _chunk_with_decode(m, p0, chunk, dec_slots, dec_pos, seed):
    """mk_decode_step_slots: a prompt chunk of slot 0 (positions p0 ..
    p0 + chunk - 1) and decode tokens of other slots in one persistent launch.
    The oracle runs the chunk token by token (each step appending its
    key/value) and the decode columns as one step on the cache before the
    launch."""
    cfg = m.cfg
    toks = synth.make_tokens(chunk + len(dec_slots), cfg.vocab, seed=seed).numpy()
    slots = np.array([0] * chunk + dec_slots, dtype=np.int32)
    pos = np.array([p0 + i for i in range(chunk)] + dec_pos, dtype=np.int32)
    kv_before = synth.bf16_bits(m.kv)
    n = len(toks)
    lg = torch.full((n, cfg.vocab), float("nan"), device=m.dev)
    m.plan.decode_step_slots(torch.from_numpy(toks.astype(np.int32)).to(m.dev),
                             torch.from_numpy(pos).to(m.dev),
                             torch.from_numpy(slots).to(m.dev), m.kv, lg)
    rc = m.plan.status()
    assert rc == mk.MK_OK, mk.lib().mk_status_string(rc)
    got = lg.cpu().numpy()
    w = synth.LazyBits(m.w)
    # the chunk, token by token, on slot 0's cache
    kv0 = kv_before[:, :, 0:1].copy()
    for i in range(chunk):
        ref, knew, vnew = oracle.decode_step(cfg, w, toks[i:i + 1], [p0 + i], kv0)
        _rows_close(got[i:i + 1], ref)
        kb = torch.from_numpy(np.ascontiguousarray(knew[:, 0])).to(torch.bfloat16).view(torch.int16).numpy()
        vb = torch.from_numpy(np.ascontiguousarray(vnew[:, 0])).to(torch.bfloat16).view(torch.int16).numpy()
        kv0[:, 0, 0, :, p0 + i, :] = kb.view(kv0.dtype)
        kv0[:, 1, 0, :, p0 + i, :] = vb.view(kv0.dtype)
    after = oracle.widen_bf16(synth.bf16_bits(m.kv))
    np.testing.assert_allclose(after[:, :, 0, :, p0:p0 + chunk], oracle.widen_bf16(kv0)[:, :, 0, :, p0:p0 + chunk],
                               rtol=2.0 ** -6, atol=2e-2)
    # the decode columns: one step of their slots (sequence b in slot b)
    lo, hi = dec_slots[0], dec_slots[-1] + 1
    assert dec_slots == list(range(lo, hi))
    kvd = kv_before[:, :, lo:hi].copy()
    ref, _, _ = oracle.decode_step(cfg, w, toks[chunk:], dec_pos, kvd)
    _rows_close(got[chunk:], ref)


def test_prompt_chunk_mixed_with_decode(small):
    """A 6-token prompt chunk of slot 0 with decode tokens of slots 1..5."""
    _chunk_with_decode(small, 150, 6, [1, 2, 3, 4, 5], [10, 299, 0, 77, 128], seed=91)
    # a slot outside the plan latches a bounds error
    small.plan.reset()
    bad = torch.tensor([0, 12], dtype=torch.int32, device=small.dev)
    lg = torch.empty((2, small.cfg.vocab), device=small.dev)
    small.plan.decode_step_slots(torch.tensor([1, 2], dtype=torch.int32, device=small.dev),
                                 torch.tensor([5, 6], dtype=torch.int32, device=small.dev), bad,
                                 small.kv, lg)
    assert small.plan.status() == mk.MK_ERR_BOUNDS
    small.plan.reset()


def test_prompt_chunk_crossing_a_key_block():
    """A chunk at positions 510..515: for its last token (516 keys, the last
    split from key 387) the chunk's first rows lie in the split's first
    128-key block and its own row in the next, so the block holding rows this
    step writes is not the block holding the column's own row; both must be
    streamed only after the projection wrote them."""
    m = BModel(BD_SMALL, max_batch=12, max_ctx=600, seed=7)
    try:
        _chunk_with_decode(m, 510, 6, [1, 2, 3], [599, 3, 300], seed=92)
    finally:
        m.close()
