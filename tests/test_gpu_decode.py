"""Decode step on the GPU through the C ABI, against the CPU oracle.

Tolerance (written here, per logits row b):
    max_v |gpu[b, v] - oracle[b, v]| <= 2e-2 * RMS_v(oracle[b, :]).
Bit-identity (exact) across repeated runs, persistent-CTA counts, random
topological queue orders, and against the kernel-per-operator runner.
"""
import numpy as np
import pytest
import torch

import oracle
from tile_level_overlap_gb300 import build, mk, synth

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _assert_rows_close(got, ref, tol=TOL):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    for b in range(ref.shape[0]):
        rms = np.sqrt((ref[b] ** 2).mean())
        err = np.abs(got[b] - ref[b]).max()
        assert err <= tol * rms, f"row {b}: max |delta| {err:.4e} > {tol} * rms {rms:.4e}"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    mk.lib()


class Model:
    def __init__(self, cfg, max_batch, max_ctx, seed=0):
        self.cfg = cfg
        self.dev = torch.device("cuda:0")
        self.w = synth.make_weights(cfg, seed=seed, device=self.dev)
        self.kv = synth.make_kv_cache(cfg, max_batch, max_ctx, device=self.dev)
        self.plan = mk.Plan(cfg, self.w, max_batch, max_ctx)
        assert self.plan.kv_cache_bytes() == self.kv.numel() * 2

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

    def oracle(self, tokens, positions, kv_bits=None):
        kv_bits = synth.bf16_bits(self.kv) if kv_bits is None else kv_bits
        return oracle.decode_step(self.cfg, synth.LazyBits(self.w), tokens, positions, kv_bits)

    def close(self):
        self.plan.close()
        del self.w, self.kv
        torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def toy():
    m = Model(synth.TOY_1L, max_batch=4, max_ctx=129)
    yield m
    m.close()


@pytest.mark.parametrize("pos", [0, 1, 5, 63, 64, 127, 128])
def test_toy_decode_matches_oracle(toy, pos):
    tokens = synth.make_tokens(1, toy.cfg.vocab, seed=pos).numpy()
    kv_before = synth.bf16_bits(toy.kv)
    got = toy.step(tokens, [pos])
    ref, knew, vnew = toy.oracle(tokens, [pos], kv_before)
    _assert_rows_close(got, ref)
    # the step wrote the new token's (rotated) key and value into slot pos, as bf16
    kv_after = oracle.widen_bf16(synth.bf16_bits(toy.kv))
    k_slot = kv_after[:, 0, 0, :, pos, :]
    v_slot = kv_after[:, 1, 0, :, pos, :]
    np.testing.assert_allclose(k_slot, knew[:, 0], rtol=1e-2, atol=1e-2)
    np.testing.assert_allclose(v_slot, vnew[:, 0], rtol=1e-2, atol=1e-2)
    # nothing else in the cache changed
    mask = np.ones(kv_after.shape[4], dtype=bool)
    mask[pos] = False
    np.testing.assert_array_equal(kv_after[:, :, :, :, mask], oracle.widen_bf16(kv_before)[:, :, :, :, mask])


@pytest.mark.parametrize("positions", [[0, 64, 128], [17, 3, 100, 128], [5]])
def test_toy_batch_ragged(toy, positions):
    B = len(positions)
    tokens = synth.make_tokens(B, toy.cfg.vocab, seed=B).numpy()
    kv_before = synth.bf16_bits(toy.kv)
    got = toy.step(tokens, positions)
    ref, _, _ = toy.oracle(tokens, positions, kv_before)
    _assert_rows_close(got, ref)


def test_toy_repeat_bit_identical(toy):
    tokens, pos = [7, 8], [100, 50]
    first = toy.step(tokens, pos)
    for _ in range(9):
        np.testing.assert_array_equal(toy.step(tokens, pos), first)


def test_toy_per_op_and_graph_bit_identical(toy):
    tokens, pos = [11, 12, 13], [128, 0, 77]
    mega = toy.step(tokens, pos)
    np.testing.assert_array_equal(toy.step(tokens, pos, per_op=True), mega)
    np.testing.assert_array_equal(toy.step(tokens, pos, per_op=True, graph=True), mega)
    np.testing.assert_array_equal(toy.step(tokens, pos, per_op=True, graph=True), mega)
    np.testing.assert_array_equal(toy.step(tokens, pos), mega)


def test_toy_lm_separate_bit_identical(toy):
    """The LM head as its own kernel-per-operator launch after the persistent
    layers gives the same logits as the all-in-one step."""
    tokens, pos = [21, 22, 23], [64, 1, 120]
    fused = toy.step(tokens, pos)
    try:
        toy.plan.set_lm_mode(mk.MK_LM_SEPARATE)
        np.testing.assert_array_equal(toy.step(tokens, pos), fused)
        toy.plan.set_debug(queue_perm_seed=5)
        np.testing.assert_array_equal(toy.step(tokens, pos), fused)
    finally:
        toy.plan.set_lm_mode(mk.MK_LM_FUSED)
        toy.plan.set_debug()
    np.testing.assert_array_equal(toy.step(tokens, pos), fused)
    with pytest.raises(mk.MkError):
        toy.plan.set_lm_mode(7)


def test_toy_cta_counts_and_queue_orders(toy):
    tokens, pos = [3, 4], [128, 9]
    ref = toy.step(tokens, pos)
    n = torch.cuda.get_device_properties(0).multi_processor_count
    for ctas in [1, 2, 7, n // 2, n]:
        toy.plan.set_debug(force_ctas=ctas)
        np.testing.assert_array_equal(toy.step(tokens, pos), ref)
    for seed in [1, 2, 3, 4, 5]:
        toy.plan.set_debug(force_ctas=0, queue_perm_seed=seed)
        np.testing.assert_array_equal(toy.step(tokens, pos), ref)
    toy.plan.set_debug()


def test_queue_unchanged_by_steps(toy):
    """Symbolic extents: one queue serves every batch and position -- the
    device queue hashes the same before and after steps at several batches
    and positions, and the hash does see the queue (a permuted order changes
    it)."""
    h0 = toy.plan.stats().queue_hash
    for tokens, pos in [([1], [0]), ([2, 3], [5, 128]), ([4, 5, 6, 7], [1, 2, 3, 4]), ([9], [128])]:
        toy.step(tokens, pos)
        assert toy.plan.stats().queue_hash == h0
    toy.plan.set_debug(queue_perm_seed=3)
    assert toy.plan.stats().queue_hash != h0
    toy.plan.set_debug()
    assert toy.plan.stats().queue_hash == h0


def _sm_counts():
    n = torch.cuda.get_device_properties(0).multi_processor_count
    return sorted({n, min(n, 132), min(n, 100)}, reverse=True)


@pytest.mark.parametrize("cfg,max_ctx,positions,batches", [
    (synth.TOY_1L, 300, [0, 63, 64, 250, 299], (1, 4)),
    (synth.LLAMA32_1B.replace(n_layers=2), 1025, [1024, 300, 7], (1,)),
])
def test_bits_independent_of_sm_count_and_max_batch(cfg, max_ctx, positions, batches):
    """Schedule invariance beyond one plan: plans tiled and launched for 152,
    132 and 100 SMs, and with room for 1 or 4 sequences (the same CUDA-core
    path), give bit-identical logits for the same sequence in slot 0 (the
    split-KV tiling is a fixed number of keys per split, a model constant)."""
    dev = torch.device("cuda:0")
    w = synth.make_weights(cfg, seed=11, device=dev)
    kv1 = synth.make_kv_cache(cfg, 1, max_ctx, device=dev)
    ref = {}
    try:
        for mb in batches:
            kv = synth.make_kv_cache(cfg, mb, max_ctx, device=dev)
            for sms in _sm_counts():
                # every plan starts from the same cache (each step writes its
                # slot, which later positions of the sequence read)
                kv[:, :, 0].copy_(kv1[:, :, 0])
                plan = mk.Plan(cfg, w, mb, max_ctx, n_sms=sms)
                assert plan.stats().decode_path == 0
                for p in positions:
                    t = synth.make_tokens(1, cfg.vocab, seed=p).to(dev)
                    pp = torch.tensor([p], dtype=torch.int32, device=dev)
                    lg = torch.empty((1, cfg.vocab), device=dev)
                    plan.decode_step(t, pp, kv, lg)
                    assert plan.status() == mk.MK_OK
                    got = lg.cpu().numpy()
                    if p in ref:
                        np.testing.assert_array_equal(got, ref[p], err_msg=f"max_batch {mb}, {sms} SMs, pos {p}")
                    else:
                        ref[p] = got
                plan.close()
    finally:
        del w, kv1
        torch.cuda.empty_cache()


def test_toy_timeout_is_reported_and_recoverable(toy):
    tokens, pos = [3], [20]
    ref = toy.step(tokens, pos)
    # host-made bad plan: the first QKV tile no longer releases its barrier
    toy.plan.set_debug(wait_limit_ns=20_000_000)
    toy.plan.debug_drop_release(0)
    t = torch.tensor(tokens, dtype=torch.int32, device=toy.dev)
    p = torch.tensor(pos, dtype=torch.int32, device=toy.dev)
    logits = torch.empty((1, toy.cfg.vocab), device=toy.dev)
    toy.plan.decode_step(t, p, toy.kv, logits)
    assert toy.plan.status() == mk.MK_ERR_TIMEOUT
    with pytest.raises(mk.MkError):  # latched: nothing launches
        toy.plan.decode_step(t, p, toy.kv, logits)
    toy.plan.set_debug()
    toy.plan.reset()
    np.testing.assert_array_equal(toy.step(tokens, pos), ref)


def test_toy_out_of_range_token_and_position(toy):
    dev = toy.dev
    logits = torch.empty((1, toy.cfg.vocab), device=dev)
    for tok, pos in [(toy.cfg.vocab, 3), (-1, 3), (2, 129), (2, -5)]:
        t = torch.tensor([tok], dtype=torch.int32, device=dev)
        p = torch.tensor([pos], dtype=torch.int32, device=dev)
        toy.plan.decode_step(t, p, toy.kv, logits)
        assert toy.plan.status() == mk.MK_ERR_BOUNDS
        toy.plan.reset()
    toy.step([1], [1])


def test_toy_bad_arguments_rejected_before_launch(toy):
    dev = toy.dev
    t = torch.zeros(5, dtype=torch.int32, device=dev)
    p = torch.zeros(5, dtype=torch.int32, device=dev)
    logits = torch.empty((5, toy.cfg.vocab), device=dev)
    with pytest.raises(mk.MkError) as e:
        toy.plan.decode_step(t, p, toy.kv, logits)  # batch 5 > max_batch 4
    assert e.value.code == mk.MK_ERR_INVALID_ARG
    assert mk.lib().mk_decode_step(toy.plan.h, None, None, 1, None, None, None) == mk.MK_ERR_INVALID_ARG


def test_toy_host_buffer_entry_point(toy):
    tokens, pos = [9, 10], [128, 1]
    ref = toy.step(tokens, pos)
    th = torch.tensor(tokens, dtype=torch.int32).pin_memory()
    ph = torch.tensor(pos, dtype=torch.int32).pin_memory()
    lh = torch.empty((2, toy.cfg.vocab), dtype=torch.float32).pin_memory()
    assert toy.plan.decode_step_host(th, ph, toy.kv, lh) == mk.MK_OK
    np.testing.assert_array_equal(lh.numpy(), ref)


def test_toy_qk_norm_decode():
    m = Model(synth.TOY_1L.replace(qk_norm=True, rms_eps=1e-6, rope_theta=1e6), 2, 65, seed=3)
    try:
        for tokens, pos in [([5], [64]), ([6, 7], [0, 33])]:
            kv_before = synth.bf16_bits(m.kv)
            got = m.step(tokens, pos)
            ref, _, _ = m.oracle(tokens, pos, kv_before)
            _assert_rows_close(got, ref)
    finally:
        m.close()


@pytest.mark.parametrize("nq,nkv,d", [(4, 4, 64), (8, 1, 64), (4, 2, 128), (4, 1, 128), (8, 8, 128)])
def test_head_layouts_decode(nq, nkv, d):
    """1, 8, 2 and 4 query heads per kv head at both head sizes: the attention
    tile's tensor-core score rows (q of each head as bf16 hi and lo rows) for up
    to 4 heads and its CUDA-core scores for 8, at positions whose splits end
    inside an 8-key product (a few keys per split)."""
    cfg = synth.TOY_1L.replace(n_q_heads=nq, n_kv_heads=nkv, head_dim=d)
    m = Model(cfg, 2, 200, seed=5)
    try:
        for tokens, pos in [([3], [0]), ([9], [101]), ([4, 11], [157, 38]), ([2, 8], [199, 7])]:
            kv_before = synth.bf16_bits(m.kv)
            got = m.step(tokens, pos)
            ref, _, _ = m.oracle(tokens, pos, kv_before)
            _assert_rows_close(got, ref)
    finally:
        m.close()


def test_llama32_1b_decode_full_size():
    m = Model(synth.LLAMA32_1B, 1, 1025)
    try:
        tokens = synth.make_tokens(1, m.cfg.vocab).numpy()
        got = m.step(tokens, [1024])
        ref, _, _ = m.oracle(tokens, [1024])
        _assert_rows_close(got, ref)
        np.testing.assert_array_equal(m.step(tokens, [1024], per_op=True), got)
        m.plan.set_lm_mode(mk.MK_LM_SEPARATE)
        np.testing.assert_array_equal(m.step(tokens, [1024]), got)
    finally:
        m.close()


def test_llama3_8b_decode_full_size():
    """The benchmarked workload: 32 layers, hidden 4096, context 4096, batch 1,
    in the persistent launch configuration the benchmark times."""
    m = Model(synth.LLAMA3_8B, 1, 4097)
    try:
        tokens = synth.make_tokens(1, m.cfg.vocab).numpy()
        kv_before = synth.bf16_bits(m.kv)
        got = m.step(tokens, [4096])
        ref, _, _ = m.oracle(tokens, [4096], kv_before)
        _assert_rows_close(got, ref)
        np.testing.assert_array_equal(m.step(tokens, [4096]), got)
        # the same step tiled and launched for 100 SMs: bit-identical
        plan100 = mk.Plan(m.cfg, m.w, 1, 4097, n_sms=min(100, _sm_counts()[0]))
        t = torch.as_tensor(tokens, dtype=torch.int32).to(m.dev)
        p = torch.tensor([4096], dtype=torch.int32, device=m.dev)
        lg = torch.empty((1, m.cfg.vocab), device=m.dev)
        plan100.decode_step(t, p, m.kv, lg)
        assert plan100.status() == mk.MK_OK
        np.testing.assert_array_equal(lg.cpu().numpy(), got)
        plan100.close()
    finally:
        m.close()


def test_toy_combine_slices_batch_ragged():
    """A 4000-token cache on the toy shape: 63 splits per (sequence, kv
    head), combined in 3 slices.  Three sequences of one batch using all,
    some and one of the splits match the oracle, and the launch on 5 CTAs
    with a permuted queue and the kernel-per-operator graph give the same
    bits."""
    m = Model(synth.TOY_1L, 3, 4000, seed=4)
    try:
        tokens = synth.make_tokens(3, m.cfg.vocab, seed=41).numpy()
        positions = [3999, 100, 0]
        kv_before = synth.bf16_bits(m.kv)
        got = m.step(tokens, positions)
        ref, _, _ = m.oracle(tokens, positions, kv_before)
        _assert_rows_close(got, ref)
        m.plan.set_debug(force_ctas=5, queue_perm_seed=2)
        np.testing.assert_array_equal(m.step(tokens, positions), got)
        m.plan.set_debug()
        np.testing.assert_array_equal(m.step(tokens, positions, per_op=True, graph=True), got)
    finally:
        m.close()


@pytest.mark.parametrize("pos", [4096, 700, 0])
def test_attention_combine_slices_all_some_and_one_split(pos):
    """The Llama-3-8B head layout (head_dim 128, 4 q heads per kv head, 2
    layers) with a 4097-token cache: the plan combines each group's splits
    in slices (several combine instructions per group, queued after every
    split).  A sequence that uses all 19 splits, 4 of them or 1 matches the
    oracle, and the launch on 7 CTAs with a permuted queue and the
    kernel-per-operator runner give the same bits."""
    cfg = synth.LLAMA3_8B.replace(n_layers=2)
    m = Model(cfg, 1, 4097, seed=9)
    try:
        tokens = synth.make_tokens(1, cfg.vocab, seed=pos).numpy()
        kv_before = synth.bf16_bits(m.kv)
        got = m.step(tokens, [pos])
        ref, _, _ = m.oracle(tokens, [pos], kv_before)
        _assert_rows_close(got, ref)
        # repeating the step rewrites the same cache entries
        m.plan.set_debug(force_ctas=7, queue_perm_seed=3)
        np.testing.assert_array_equal(m.step(tokens, [pos]), got)
        m.plan.set_debug()
        np.testing.assert_array_equal(m.step(tokens, [pos], per_op=True), got)
    finally:
        m.close()


def test_multi_step_greedy_decode():
    """mk_decode_steps: n greedy steps in one launch equal n single steps fed
    the argmax of each step's logits (same tile arithmetic: bit-identical
    logits and cache); each chosen token is a maximum of the oracle's logits
    for that step within the tolerance (teacher-forced with the chosen tokens),
    and the last step's logits match the oracle's."""
    cfg = synth.LLAMA32_1B.replace(n_layers=2)
    n, pos0 = 5, 250
    m = Model(cfg, 1, 300, seed=6)
    try:
        kv0 = m.kv.clone()
        tok0 = synth.make_tokens(1, cfg.vocab, seed=31)
        t = tok0.to(m.dev)
        p = torch.tensor([pos0], dtype=torch.int32, device=m.dev)
        out = torch.full((n,), -1, dtype=torch.int32, device=m.dev)
        lg = torch.full((cfg.vocab,), float("nan"), device=m.dev)
        m.plan.decode_steps(t, p, n, m.kv, out, lg)
        assert m.plan.status() == mk.MK_OK
        chosen = out.cpu().numpy()
        multi_logits = lg.cpu().numpy()
        kv_multi = m.kv.clone()
        # the same steps one launch each, the argmax taken on the host
        m.kv.copy_(kv0)
        tok = int(tok0[0])
        ref_tokens = []
        for s in range(n):
            got = m.step([tok], [pos0 + s])[0]
            tok = int(np.argmax(got))  # first index among equal maxima
            ref_tokens.append(tok)
        np.testing.assert_array_equal(chosen, np.array(ref_tokens, dtype=np.int32))
        np.testing.assert_array_equal(multi_logits, got)
        assert torch.equal(m.kv, kv_multi)
        # oracle, teacher-forced with the chosen tokens, its own cache appends
        kvb = synth.bf16_bits(kv0)
        w = synth.LazyBits(m.w)
        tok = int(tok0[0])
        for s in range(n):
            ref, knew, vnew = oracle.decode_step(cfg, w, [tok], [pos0 + s], kvb)
            row = ref[0]
            rms = np.sqrt((row ** 2).mean())
            assert row[chosen[s]] >= row.max() - 2 * TOL * rms, f"step {s}: token {chosen[s]} is not a maximum"
            kb = torch.from_numpy(np.ascontiguousarray(knew[:, 0])).to(torch.bfloat16).view(torch.int16).numpy()
            vb = torch.from_numpy(np.ascontiguousarray(vnew[:, 0])).to(torch.bfloat16).view(torch.int16).numpy()
            kvb[:, 0, 0, :, pos0 + s, :] = kb.view(kvb.dtype)
            kvb[:, 1, 0, :, pos0 + s, :] = vb.view(kvb.dtype)
            tok = int(chosen[s])
        _assert_rows_close(multi_logits[None, :], ref[None, :])
        # past the end of the cache: latched bounds error, nothing else
        m.plan.reset()
        p2 = torch.tensor([300 - 2], dtype=torch.int32, device=m.dev)
        m.plan.decode_steps(t, p2, 3, m.kv, out, lg)
        assert m.plan.status() == mk.MK_ERR_BOUNDS
        m.plan.reset()
    finally:
        m.close()
