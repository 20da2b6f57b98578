"""Prefill on the GPU (tensor-core tiles with tile-level dependencies) through
the C ABI, against the CPU oracle.

Tolerances (written here): last-token logits per row within
2e-2 * RMS(oracle logits); the K/V the prefill wrote into the cache are bf16
values like the oracle's (which rounds them the same way): float32 rounding
differences move a value across a bf16 rounding boundary now and then (one
spacing, 2^-8..2^-7 relative, more often in later layers), so each element is
within two spacings plus 2e-2 * RMS of the oracle's, and the RMS difference is
below 3e-3 * RMS; prefill(S) followed by decode(1) against the
oracle's prefill(S+1) within 2e-2 * RMS.  Kernel-per-operator prefill is
bit-identical to the persistent one.
"""
import numpy as np
import pytest
import torch

import oracle
from tile_level_overlap_gb300 import build, mk, synth

pytestmark = pytest.mark.gpu

PF_SMALL = synth.ModelCfg(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512,
                          vocab=1024, rms_eps=1e-5, rope_theta=1e4)
PF_D128_QK = synth.ModelCfg(n_layers=2, hidden=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                            ffn=768, vocab=512, rms_eps=1e-6, rope_theta=1e6, qk_norm=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    mk.lib()


def _rows_close(got, ref, tol=2e-2):
    got = np.atleast_2d(np.asarray(got, np.float64))
    ref = np.atleast_2d(np.asarray(ref, np.float64))
    for b in range(ref.shape[0]):
        rms = np.sqrt((ref[b] ** 2).mean())
        err = np.abs(got[b] - ref[b]).max()
        assert err <= tol * rms, f"max |delta| {err:.4e} > {tol} * rms {rms:.4e}"


def _kv_close(name, gpu, orc):
    gpu = np.asarray(gpu, np.float64)
    orc = np.asarray(orc, np.float64)
    rms = np.sqrt((orc ** 2).mean())
    bad = np.abs(gpu - orc) > 2.0 ** -6 * np.abs(orc) + 2e-2 * rms
    assert not bad.any(), f"{name}: {bad.sum()} elements off by more than two bf16 spacings"
    drms = np.sqrt(((gpu - orc) ** 2).mean())
    assert drms <= 3e-3 * rms, f"{name}: rms |delta| {drms:.3e} > 3e-3 * {rms:.3e}"


class PfModel:
    def __init__(self, cfg, max_ctx, seed=0):
        self.cfg = cfg
        self.dev = torch.device("cuda:0")
        self.w = synth.make_weights(cfg, seed=seed, device=self.dev)
        self.kv = torch.zeros(synth.kv_cache_shape(cfg, 1, max_ctx), dtype=torch.bfloat16,
                              device=self.dev)
        self.plan = mk.Plan(cfg, self.w, 1, max_ctx)
        self.max_ctx = max_ctx

    def prefill(self, tokens, per_op=False, graph=False):
        t = torch.as_tensor(tokens, dtype=torch.int32).to(self.dev)
        logits = torch.full((self.cfg.vocab,), float("nan"), device=self.dev)
        if per_op:
            self.plan.run_per_op(mk.MK_PREFILL, t, None, self.kv, logits, use_graph=graph)
        else:
            self.plan.prefill(t, self.kv, logits)
        rc = self.plan.status()
        assert rc == mk.MK_OK, mk.lib().mk_status_string(rc)
        return logits.cpu().numpy()

    def decode(self, token, pos):
        t = torch.tensor([token], dtype=torch.int32, device=self.dev)
        p = torch.tensor([pos], dtype=torch.int32, device=self.dev)
        logits = torch.empty((1, self.cfg.vocab), device=self.dev)
        self.plan.decode_step(t, p, self.kv, logits)
        assert self.plan.status() == mk.MK_OK
        return logits.cpu().numpy()[0]

    def oracle_prefill(self, tokens):
        return oracle.prefill(self.cfg, synth.LazyBits(self.w), np.asarray(tokens))

    def close(self):
        self.plan.close()
        del self.w, self.kv
        torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def small():
    m = PfModel(PF_SMALL, max_ctx=384)
    yield m
    m.close()


@pytest.mark.parametrize("S", [1, 7, 128, 129, 300, 384])
def test_prefill_matches_oracle(small, S):
    tokens = synth.make_tokens(S, small.cfg.vocab, seed=S).numpy()
    got = small.prefill(tokens)
    ref, K, V = small.oracle_prefill(tokens)
    _rows_close(got, ref)
    kv = oracle.widen_bf16(synth.bf16_bits(small.kv))
    for name, gpu, orc in [("K", kv[:, 0, 0, :, :S, :], K), ("V", kv[:, 1, 0, :, :S, :], V)]:
        _kv_close(name, gpu, orc)


def test_prefill_then_decode_matches_longer_prefill(small):
    tokens = synth.make_tokens(201, small.cfg.vocab, seed=11).numpy()
    small.prefill(tokens[:200])
    got = small.decode(int(tokens[200]), 200)
    ref, _, _ = small.oracle_prefill(tokens)
    _rows_close(got, ref)


def test_prefill_per_op_and_graph_bit_identical(small):
    tokens = synth.make_tokens(250, small.cfg.vocab, seed=12).numpy()
    mega = small.prefill(tokens)
    np.testing.assert_array_equal(small.prefill(tokens), mega)
    np.testing.assert_array_equal(small.prefill(tokens, per_op=True), mega)
    np.testing.assert_array_equal(small.prefill(tokens, per_op=True, graph=True), mega)


@pytest.mark.parametrize("S", [5, 256, 333])
def test_prefill_head_dim_128_qk_norm(S):
    m = PfModel(PF_D128_QK, max_ctx=512, seed=4)
    try:
        tokens = synth.make_tokens(S, m.cfg.vocab, seed=S + 1).numpy()
        got = m.prefill(tokens)
        ref, _, _ = m.oracle_prefill(tokens)
        _rows_close(got, ref)
    finally:
        m.close()


def test_llama3_8b_width_prefill_2048_tokens():
    """Full Llama-3-8B widths (hidden 4096, 32/8 heads, head_dim 128, FFN
    14336, vocab 128256) with 2 of the 32 layers, on the 2048-token prompt."""
    cfg = synth.LLAMA3_8B.replace(n_layers=2)
    m = PfModel(cfg, max_ctx=2049, seed=0)
    try:
        tokens = synth.make_tokens(2048, cfg.vocab).numpy()
        got = m.prefill(tokens)
        ref, K, V = m.oracle_prefill(tokens)
        _rows_close(got, ref)
        kv = oracle.widen_bf16(synth.bf16_bits(m.kv))
        _kv_close("K", kv[:, 0, 0, :, :2048, :], K)
        _kv_close("V", kv[:, 1, 0, :, :2048, :], V)
    finally:
        m.close()


def _prefill_logits(m, tokens):
    t = torch.as_tensor(tokens, dtype=torch.int32).to(m.dev)
    logits = torch.full((len(tokens), m.cfg.vocab), float("nan"), device=m.dev)
    m.plan.prefill_logits(t, m.kv, logits)
    rc = m.plan.status()
    assert rc == mk.MK_OK, mk.lib().mk_status_string(rc)
    return logits.cpu().numpy()


@pytest.mark.parametrize("S", [1, 130, 300])
def test_prefill_all_token_logits(small, S):
    """Every row of mk_prefill_logits against the oracle's all-token logits;
    the cache as mk_prefill writes it; repeat runs bit-identical."""
    tokens = synth.make_tokens(S, small.cfg.vocab, seed=S + 40).numpy()
    got = _prefill_logits(small, tokens)
    ref, K, V = oracle.prefill(small.cfg, synth.LazyBits(small.w), tokens, all_logits=True)
    _rows_close(got, ref)
    kv = oracle.widen_bf16(synth.bf16_bits(small.kv))
    _kv_close("K", kv[:, 0, 0, :, :S, :], K)
    _kv_close("V", kv[:, 1, 0, :, :S, :], V)
    np.testing.assert_array_equal(_prefill_logits(small, tokens), got)
    # the last-token entry point still gives its own (CUDA-core) last row
    _rows_close(small.prefill(tokens)[None, :], ref[-1:])


def test_prefill_all_token_logits_ragged_vocab():
    """A vocabulary that is not a multiple of the 256-row LM tile."""
    cfg = PF_SMALL.replace(vocab=1000)
    m = PfModel(cfg, max_ctx=200, seed=2)
    try:
        tokens = synth.make_tokens(150, cfg.vocab, seed=3).numpy()
        got = _prefill_logits(m, tokens)
        ref, _, _ = oracle.prefill(cfg, synth.LazyBits(m.w), tokens, all_logits=True)
        _rows_close(got, ref)
    finally:
        m.close()


def test_llama3_8b_width_prefill_all_token_logits_sampled():
    """Llama-3-8B widths, 2 layers, 2048 tokens: sampled rows of the all-token
    logits against the oracle's last-token logits of the prompt's prefixes
    (row r depends on tokens 0..r only)."""
    cfg = synth.LLAMA3_8B.replace(n_layers=2)
    m = PfModel(cfg, max_ctx=2049, seed=0)
    try:
        tokens = synth.make_tokens(2048, cfg.vocab).numpy()
        got = _prefill_logits(m, tokens)
        for r in [0, 129, 2047]:
            ref, _, _ = oracle.prefill(cfg, synth.LazyBits(m.w), tokens[:r + 1])
            _rows_close(got[r:r + 1], ref[None, :])
    finally:
        m.close()


@pytest.mark.parametrize("max_ctx", [320, 700])
def test_prefill_batch_slots(max_ctx):
    """mk_prefill_batch: three prompts of different lengths into cache slots
    0..2: each slot's keys/values and last-token logits against the oracle,
    then one batched decode step over the three slots against the oracle's
    prefill of each prompt plus the decoded token.  With a 700-token context
    all five 128-token blocks share one launch; with 320 (three blocks per
    launch) the first two prompts share one and the third has its own."""
    cfg = PF_SMALL
    m = PfModel(cfg, max_ctx=max_ctx, seed=8)
    try:
        m.kv = torch.zeros(synth.kv_cache_shape(cfg, 3, max_ctx), dtype=torch.bfloat16, device=m.dev)
        m.plan.close()
        m.plan = mk.Plan(cfg, m.w, 3, max_ctx)
        lens = [200, 7, 129]
        stride = 256
        toks = np.zeros((3, stride), dtype=np.int32)
        seqs = [synth.make_tokens(n, cfg.vocab, seed=50 + b).numpy() for b, n in enumerate(lens)]
        for b, sq in enumerate(seqs):
            toks[b, :len(sq)] = sq
        t = torch.from_numpy(toks).to(m.dev)
        lg = torch.full((3, cfg.vocab), float("nan"), device=m.dev)
        m.plan.prefill_batch(t, lens, m.kv, lg)
        assert m.plan.status() == mk.MK_OK
        got = lg.cpu().numpy()
        kv = oracle.widen_bf16(synth.bf16_bits(m.kv))
        for b, sq in enumerate(seqs):
            ref, K, V = oracle.prefill(cfg, synth.LazyBits(m.w), sq)
            _rows_close(got[b:b + 1], ref[None, :])
            _kv_close(f"K{b}", kv[:, 0, b, :, :lens[b], :], K)
            _kv_close(f"V{b}", kv[:, 1, b, :, :lens[b], :], V)
        nxt = synth.make_tokens(3, cfg.vocab, seed=60).numpy()
        dl = torch.empty((3, cfg.vocab), device=m.dev)
        m.plan.decode_step(torch.from_numpy(nxt.astype(np.int32)).to(m.dev),
                           torch.tensor(lens, dtype=torch.int32, device=m.dev), m.kv, dl)
        assert m.plan.status() == mk.MK_OK
        dec = dl.cpu().numpy()
        for b, sq in enumerate(seqs):
            ref, _, _ = oracle.prefill(cfg, synth.LazyBits(m.w), np.concatenate([sq, nxt[b:b + 1]]))
            _rows_close(dec[b:b + 1], ref[None, :])
        with pytest.raises(mk.MkError):
            m.plan.prefill_batch(t, [200, 0, 5], m.kv, lg)
    finally:
        m.close()


def test_prefill_batch_bit_identical_to_single_prompts():
    """One launch over three prompts (their blocks end to end in the
    activation planes) computes every row as the prompt's own launch does:
    logits and cache entries bit-identical to three one-prompt calls (head_dim
    128 with q/k norm)."""
    cfg = PF_D128_QK
    dev = torch.device("cuda:0")
    w = synth.make_weights(cfg, seed=9, device=dev)
    plan = mk.Plan(cfg, w, 3, 700)
    try:
        lens = [300, 5, 256]
        stride = 320
        toks = np.zeros((3, stride), dtype=np.int32)
        seqs = [synth.make_tokens(n, cfg.vocab, seed=70 + b).numpy() for b, n in enumerate(lens)]
        for b, sq in enumerate(seqs):
            toks[b, :len(sq)] = sq
        kv = torch.zeros(synth.kv_cache_shape(cfg, 3, 700), dtype=torch.bfloat16, device=dev)
        lg = torch.full((3, cfg.vocab), float("nan"), device=dev)
        plan.prefill_batch(torch.from_numpy(toks).to(dev), lens, kv, lg)
        assert plan.status() == mk.MK_OK
        got = lg.cpu().numpy()
        for b, sq in enumerate(seqs):
            kv1 = torch.zeros_like(kv)
            lg1 = torch.full((1, cfg.vocab), float("nan"), device=dev)
            one = np.zeros((1, stride), dtype=np.int32)
            one[0, :len(sq)] = sq
            plan.prefill_batch(torch.from_numpy(one).to(dev), [lens[b]], kv1, lg1)
            assert plan.status() == mk.MK_OK
            np.testing.assert_array_equal(got[b], lg1.cpu().numpy()[0])
            assert torch.equal(kv[:, :, b, :, :lens[b]], kv1[:, :, 0, :, :lens[b]])
    finally:
        plan.close()
        del w
        torch.cuda.empty_cache()


@pytest.mark.parametrize("max_ctx", [320, 512])
def test_prefill_chunks_mixed_with_decode(max_ctx):
    """mk_prefill_chunks: the tensor-core prefill kernel running a prompt
    continuation and decode tokens together -- 130 tokens of slot 0 at cache
    positions 150..279 (not aligned to 128 positions, crossing a key-block
    boundary) and one decode token each for slots 1 and 2 -- after the three
    prompts were prefilled.  Each chunk's last logits against the oracle's
    prefill of the whole sequence; the cache entries the chunks wrote against
    the oracle's keys and values.  With a 512-token context all four 128-token
    blocks share one launch; with 320 the packing needs two."""
    cfg = PF_SMALL
    dev = torch.device("cuda:0")
    w = synth.make_weights(cfg, seed=12, device=dev)
    plan = mk.Plan(cfg, w, 3, max_ctx)
    try:
        kv = torch.zeros(synth.kv_cache_shape(cfg, 3, max_ctx), dtype=torch.bfloat16, device=dev)
        lens = [150, 40, 90]
        stride = 160
        prompts = [synth.make_tokens(n, cfg.vocab, seed=80 + b).numpy() for b, n in enumerate(lens)]
        toks = np.zeros((3, stride), dtype=np.int32)
        for b, sq in enumerate(prompts):
            toks[b, :len(sq)] = sq
        lg = torch.empty((3, cfg.vocab), device=dev)
        plan.prefill_batch(torch.from_numpy(toks).to(dev), lens, kv, lg)
        assert plan.status() == mk.MK_OK
        cont = synth.make_tokens(130, cfg.vocab, seed=90).numpy()
        dec = synth.make_tokens(2, cfg.vocab, seed=91).numpy()
        ctoks = np.concatenate([cont, dec]).astype(np.int32)
        chunks = [(0, 150, 130, 0), (1, 40, 1, 130), (2, 90, 1, 131)]
        clg = torch.full((3, cfg.vocab), float("nan"), device=dev)
        plan.prefill_chunks(torch.from_numpy(ctoks).to(dev), chunks, kv, clg)
        assert plan.status() == mk.MK_OK
        got = clg.cpu().numpy()
        cache = oracle.widen_bf16(synth.bf16_bits(kv))
        seqs = [np.concatenate([prompts[0], cont]), np.concatenate([prompts[1], dec[:1]]),
                np.concatenate([prompts[2], dec[1:]])]
        for b, sq in enumerate(seqs):
            ref, K, V = oracle.prefill(cfg, synth.LazyBits(w), sq)
            _rows_close(got[b:b + 1], ref[None, :])
            p0, n = chunks[b][1], chunks[b][2]
            _kv_close(f"K{b}", cache[:, 0, b, :, p0:p0 + n, :], K[:, :, p0:p0 + n, :])
            _kv_close(f"V{b}", cache[:, 1, b, :, p0:p0 + n, :], V[:, :, p0:p0 + n, :])
        # a chunk that does not continue its slot's previous chunk is refused
        with pytest.raises(mk.MkError):
            plan.prefill_chunks(torch.from_numpy(ctoks).to(dev), [(0, 10, 5, 0), (0, 20, 5, 5)], kv, clg)
    finally:
        plan.close()
        del w
        torch.cuda.empty_cache()


def test_prefill_chunks_rejects_bad_chunks():
    """Chunks outside the plan are refused before any device work: a slot
    past max_batch, a negative first position, an empty chunk, a chunk past
    the context, a negative token offset."""
    cfg = PF_SMALL
    dev = torch.device("cuda:0")
    w = synth.make_weights(cfg, seed=12, device=dev)
    plan = mk.Plan(cfg, w, 2, 300)
    try:
        kv = torch.zeros(synth.kv_cache_shape(cfg, 2, 300), dtype=torch.bfloat16, device=dev)
        toks = torch.zeros(64, dtype=torch.int32, device=dev)
        lg = torch.empty((1, cfg.vocab), device=dev)
        for bad in [(2, 0, 4, 0), (0, -1, 4, 0), (0, 0, 0, 0), (0, 290, 20, 0), (0, 0, 4, -1)]:
            with pytest.raises(mk.MkError):
                plan.prefill_chunks(toks, [bad], kv, lg)
        assert plan.status() == mk.MK_OK
    finally:
        plan.close()
        del w
        torch.cuda.empty_cache()
