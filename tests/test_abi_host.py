"""The C ABI library loads, exports every symbol include/mk.h declares, and its
host-only plan builder produces queues that a sequential barrier simulator
accepts.  No GPU needed (no compute calls)."""
import ctypes
import os
import re

import pytest
import torch

from tile_level_overlap_gb300 import build, mk, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mk.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mk.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mk.EXPORTED)


def test_status_strings(lib):
    for code in range(7):
        assert lib.mk_status_string(code)
    assert lib.mk_status_string(0) == b"ok"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_device_reports_no_device(lib):
    cfg = mk.model_cfg(synth.TOY_1L)
    w = mk.mk_weight_ptrs()
    h = ctypes.c_void_p()
    assert lib.mk_plan_create(ctypes.byref(cfg), ctypes.byref(w), 1, 16, ctypes.byref(h)) in (
        mk.MK_ERR_NO_DEVICE, mk.MK_ERR_INVALID_ARG)


def _expected_weight_bytes(c):
    qkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim * c.hidden
    o = c.hidden * c.n_q_heads * c.head_dim
    ffn = 3 * c.ffn * c.hidden
    return 2 * (c.n_layers * (qkv + o + ffn) + c.vocab * c.hidden)


def _keys_per_split(head_dim):
    # the model constant of the decode attention tiling (mk_plan.h)
    return 216 if head_dim >= 128 else 64


def _combine_instructions(ns, rep, head_dim):
    # extra combine instructions per (sequence, kv head) group (mk_plan.h): one
    # slice per 20 KB of partial words at max_ctx, at most 8; with one slice
    # the group's last split combines instead (no extra instruction)
    if ns <= 1:
        return 0
    n = min(8, max(1, ns * rep * head_dim * 8 // 20480))
    return n if n > 1 else 0


@pytest.mark.parametrize("cfg,mb,mc", [
    (synth.TOY_1L, 1, 129), (synth.TOY_1L, 8, 129), (synth.TOY_1L, 3, 17),
    (synth.LLAMA32_1B, 1, 1025), (synth.LLAMA3_8B, 1, 4097),
    (synth.TOY_1L.replace(qk_norm=True), 2, 64),
])
def test_plan_check_valid(lib, cfg, mb, mc):
    rc, st = mk.plan_check(cfg, mb, mc)
    assert rc == mk.MK_OK
    assert st.weight_bytes == _expected_weight_bytes(cfg)
    ns = -(-mc // _keys_per_split(cfg.head_dim))
    assert st.n_splits == ns
    # per layer: QKV, the attention splits, the combining splits (when a group
    # has more than one split), O, gate/up, down; then the LM head
    assert st.n_launches_per_op_decode == (5 + (ns > 1)) * cfg.n_layers + 1


@pytest.mark.parametrize("cfg,mc", [(synth.TOY_1L, 129), (synth.LLAMA32_1B, 1025),
                                    (synth.LLAMA3_8B, 4097), (synth.TOY_1L, 2000),
                                    (synth.TOY_1L, 4000)])
def test_split_tiling_independent_of_max_batch(lib, cfg, mc):
    """The split-KV tiling is fixed keys per split (a model constant): the
    split count is ceil(max_ctx / KPS) whatever max_batch is, and only the
    attention part of the queue grows with max_batch (one set of splits, and
    of combine slices when there are several splits, per sequence slot)."""
    kps = _keys_per_split(cfg.head_dim)
    counts = {}
    for mb in (1, 2, 3):
        if mb * max(cfg.hidden, cfg.ffn) > 6144 and mb > 1:
            continue  # beyond the CUDA-core path's shared-memory activation buffer
        rc, st = mk.plan_check(cfg, mb, mc)
        assert rc == mk.MK_OK
        assert st.n_splits == -(-mc // kps)
        counts[mb] = st.n_instr_decode
    for mb in counts:
        if mb > 1:
            ns = -(-mc // kps)
            rep = cfg.n_q_heads // cfg.n_kv_heads
            per_slot = cfg.n_layers * cfg.n_kv_heads * (ns + _combine_instructions(ns, rep, cfg.head_dim))
            assert counts[mb] - counts[1] == (mb - 1) * per_slot


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5])
def test_plan_check_random_topological_orders(lib, seed):
    rc, _ = mk.plan_check(synth.LLAMA32_1B.replace(n_layers=3), 1, 1025, seed=seed)
    assert rc == mk.MK_OK
    rc, _ = mk.plan_check(synth.TOY_1L, 4, 65, seed=seed)
    assert rc == mk.MK_OK
    # a cache long enough for the combine in slices (63 splits, 3 slices)
    rc, _ = mk.plan_check(synth.TOY_1L, 3, 4000, seed=seed)
    assert rc == mk.MK_OK


@pytest.mark.parametrize("cfg,mb,mc", [
    (synth.LLAMA3_8B.replace(n_layers=2), 8, 4097),
    (synth.QWEN3_8B.replace(n_layers=2), 32, 2049),
    (synth.ModelCfg(n_layers=2, hidden=2048, n_q_heads=16, n_kv_heads=4, head_dim=128, ffn=3072,
                    vocab=1000, rms_eps=1e-5, rope_theta=1e4), 12, 300),
    (synth.ModelCfg(n_layers=2, hidden=512, n_q_heads=8, n_kv_heads=8, head_dim=64, ffn=768,
                    vocab=1000, rms_eps=1e-5, rope_theta=1e4), 20, 200),
])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_batched_plan_check_random_orders(lib, cfg, mb, mc, seed):
    """The tensor-core batched-decode queue and random topological orders of
    it pass the host simulator: every wait (including the O chunks' waits on
    their kv groups and the down chunks' waits on their gate/up row tiles) is
    met when reached, and every barrier ends with exactly the releases its
    waiters expect."""
    rc, st = mk.plan_check(cfg, mb, mc, seed=seed)
    assert rc == mk.MK_OK
    assert st.decode_path == 1


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), mk.MK_ERR_UNSUPPORTED),
    (dict(n_q_heads=5), mk.MK_ERR_INVALID_ARG),
    (dict(n_q_heads=6), mk.MK_ERR_UNSUPPORTED),
    (dict(n_q_heads=48, n_kv_heads=2), mk.MK_ERR_UNSUPPORTED),
    (dict(n_layers=0), mk.MK_ERR_INVALID_ARG),
    (dict(hidden=260), mk.MK_ERR_UNSUPPORTED),
])
def test_plan_check_rejects(lib, bad, code):
    rc, _ = mk.plan_check(synth.TOY_1L.replace(**bad), 1, 64)
    assert rc == code


def test_plan_check_rejects_sizes(lib):
    assert mk.plan_check(synth.TOY_1L, 0, 64)[0] == mk.MK_ERR_INVALID_ARG
    assert mk.plan_check(synth.TOY_1L, 1, 0)[0] == mk.MK_ERR_INVALID_ARG
    assert mk.plan_check(synth.TOY_1L, 64, 64)[0] == mk.MK_ERR_UNSUPPORTED
