#!/usr/bin/env python3
"""Decode benchmark: Llama-3-8B-shape decode step, batch 1, context 4096.

One step = one whole decode step of the model (32 layers + LM head) for one
new token, run as one persistent kernel launch through the C ABI.  Prints one
JSON line (rank 0): tokens/s of the persistent step, its HBM bytes per second
against the measured copy bandwidth (algorithmic bytes: every weight once plus
the cached and new K/V), and the comparison legs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama3-8b|llama3.2-1b] [--no-per-op] [--no-prefill]
                  [--no-cpu-baseline]

--workload llama3.2-1b (Llama-3.2-1B shape, context 1024) is a smaller case of
the same step for profiling; the default is the headline workload.

--impl reference times the CPU oracle (plain NumPy forward pass) on the host
cores: one whole decode step of the same workload per step (--ref-layers N
times N layers + the LM head instead, scaled to the full layer count).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and HBM GB/s (% of ~8 TB/s), Llama-3-8B shape, batch 1, 1xGB300"
UNIT = "tokens/s"
PREFILL_TOKENS = 2048
MULTI_STEPS = 8  # tokens per launch of the multi-step greedy decode leg
DEP_WAIT_STEPS = 5  # traced steps the dependency-wait share is averaged over
BATCHED_LEGS = ("llama3-8b-b8", "qwen3-8b-b32")
BATCH_PREFILL_PROMPTS, BATCH_PREFILL_TOKENS = 4, 512  # the several-prompt prefill leg
# name -> (shape in synth, batch, largest cached context, smallest (ragged
# contexts U[lo, ctx], seeded) or None (all at ctx), metric, description,
# traffic key)
WORKLOADS = {
    "llama3-8b": ("LLAMA3_8B", 1, 4096, None, METRIC,
                  "Llama-3-8B-shape decode, batch 1, context 4096", "llama3-8b-decode-b1-ctx4096"),
    "llama3.2-1b": ("LLAMA32_1B", 1, 1024, None,
                    "decode tokens/s and HBM GB/s, Llama-3.2-1B shape, batch 1, 1xGB300",
                    "Llama-3.2-1B-shape decode, batch 1, context 1024",
                    "llama3.2-1b-decode-b1-ctx1024"),
    "llama3-8b-b8": ("LLAMA3_8B", 8, 4096, None,
                     "decode tokens/s and HBM GB/s, Llama-3-8B shape, batch 8, 1xGB300",
                     "Llama-3-8B-shape decode, batch 8, context 4096 each",
                     "llama3-8b-decode-b8-ctx4096"),
    "qwen3-8b-b32": ("QWEN3_8B", 32, 2048, 512,
                     "decode tokens/s and HBM GB/s, Qwen3-8B shape, batch 32, 1xGB300",
                     "Qwen3-8B-shape decode, batch 32, contexts U[512, 2048] (seeded)",
                     "qwen3-8b-decode-b32-ragged"),
}


def workload(name):
    """(model shape, batch, positions [batch], metric, description, traffic key)."""
    from tile_level_overlap_gb300 import synth
    shape, batch, ctx, lo, metric, desc, key = WORKLOADS[name]
    if lo is None:
        positions = [ctx] * batch
    else:
        positions = [int(v) for v in synth.make_contexts(batch, lo, ctx)]
    return getattr(synth, shape), batch, positions, metric, desc, key


def algorithmic_bytes(cfg, batch, positions) -> int:
    """Bytes one decode step must move at minimum: every weight once, the
    cached K/V of every sequence once, the new K/V written; activations are
    negligible (< 1 MB) and left out."""
    H, d, F = cfg.hidden, cfg.head_dim, cfg.ffn
    qd = cfg.n_q_heads * d
    per_layer = (cfg.n_q_heads + 2 * cfg.n_kv_heads) * d * H + H * qd + 3 * F * H
    weights = 2 * (cfg.n_layers * per_layer + cfg.vocab * H)
    kv_read = sum(2 * cfg.n_layers * cfg.n_kv_heads * int(p) * d * 2 for p in positions)
    kv_write = batch * 2 * cfg.n_layers * cfg.n_kv_heads * d * 2
    return weights + kv_read + kv_write


def prefill_flops(cfg, S) -> float:
    """Algorithmic FLOPs of a causal prefill of S tokens: every projection
    (2 * S * params per layer) plus causal attention (QK^T and PV over the
    S(S+1)/2 visible pairs per head), plus the last token's LM head."""
    H, d, F = cfg.hidden, cfg.head_dim, cfg.ffn
    qd = cfg.n_q_heads * d
    per_layer_params = (cfg.n_q_heads + 2 * cfg.n_kv_heads) * d * H + H * qd + 3 * F * H
    gemm = 2.0 * S * per_layer_params * cfg.n_layers
    attn = 2.0 * 2.0 * qd * (S * (S + 1) / 2.0) * cfg.n_layers
    return gemm + attn + 2.0 * cfg.vocab * H


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Sources that make up each profiled kernel: a recorded traffic figure stands
# only while none of them has changed.
KERNEL_SOURCES = {
    "mk_interpreter": ("mk_kernel.cuh", "mk_device.cuh", "mk_internal.h", "mk_plan.h", "mk_plan.cpp",
                       "mk_variants.h", "mk_k_generic.cu", "mk_k_h1_f4_d64_r4.cu",
                       "mk_k_h2_f7_d128_r4.cu", "mk_k_h2_f6_d128_r4.cu"),
    "mk_bdecode_kernel": ("mk_bdecode_kernel.cu", "mk_bdecode.h", "mk_bdecode_plan.cpp", "mk_device.cuh",
                          "mk_internal.h", "mk_tc.cuh", "mk_plan.h"),
}


def source_hash(kernel: str = "mk_interpreter") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tile_level_overlap_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != source_hash(kernel):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
                if out.returncode == 0 and out.stdout.strip():
                    self.rows.append([s.strip() for s in out.stdout.strip().split(",")])
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        import statistics
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """Max of a host float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Whole-job rate: units every rank processed / the slowest rank's time
    (replicas: every rank runs the same per-rank work)."""
    return world * units_per_rank / seconds_max


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm: the oracle
class OracleSample:
    """The CPU oracle on the decode step: `n_layers_sample` layers + the LM
    head per step (0 or the model's depth = the whole model, no scaling).
    Weights are the caller's tensors copied to the host, else drawn with the
    same recipe (on the GPU when one is present, for speed)."""

    def __init__(self, cfg, n_layers_sample: int, positions, weights=None, seed: int = 0):
        import torch

        from tile_level_overlap_gb300 import synth

        torch.set_num_threads(cpu_cores())
        self.cfg = cfg
        self.n = cfg.n_layers if n_layers_sample <= 0 else min(n_layers_sample, cfg.n_layers)
        self.sub = cfg.replace(n_layers=self.n)
        if weights is None:
            dev = "cuda" if torch.cuda.is_available() else "cpu"
            weights = synth.make_weights(self.sub, seed=seed, device=dev)
        names = synth.weight_shapes(self.sub)
        self.w = {k: synth.bf16_bits(weights[k]) for k in names}
        self.positions = list(positions)
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        self.kv = synth.bf16_bits(synth.make_kv_cache(self.sub, len(self.positions),
                                                      max(self.positions) + 1, device=dev))
        self.tok = synth.make_tokens(len(self.positions), cfg.vocab).numpy()

    def describe(self, wl_desc: str, batch: int) -> str:
        if self.n == self.cfg.n_layers:
            return (f"one whole batch-{batch} decode step ({wl_desc}): all {self.cfg.n_layers} layers "
                    f"+ the LM head, per step")
        return (f"{self.n} of {self.cfg.n_layers} layers + the LM head of one batch-{batch} decode step "
                f"({wl_desc}), per step; time scaled to {self.cfg.n_layers} layers")

    def step(self):
        """Returns (seconds for the whole model, seconds measured)."""
        import numpy as np

        import oracle
        from oracle import model as om

        t0 = time.perf_counter()
        oracle.decode_step(self.sub, self.w, self.tok, self.positions, self.kv)
        t_all = time.perf_counter() - t0
        if self.n == self.cfg.n_layers:
            return t_all, t_all
        # the LM head alone, so that only the layer part is scaled
        x = np.random.default_rng(0).normal(size=(len(self.positions), self.cfg.hidden)).astype(np.float32)
        t1 = time.perf_counter()
        lm = self.w["embed"] if self.cfg.tied_embeddings else self.w["lm_head"]
        om.linear(lm, om.rmsnorm(x, self.w["final_norm"], self.cfg.rms_eps))
        t_lm = time.perf_counter() - t1
        t_layers = max(t_all - t_lm, 1e-9)
        return t_layers * self.cfg.n_layers / self.n + t_lm, t_all


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cfg, batch, positions, metric, wl_desc, _ = workload(args.workload)
    sample_run = OracleSample(cfg, args.ref_layers, positions)
    for _ in range(args.warmup):
        sample_run.step()
    times, measured = [], 0.0
    for _ in range(args.steps):
        t, tm = sample_run.step()
        times.append(t)
        measured += tm
    ms = 1e3 * sum(times) / len(times)
    value = batch / (ms / 1e3)
    line = {
        "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": {"workload": wl_desc,
                   "weights": "bf16", "kv_cache": "bf16"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample_run.describe(wl_desc, batch)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    from tile_level_overlap_gb300 import mk, synth

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    cfg, BATCH, pos_list, metric, wl_desc, traffic_key = workload(args.workload)
    CONTEXT = max(pos_list)
    max_ctx = CONTEXT + 1
    w = synth.make_weights(cfg, seed=synth.SEED_WEIGHTS + rank, device=dev)
    kv = synth.make_kv_cache(cfg, BATCH, max_ctx, device=dev)
    plan = mk.Plan(cfg, w, BATCH, max_ctx)
    tokens = synth.make_tokens(BATCH, cfg.vocab).to(dev)
    positions = torch.tensor(pos_list, dtype=torch.int32, device=dev)
    logits = torch.empty((BATCH, cfg.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    nbytes = algorithmic_bytes(cfg, BATCH, positions.tolist())

    def barrier():
        torch.cuda.synchronize(dev)
        if pg:
            pg.barrier()

    def timed(fn, steps, per_step=None):
        """Total ms of `steps` calls (max over ranks), one CUDA event pair per
        step on the launching stream; per-step ms into `per_step` if given."""
        barrier()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for i in range(steps):
                fn()
                evs[i + 1].record(stream)
        barrier()
        if per_step is not None:
            per_step.extend(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
        return max_over_ranks(evs[0].elapsed_time(evs[-1]), pg, dev)

    def mega():
        plan.decode_step(tokens, positions, kv, logits, stream=stream)

    def perop():
        plan.run_per_op(mk.MK_DECODE, tokens, positions, kv, logits, use_graph=False, stream=stream)

    def perop_graph():
        plan.run_per_op(mk.MK_DECODE, tokens, positions, kv, logits, use_graph=True, stream=stream)

    for _ in range(args.warmup):
        mega()
    rc = plan.status(stream)
    if rc != mk.MK_OK:
        raise RuntimeError(f"device status {rc}")

    step_ms = []
    with ClockSampler(local) as clk:
        ms_total = timed(mega, args.steps, step_ms)
    rc = plan.status(stream)
    if rc != mk.MK_OK:
        raise RuntimeError(f"device status {rc}")
    ms = ms_total / args.steps
    value = job_throughput(BATCH * args.steps, world, ms_total / 1e3)

    # the same tile routines, kernel-per-operator (eager and CUDA graph)
    per_op = None
    if not args.no_per_op:
        for _ in range(max(1, args.warmup // 2)):
            perop()
            perop_graph()
        ms_perop = timed(perop, args.steps) / args.steps
        ms_graph = timed(perop_graph, args.steps) / args.steps
        per_op = {"ms_per_step_eager": ms_perop, "ms_per_step_graph": ms_graph,
                  "tokens_per_s_eager": BATCH / (ms_perop / 1e3),
                  "tokens_per_s_graph": BATCH / (ms_graph / 1e3),
                  "launches_per_step": plan.stats().n_launches_per_op_decode,
                  "speedup_persistent_vs_graph": ms_graph / ms}
        # mixed composition: persistent layers, then the LM head as its own
        # kernel-per-operator launch ("One Megakernel is Not Enough")
        plan.set_lm_mode(mk.MK_LM_SEPARATE)
        for _ in range(max(1, args.warmup // 2)):
            mega()
        ms_mixed = timed(mega, args.steps) / args.steps
        plan.set_lm_mode(mk.MK_LM_FUSED)
        rc = plan.status(stream)
        if rc != mk.MK_OK:
            raise RuntimeError(f"device status {rc}")
        per_op["ms_per_step_lm_separate"] = ms_mixed
        per_op["speedup_fused_vs_lm_separate"] = ms_mixed / ms

    # end to end through the host-buffer entry point: pinned host tokens and
    # positions in, logits out, every step
    th = tokens.cpu().pin_memory()
    ph = positions.cpu().pin_memory()
    lh = torch.empty((BATCH, cfg.vocab), dtype=torch.float32).pin_memory()
    for _ in range(2):
        plan.decode_step_host(th, ph, kv, lh, stream=stream)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rc = plan.decode_step_host(th, ph, kv, lh, stream=stream)
        if rc != mk.MK_OK:
            raise RuntimeError(f"device status {rc}")
    e2e_s = max_over_ranks(time.perf_counter() - t0, pg, dev)
    e2e = job_throughput(BATCH * args.steps, world, e2e_s)

    # dependency-wait share from traced steps (not timed; the CUDA-core
    # batch-1 path records the trace): per step, the time consumers spent from
    # taking an instruction until its inputs were ready, over CTAs x span
    dep_wait = None
    if BATCH == 1:
        plan.set_debug(trace=True)
        fr = []
        for _ in range(DEP_WAIT_STEPS):
            mega()
            torch.cuda.synchronize(dev)
            rec = plan.trace().astype(np.int64)
            span = rec[:, 3].max() - rec[:, 1].min()
            n_ctas = plan.stats().n_ctas
            if span > 0:
                fr.append(float((rec[:, 2] - rec[:, 1]).sum()) / float(n_ctas * span))
        plan.set_debug(trace=False)
        if fr:
            dep_wait = {"mean": float(np.mean(fr)), "min": float(np.min(fr)),
                        "max": float(np.max(fr)), "steps": len(fr)}

    # greedy decode of MULTI_STEPS tokens per launch (mk_decode_steps, batch
    # 1): positions CONTEXT - MULTI_STEPS .. CONTEXT - 1 so the steps fit the
    # cache; tokens chosen on the device, the host out of the loop
    multi = None
    if BATCH == 1 and CONTEXT > MULTI_STEPS:
        p0 = torch.tensor([CONTEXT - MULTI_STEPS], dtype=torch.int32, device=dev)
        out_tok = torch.empty(MULTI_STEPS, dtype=torch.int32, device=dev)
        lg1 = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)

        def multi_step():
            plan.decode_steps(tokens, p0, MULTI_STEPS, kv, out_tok, lg1, stream=stream)

        try:
            multi_step()
        except mk.MkError as e:
            if e.code != mk.MK_ERR_UNSUPPORTED:
                raise
        else:
            for _ in range(max(1, args.warmup // 2)):
                multi_step()
            launches = max(1, args.steps // MULTI_STEPS)
            ms_launch = timed(multi_step, launches) / launches
            rc = plan.status(stream)
            if rc != mk.MK_OK:
                raise RuntimeError(f"device status {rc}")
            multi = {"steps_per_launch": MULTI_STEPS, "launches": launches,
                     "ms_per_token": ms_launch / MULTI_STEPS,
                     "tokens_per_s": MULTI_STEPS / (ms_launch / 1e3),
                     "positions": [CONTEXT - MULTI_STEPS, CONTEXT - 1]}

    # chunked prefill mixed with decode (tensor-core batched plans): the last
    # half of the columns become a prompt chunk of one slot (consecutive
    # positions before that slot's context), the rest decode as before
    mixed = None
    if plan.stats().decode_path == 1 and BATCH >= 4:
        half = BATCH // 2
        cslot = BATCH - 1
        cpos = pos_list[cslot] - half
        slots_m = torch.tensor(list(range(BATCH - half)) + [cslot] * half, dtype=torch.int32, device=dev)
        pos_m = torch.tensor(pos_list[:BATCH - half] + [cpos + i for i in range(half)],
                             dtype=torch.int32, device=dev)

        def mixed_step():
            plan.decode_step_slots(tokens, pos_m, slots_m, kv, logits, stream=stream)

        for _ in range(max(1, args.warmup // 2)):
            mixed_step()
        ms_mixed = timed(mixed_step, args.steps) / args.steps
        rc = plan.status(stream)
        if rc != mk.MK_OK:
            raise RuntimeError(f"device status {rc}")
        mixed = {"decode_columns": BATCH - half, "chunk_tokens": half, "ms_per_step": ms_mixed,
                 "tokens_per_s": BATCH / (ms_mixed / 1e3)}

    # prefill of a 2048-token prompt into sequence slot 0 (after the decode
    # timing, since it rewrites that cache slot)
    prefill = None
    if not args.no_prefill:
        S = min(PREFILL_TOKENS, CONTEXT)  # the prompt must fit the cache
        ptok = synth.make_tokens(S, cfg.vocab, seed=synth.SEED_TOKENS + 7).to(dev)
        plog = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)

        def pf():
            plan.prefill(ptok, kv, plog, stream=stream)

        for _ in range(2):
            pf()
        rc = plan.status(stream)
        if rc != mk.MK_OK:
            raise RuntimeError(f"prefill device status {rc}")
        pf_steps = max(3, args.steps // 10)
        ms_pf = timed(pf, pf_steps) / pf_steps
        flops = prefill_flops(cfg, S)
        peaks_p, kind_p = measured_peaks()
        tf = flops / (ms_pf / 1e3) / 1e12
        prefill = {"tokens": S, "ms": ms_pf, "tokens_per_s": S / (ms_pf / 1e3),
                   "tflops": tf, "peak_tflops": peaks_p["bf16_tflops_sustained"],
                   "frac_of_tensor_peak": tf / peaks_p["bf16_tflops_sustained"],
                   "peak_kind": kind_p + " (sustained bf16)", "steps": pf_steps,
                   "kernels_per_step": 2}
        # the same prompt with the logits of every token (final norm and LM
        # head as tensor-core tiles inside the one persistent launch)
        pall = torch.empty((S, cfg.vocab), dtype=torch.float32, device=dev)

        def pf_all():
            plan.prefill_logits(ptok, kv, pall, stream=stream)

        pf_all()
        rc = plan.status(stream)
        if rc != mk.MK_OK:
            raise RuntimeError(f"prefill device status {rc}")
        ms_all = timed(pf_all, pf_steps) / pf_steps
        flops_all = flops + 2.0 * (S - 1) * cfg.vocab * cfg.hidden
        tf_all = flops_all / (ms_all / 1e3) / 1e12
        prefill["all_token_logits"] = {
            "ms": ms_all, "tokens_per_s": S / (ms_all / 1e3), "tflops": tf_all,
            "frac_of_tensor_peak": tf_all / peaks_p["bf16_tflops_sustained"], "kernels_per_step": 1}
        del pall

    # batched decode on the tensor-core path (the Llama-3-8B batch-8 and
    # Qwen3-8B batch-32 ragged workloads), each with its own roofline
    batched = None
    decode_path = plan.stats().decode_path
    if not args.no_batched and world == 1:
        plan.close()
        del w, kv
        torch.cuda.empty_cache()
        batched = {name: batched_leg(name, dev, stream, timed, args)
                   for name in BATCHED_LEGS if not args.batched_leg or name in args.batched_leg}

    if rank != 0:
        return 0
    peaks, kind = measured_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    traffic = recorded_traffic("mk_interpreter", traffic_key) if decode_path == 0 else None
    line = {
        "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "ms_per_step_stats": step_stats(step_ms),
        "config": {"workload": wl_desc,
                   "layers": cfg.n_layers, "hidden": cfg.hidden, "ffn": cfg.ffn,
                   "q_heads": cfg.n_q_heads, "kv_heads": cfg.n_kv_heads,
                   "head_dim": cfg.head_dim, "vocab": cfg.vocab, "batch": BATCH,
                   "context": CONTEXT if BATCH == 1 else pos_list,
                   "path": "tensor-core persistent" if decode_path == 1
                           else "cuda-core persistent",
                   "weights": "bf16", "kv_cache": "bf16",
                   "activations": "f32",
                   "l2": f"inputs larger than L2: {nbytes / 1e9:.2f} GB streamed per step",
                   "parallelism": "replicas" if world > 1 else "single"},
        "hbm_gbs": achieved,
        "hbm_frac_of_8tbs": achieved / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_kind": kind,
                     "kernel": "mk_bdecode_kernel" if decode_path == 1 else "mk_interpreter",
                     "algorithmic_bytes_per_launch": nbytes},
        "per_op": per_op,
        "dep_wait_fraction": dep_wait,
        "clocks": clk.summary(),
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": 8 * BATCH,
                "d2h_bytes_per_step": 4 * BATCH * cfg.vocab + 4},
        "gpu_launches": args.steps,
        "prefill": prefill,
        "multi_step": multi,
        "mixed_chunk": mixed,
        "batched": batched,
    }
    if world == 1 and not args.no_cpu_baseline:
        # the oracle as it stands on the host cores: the whole decode step of
        # the same workload (same weights, copied to the host), median of 3
        sample_run = OracleSample(cfg, args.ref_layers, pos_list,
                                  weights=None if batched is not None else w)
        sample_run.step()
        t = sorted(sample_run.step()[0] for _ in range(3))[1]
        line["cpu_baseline"] = {
            "value": BATCH / t, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": sample_run.describe(wl_desc, BATCH) + " (median of 3)"}
    print(json.dumps(line), flush=True)
    if batched is None:
        plan.close()
    if pg:
        pg.destroy_process_group()
    return 0


def step_stats(ms_list):
    """Median, p10, p90 and mean of per-step times (ms)."""
    import numpy as np
    a = np.asarray(ms_list, dtype=np.float64)
    if a.size == 0:
        return None
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "mean": float(a.mean()), "n": int(a.size)}


def batched_leg(name, dev, stream, timed, args):
    """One batched-decode workload: the persistent step (per-step times and
    roofline), the same tile routines kernel-per-operator in a CUDA graph, and
    a prompt chunk mixed with decode columns."""
    import torch

    from tile_level_overlap_gb300 import mk, synth

    cfg, batch, pos_list, metric, desc, _ = workload(name)
    if args.batched_layers:
        # profiling case only: the same step on fewer layers
        cfg = cfg.replace(n_layers=args.batched_layers)
        desc = f"{desc}, first {args.batched_layers} layers (profiling case)"
    max_ctx = max(pos_list) + 1
    w = synth.make_weights(cfg, device=dev)
    kv = synth.make_kv_cache(cfg, batch, max_ctx, device=dev)
    plan = mk.Plan(cfg, w, batch, max_ctx)
    tokens = synth.make_tokens(batch, cfg.vocab).to(dev)
    positions = torch.tensor(pos_list, dtype=torch.int32, device=dev)
    logits = torch.empty((batch, cfg.vocab), dtype=torch.float32, device=dev)

    def mega():
        plan.decode_step(tokens, positions, kv, logits, stream=stream)

    def graph():
        plan.run_per_op(mk.MK_DECODE, tokens, positions, kv, logits, use_graph=True, stream=stream)

    for _ in range(args.warmup):
        mega()
    per = []
    ms = timed(mega, args.steps, per) / args.steps
    for _ in range(max(1, args.warmup // 2)):
        graph()
    ms_graph = timed(graph, args.steps) / args.steps
    # a prompt chunk of the last slot (half the columns, consecutive positions
    # before its context) mixed with decode tokens of the other slots
    half = batch // 2
    cslot = batch - 1
    cpos = pos_list[cslot] - half
    slots_m = torch.tensor(list(range(batch - half)) + [cslot] * half, dtype=torch.int32, device=dev)
    pos_m = torch.tensor(pos_list[:batch - half] + [cpos + i for i in range(half)], dtype=torch.int32,
                         device=dev)

    def mixed():
        plan.decode_step_slots(tokens, pos_m, slots_m, kv, logits, stream=stream)

    for _ in range(max(1, args.warmup // 2)):
        mixed()
    ms_mixed = timed(mixed, args.steps) / args.steps
    rc = plan.status(stream)
    if rc != mk.MK_OK:
        raise RuntimeError(f"{name}: device status {rc}")
    # several prompts prefilled in one launch (each weight tile streamed once
    # for all of them) against one launch per prompt
    batch_prefill = None
    if batch >= BATCH_PREFILL_PROMPTS:
        n_p = BATCH_PREFILL_PROMPTS
        ptoks = synth.make_tokens(n_p * BATCH_PREFILL_TOKENS, cfg.vocab, seed=synth.SEED_TOKENS + 11)
        ptoks = ptoks.view(n_p, BATCH_PREFILL_TOKENS).to(dev)
        lens = [BATCH_PREFILL_TOKENS] * n_p
        plog = torch.empty((n_p, cfg.vocab), dtype=torch.float32, device=dev)

        def one_launch():
            plan.prefill_batch(ptoks, lens, kv, plog, stream=stream)

        def per_prompt():
            for b in range(n_p):
                plan.prefill_batch(ptoks[b:b + 1], lens[:1], kv, plog[b:b + 1], stream=stream)

        one_launch()
        per_prompt()
        pf_steps = max(3, args.steps // 10)
        ms_one = timed(one_launch, pf_steps) / pf_steps
        ms_each = timed(per_prompt, pf_steps) / pf_steps
        rc = plan.status(stream)
        if rc != mk.MK_OK:
            raise RuntimeError(f"{name}: batch prefill device status {rc}")
        ntok = n_p * BATCH_PREFILL_TOKENS
        batch_prefill = {"prompts": n_p, "tokens_each": BATCH_PREFILL_TOKENS,
                         "ms_one_launch": ms_one, "ms_one_launch_per_prompt": ms_each,
                         "tokens_per_s_one_launch": ntok / (ms_one / 1e3),
                         "tokens_per_s_per_prompt": ntok / (ms_each / 1e3),
                         "speedup": ms_each / ms_one}
    peaks, kind = measured_peaks()
    nbytes = algorithmic_bytes(cfg, batch, pos_list)
    achieved = nbytes / (ms / 1e3) / 1e9
    out = {"workload": desc, "metric": metric, "batch": batch,
           "path": "tensor-core persistent" if plan.stats().decode_path == 1 else "cuda-core persistent",
           "ms_per_step": ms, "ms_per_step_stats": step_stats(per),
           "tokens_per_s": batch / (ms / 1e3),
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "peak_kind": kind,
                        "kernel": "mk_bdecode_kernel" if plan.stats().decode_path == 1 else "mk_interpreter",
                        "algorithmic_bytes_per_launch": nbytes,
                        "traffic": None if args.batched_layers else recorded_traffic("mk_bdecode_kernel", name)},
           "per_op_graph_ms_per_step": ms_graph, "speedup_persistent_vs_graph": ms_graph / ms,
           "mixed_chunk": {"decode_columns": batch - half, "chunk_tokens": half, "ms_per_step": ms_mixed,
                           "tokens_per_s": batch / (ms_mixed / 1e3)},
           "batch_prefill": batch_prefill}
    plan.close()
    del w, kv
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-layers", type=int, default=0,
                    help="oracle layers per reference step (0: the whole model)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-per-op", action="store_true")
    ap.add_argument("--no-batched", action="store_true",
                    help="skip the batch-8 and batch-32 tensor-core decode legs")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama3-8b")
    ap.add_argument("--batched-layers", type=int, default=0,
                    help="run the batched legs on their first N layers (an ncu profiling case)")
    ap.add_argument("--batched-leg", action="append", choices=BATCHED_LEGS,
                    help="run only this batched leg (repeatable; default: all)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
