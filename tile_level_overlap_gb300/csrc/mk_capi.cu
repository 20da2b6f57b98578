// C ABI of libmk (declared in include/mk.h).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_bdecode.h"
#include "mk_internal.h"
#include "mk_plan.h"
#include "mk_prefill.h"
#include "mk_tmap.h"
#include "mk_variants.h"

namespace mk {
cudaError_t pf_setup();
cudaError_t pf_launch_mega(const PfParams& p, int ctas, cudaStream_t st);
cudaError_t pf_launch_perop(const PfParams& p, uint32_t first, uint32_t count, cudaStream_t st);
}  // namespace mk

using namespace mk;

// Prefill state of a plan, built on the first prefill call.
struct PrefillState {
  bool built = false;
  PrefillPlan pp;
  void* mem = nullptr;
  size_t bytes = 0;
  PfParams base{};
  CUtensorMap* d_tm = nullptr;          // device copy of the tensor-map table
  std::vector<CUtensorMap> h_tm;        // host copy (source of the uploads)
  const void* kv_mapped = nullptr;      // KV cache the table's cache map points at
  int4* d_blk = nullptr;                // block table of a several-prompt launch [n_blocks]
};

// Tensor-core batched decode state of a plan (shapes whose batch the CUDA-core
// decode path does not take).
struct BdState {
  bool on = false;
  BdPlan bp;
  void* mem = nullptr;
  CUtensorMap* d_tm = nullptr;
  std::vector<CUtensorMap> h_tm;
  const void* kv_mapped = nullptr;
  Instr* d_queue = nullptr;
  BdParams base{};
  size_t arrive_words = 0;
};

struct mk_plan {
  HostPlan hp;  // CUDA-core decode plan (batch 1 only when bd.on: it serves the prefill's LM head)
  BdState bd;
  int max_batch = 0;  // sequences a decode step may carry (the caller's)
  KernelVariant kv{};
  std::vector<LayerW> lw;  // host copy of the per-layer weight pointers
  PrefillState pf;
  int device = 0, n_sms = 0, max_ctas = 0;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  size_t tagged_bytes = 0;      // the tagged intermediate tensors at the scratch's start
  Instr* d_queue = nullptr;     // default topological order (per-op ranges index it)
  Instr* d_queue_mk = nullptr;  // order popped by the persistent kernel
  unsigned long long* d_trace = nullptr;
  int32_t* d_tok = nullptr;     // staging for the host-buffer entry point
  int32_t* d_pos = nullptr;
  float* d_logits = nullptr;
  uint32_t* d_ctl = nullptr;
  uint8_t* d_msteps = nullptr;  // multi-step decode: one word per (step, CTA)
  KParams base{};
  int force_ctas = 0, trace = 0;
  int lm_separate = 0;  // MK_LM_SEPARATE: the LM head runs as its own kernel-per-op launch
  uint64_t wait_limit_ns = 2000000000ull;
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t graph = nullptr;
  uintptr_t graph_key[6] = {0, 0, 0, 0, 0, 0};
  size_t kv_bytes = 0;
  int latched = 0;  // device error seen by mk_status / the host-buffer step
};

namespace {

struct Bump {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  }
};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int cuda_err(cudaError_t e) { return e == cudaSuccess ? MK_OK : MK_ERR_CUDA; }

// The compiled interpreter specialisation for this shape, else the generic one.
KernelVariant pick_variant(const HostPlan& hp) {
  const mk_model_cfg& c = hp.cfg;
  if (hp.fast_b1) {
    const KernelVariant cands[] = {variant_h1_f4_d64_r4(), variant_h2_f7_d128_r4(),
                                   variant_h2_f6_d128_r4()};
    for (const KernelVariant& v : cands)
      if (v.mh * FAST_K_UNIT == c.hidden && v.mf * FAST_K_UNIT == c.ffn && v.ad == c.head_dim &&
          v.arep == hp.rep)
        return v;
  }
  return variant_generic();
}

#define MK_CUDA(call)                        \
  do {                                       \
    cudaError_t e_ = (call);                 \
    if (e_ != cudaSuccess) return MK_ERR_CUDA; \
  } while (0)

int upload_mk_queue(mk_plan* p, uint64_t seed) {
  const std::vector<Instr>& q = p->hp.decode;
  if (seed == 0)
    return cuda_err(cudaMemcpy(p->d_queue_mk, q.data(), q.size() * sizeof(Instr),
                               cudaMemcpyHostToDevice));
  std::vector<Instr> perm;
  random_topological(p->hp, q, seed, &perm);
  std::string why;
  if (perm.size() != q.size() || simulate(p->hp, perm, &why) != MK_OK) return MK_ERR_INVALID_ARG;
  return cuda_err(cudaMemcpy(p->d_queue_mk, perm.data(), perm.size() * sizeof(Instr),
                             cudaMemcpyHostToDevice));
}

// ---------------------------------------------------------------- batched decode (tensor cores)
// Buffers, tensor maps and launch parameters of the tensor-core batched path.
int bd_init(mk_plan* p, const mk_weight_ptrs* w) {
  BdState& s = p->bd;
  const BdPlan& bp = s.bp;
  if (bd_setup() != cudaSuccess) return MK_ERR_CUDA;
  const mk_model_cfg& c = bp.cfg;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, F = c.ffn, nkv = c.n_kv_heads;
  const int qd = c.n_q_heads * d, kd = nkv * d, NB = bp.nb;
  // split-K partials and arrival counters in two regions: O and down in the
  // first, QKV and gate/up in the second (neighbouring operators overlap)
  const size_t pairs_a = std::max((size_t)bp.n_o_m * bp.c_q, (size_t)bp.n_down_m * bp.c_f);
  const size_t pairs_b = std::max((size_t)bp.n_qkv_m * bp.c_k, (size_t)bp.n_gu_m * bp.c_g);
  const uint32_t m_a = std::max(bp.n_o_m, bp.n_down_m), m_b = std::max(bp.n_qkv_m, bp.n_gu_m);
  const int n_maps = L * BD_TM_PER_LAYER + TMB_COUNT;
  Bump bm;
  const size_t o_bars = bm.take(sizeof(uint32_t) * bp.bl.total);
  const size_t o_ctl = bm.take(sizeof(uint32_t) * CTL_WORDS);
  const size_t o_q = bm.take(sizeof(Instr) * bp.queue.size());
  const size_t o_qmk = bm.take(sizeof(Instr) * bp.queue.size());
  const size_t o_tm = bm.take(sizeof(CUtensorMap) * n_maps);
  const size_t o_xa = bm.take(sizeof(float) * NB * H);
  const size_t o_xb = bm.take(sizeof(float) * NB * H);
  const size_t o_hn = bm.take(4 * (size_t)NB * H);
  const size_t o_ao = bm.take(4 * (size_t)NB * qd);
  const size_t o_act = bm.take(4 * (size_t)NB * F);
  const size_t o_qv = bm.take(sizeof(float) * NB * qd);
  const size_t o_ss1 = bm.take(sizeof(float) * std::max<uint32_t>(bp.n_down_m, 1) * BD_NMAX);
  const size_t o_ss2 = bm.take(sizeof(float) * bp.n_o_m * BD_NMAX);
  const size_t o_part = bm.take(sizeof(float) * (pairs_a + pairs_b) * BD_NMAX * BD_M);
  const size_t o_apart = bm.take(sizeof(float) * bp.max_batch * nkv * bp.nsplit * bp.rep * (d + 2));
  s.arrive_words = (size_t)m_a + m_b + (size_t)bp.max_batch * nkv;
  const size_t o_arr = bm.take(sizeof(uint32_t) * s.arrive_words);
  if (cudaMalloc(&s.mem, bm.off) != cudaSuccess) {
    cudaGetLastError();
    s.mem = nullptr;
    return MK_ERR_CUDA;
  }
  p->scratch_bytes += bm.off;
  uint8_t* b = (uint8_t*)s.mem;
  MK_CUDA(cudaMemset(s.mem, 0, bm.off));
  MK_CUDA(cudaMemcpy(b + o_q, bp.queue.data(), sizeof(Instr) * bp.queue.size(), cudaMemcpyHostToDevice));
  MK_CUDA(cudaMemcpy(b + o_qmk, bp.queue.data(), sizeof(Instr) * bp.queue.size(), cudaMemcpyHostToDevice));
  s.d_queue = (Instr*)(b + o_q);
  s.d_tm = (CUtensorMap*)(b + o_tm);
  s.h_tm.assign(n_maps, CUtensorMap{});
  bool ok = true;
  for (int l = 0; l < L && ok; ++l) {
    const LayerW& x = p->lw[l];
    CUtensorMap* t = &s.h_tm[l * BD_TM_PER_LAYER];
    ok = make_tmap_bf16(t + TMB_WQ, x.wq, qd, H, BD_M) && make_tmap_bf16(t + TMB_WK, x.wk, kd, H, BD_M) &&
         make_tmap_bf16(t + TMB_WV, x.wv, kd, H, BD_M) && make_tmap_bf16(t + TMB_WO, x.wo, H, qd, BD_M) &&
         make_tmap_bf16(t + TMB_WG, x.wg, F, H, BD_M / 2) &&
         make_tmap_bf16(t + TMB_WU, x.wu, F, H, BD_M / 2) && make_tmap_bf16(t + TMB_WD, x.wd, H, F, BD_M);
  }
  CUtensorMap* gm = &s.h_tm[L * BD_TM_PER_LAYER];
  const void* lm = c.tied_embeddings ? w->embed : w->lm_head;
  ok = ok && make_tmap_bf16(gm + TMB_LM, lm, c.vocab, H, BD_M) &&
       make_tmap_bf16(gm + TMB_HN, b + o_hn, 2 * NB, H, NB) &&
       make_tmap_bf16(gm + TMB_AO, b + o_ao, 2 * NB, qd, NB) &&
       make_tmap_bf16(gm + TMB_ACT, b + o_act, 2 * NB, F, NB);
  if (!ok) return MK_ERR_CUDA;
  MK_CUDA(cudaMemcpy(s.d_tm, s.h_tm.data(), sizeof(CUtensorMap) * n_maps, cudaMemcpyHostToDevice));
  BdParams& k = s.base;
  std::memset(&k, 0, sizeof(k));
  k.L = L; k.H = H; k.nq = c.n_q_heads; k.nkv = nkv; k.d = d; k.F = F; k.V = c.vocab;
  k.qk_norm = c.qk_norm; k.rep = bp.rep; k.qkv_rows = bp.qkv_rows; k.max_ctx = bp.max_ctx;
  k.max_batch = bp.max_batch; k.nb = NB; k.n_rg = bp.n_rg; k.nsplit = bp.nsplit; k.eps = c.rms_eps;
  k.n_qkv_m = bp.n_qkv_m; k.n_o_m = bp.n_o_m; k.n_gu_m = bp.n_gu_m; k.n_down_m = bp.n_down_m;
  k.n_lm_m = bp.n_lm_m; k.c_h = bp.c_h; k.c_q = bp.c_q; k.c_f = bp.c_f; k.c_g = bp.c_g; k.c_k = bp.c_k;
  k.embed = (const uint16_t*)w->embed;
  k.final_norm = (const uint16_t*)w->final_norm;
  k.layers = p->base.layers;
  k.tm = s.d_tm;
  k.xa = (float*)(b + o_xa);
  k.xb = (float*)(b + o_xb);
  k.hn = (uint16_t*)(b + o_hn);
  k.ao = (uint16_t*)(b + o_ao);
  k.act = (uint16_t*)(b + o_act);
  k.q = (float*)(b + o_qv);
  k.ss1 = (float*)(b + o_ss1);
  k.ss2 = (float*)(b + o_ss2);
  k.part = (float*)(b + o_part);
  k.apart = (float*)(b + o_apart);
  k.arrive = (uint32_t*)(b + o_arr);
  k.part_b = (uint32_t)pairs_a;
  k.arrive_b = m_a;
  k.n_arrive_gemm = m_a + m_b;
  k.rope = p->base.rope;
  k.bars = (uint32_t*)(b + o_bars);
  k.ctl = (uint32_t*)(b + o_ctl);
  k.queue = (const Instr*)(b + o_qmk);
  k.n_instr = (uint32_t)bp.queue.size();
  return MK_OK;
}

// Point the table's cache map at this call's KV cache.
int bd_bind_kv(mk_plan* p, void* kv, cudaStream_t st) {
  BdState& s = p->bd;
  if (s.kv_mapped == kv) return MK_OK;
  const mk_model_cfg& c = s.bp.cfg;
  const int idx = c.n_layers * BD_TM_PER_LAYER + TMB_KV;
  const uint64_t rows = (uint64_t)c.n_layers * 2 * p->max_batch * c.n_kv_heads * s.bp.max_ctx;
  if (!make_tmap_bf16(&s.h_tm[idx], kv, rows, (uint64_t)c.head_dim, BD_KEYS)) return MK_ERR_CUDA;
  MK_CUDA(cudaMemcpyAsync(s.d_tm + idx, &s.h_tm[idx], sizeof(CUtensorMap), cudaMemcpyHostToDevice, st));
  MK_CUDA(cudaStreamSynchronize(st));
  s.kv_mapped = kv;
  return MK_OK;
}

BdParams bd_params(mk_plan* p, const int32_t* tokens, const int32_t* positions, int batch, void* kv,
                   float* logits) {
  BdParams k = p->bd.base;
  k.tokens = tokens;
  k.positions = positions;
  k.B = batch;
  k.kv = (uint16_t*)kv;
  k.logits = logits;
  k.mode = MODE_MEGA;
  k.wait_limit_ns = p->wait_limit_ns;
  k.trace = p->trace ? p->d_trace : nullptr;
  return k;
}

int bd_upload_queue(mk_plan* p, uint64_t seed) {
  BdState& s = p->bd;
  std::vector<Instr> q = s.bp.queue;
  if (seed) {
    random_order_bdecode(s.bp, seed, &q);
    std::string why;
    if (q.size() != s.bp.queue.size() || simulate_bdecode(s.bp, q, &why) != MK_OK) return MK_ERR_INVALID_ARG;
  }
  return cuda_err(cudaMemcpy(const_cast<Instr*>(s.base.queue), q.data(), q.size() * sizeof(Instr),
                             cudaMemcpyHostToDevice));
}

}  // namespace

extern "C" {

const char* mk_status_string(int code) {
  switch (code) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID_ARG: return "invalid argument";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_TIMEOUT: return "device-side wait timed out";
    case MK_ERR_BOUNDS: return "token, position or operand out of range";
    case MK_ERR_UNSUPPORTED: return "shape not supported by this build";
    case MK_ERR_NO_DEVICE: return "no CUDA device";
    default: return "unknown status";
  }
}

int mk_plan_check(const mk_model_cfg* cfg, int max_batch, int max_ctx, uint64_t queue_perm_seed,
                  mk_plan_stats* out) {
  if (!cfg) return MK_ERR_INVALID_ARG;
  HostPlan hp;
  std::string why;
  int rc = build_plan(*cfg, max_batch, max_ctx, 0, &hp, &why);
  if (rc == MK_ERR_UNSUPPORTED && max_batch > 1) {
    BdPlan bp;
    if (build_bdecode(*cfg, max_batch, max_ctx, 0, &bp, &why) != MK_OK) return rc;
    std::vector<Instr> q = bp.queue;
    if (queue_perm_seed) random_order_bdecode(bp, queue_perm_seed, &q);
    if (q.size() != bp.queue.size()) return MK_ERR_INVALID_ARG;
    rc = simulate_bdecode(bp, q, &why);
    if (out) {
      std::memset(out, 0, sizeof(*out));
      out->n_instr_decode = (uint32_t)bp.queue.size();
      out->n_barriers = bp.bl.total;
      out->n_launches_per_op_decode = (uint32_t)bp.perop.size();
      out->n_splits = (uint32_t)bp.nsplit;
      out->decode_path = 1;
    }
    return rc;
  }
  if (rc != MK_OK) return rc;
  std::vector<Instr> q = hp.decode;
  if (queue_perm_seed) {
    random_topological(hp, hp.decode, queue_perm_seed, &q);
    if (q.size() != hp.decode.size()) return MK_ERR_INVALID_ARG;
  }
  rc = simulate(hp, q, &why);
  // the prefill queue, when this shape has a prefill path
  PrefillPlan pp;
  const bool has_pf = build_prefill(*cfg, max_ctx, &pp, &why) == MK_OK;
  if (rc == MK_OK && has_pf) rc = simulate_prefill(pp, pp.queue, &why);
  if (out) {
    std::memset(out, 0, sizeof(*out));
    out->n_instr_decode = (uint32_t)hp.decode.size();
    out->n_instr_prefill = has_pf ? (uint32_t)pp.queue.size() : 0u;
    out->n_barriers = hp.bl.total;
    out->n_launches_per_op_decode = (uint32_t)hp.perop_decode.size();
    out->n_splits = (uint32_t)hp.n_splits;
    out->weight_bytes = hp.weight_bytes;
  }
  return rc;
}

int mk_plan_create(const mk_model_cfg* cfg, const mk_weight_ptrs* w, int max_batch, int max_ctx,
                   mk_plan** out) {
  return mk_plan_create_for_sms(cfg, w, max_batch, max_ctx, 0, out);
}

int mk_plan_create_for_sms(const mk_model_cfg* cfg, const mk_weight_ptrs* w, int max_batch,
                           int max_ctx, int n_sms, mk_plan** out) {
  if (!cfg || !w || !out || n_sms < 0) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return MK_ERR_NO_DEVICE;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  if (n_sms > sms) return MK_ERR_INVALID_ARG;
  if (n_sms > 0) sms = n_sms;  // tile the plan, and launch it, as on a device with n_sms SMs
  mk_plan* p = new mk_plan();
  std::string why;
  p->max_batch = max_batch;
  int rc = build_plan(*cfg, max_batch, max_ctx, sms, &p->hp, &why);
  if (rc == MK_ERR_UNSUPPORTED && max_batch > 1 &&
      build_bdecode(*cfg, max_batch, max_ctx, sms, &p->bd.bp, &why) == MK_OK) {
    // the batch goes to the tensor-core path; the CUDA-core plan keeps one
    // sequence for the prefill's LM head
    p->bd.on = true;
    rc = build_plan(*cfg, 1, max_ctx, sms, &p->hp, &why);
  }
  if (rc != MK_OK) {
    delete p;
    return rc;
  }
  const HostPlan& hp = p->hp;
  const mk_model_cfg& c = hp.cfg;
  const int L = c.n_layers;
  // weight pointers
  std::vector<LayerW> lw(L);
  auto ok = [](const void* q) { return q != nullptr && aligned16(q); };
  bool good = ok(w->embed) && ok(w->final_norm) && (c.tied_embeddings || ok(w->lm_head)) &&
              w->attn_norm && w->wq && w->wk && w->wv && w->wo && w->ffn_norm && w->w_gate &&
              w->w_up && w->w_down && (!c.qk_norm || (w->q_norm && w->k_norm));
  for (int l = 0; good && l < L; ++l) {
    LayerW& x = lw[l];
    x.attn_norm = (const uint16_t*)w->attn_norm[l];
    x.wq = (const uint16_t*)w->wq[l];
    x.wk = (const uint16_t*)w->wk[l];
    x.wv = (const uint16_t*)w->wv[l];
    x.wo = (const uint16_t*)w->wo[l];
    x.q_norm = c.qk_norm ? (const uint16_t*)w->q_norm[l] : nullptr;
    x.k_norm = c.qk_norm ? (const uint16_t*)w->k_norm[l] : nullptr;
    x.ffn_norm = (const uint16_t*)w->ffn_norm[l];
    x.wg = (const uint16_t*)w->w_gate[l];
    x.wu = (const uint16_t*)w->w_up[l];
    x.wd = (const uint16_t*)w->w_down[l];
    good = ok(x.attn_norm) && ok(x.wq) && ok(x.wk) && ok(x.wv) && ok(x.wo) && ok(x.ffn_norm) &&
           ok(x.wg) && ok(x.wu) && ok(x.wd) && (!c.qk_norm || (ok(x.q_norm) && ok(x.k_norm)));
  }
  if (!good) {
    delete p;
    return MK_ERR_INVALID_ARG;
  }

  auto fail = [&](int code) {
    mk_plan_destroy(p);
    return code;
  };
  if (cudaGetDevice(&p->device) != cudaSuccess) return fail(MK_ERR_CUDA);
  p->n_sms = sms;
  p->kv = pick_variant(p->hp);
  if (p->kv.setup() != cudaSuccess) return fail(MK_ERR_CUDA);
  int per_sm = 0;
  if (p->kv.occupancy(&per_sm) != cudaSuccess || per_sm < 1) return fail(MK_ERR_CUDA);
  p->max_ctas = p->n_sms;

  // one scratch allocation: the decode layout (shared with the no-allocation
  // entry point), then a second copy of the queue, the host-buffer staging and
  // the multi-step words
  const int H = c.hidden, d = c.head_dim, F = c.ffn, nkv = c.n_kv_heads;
  const DecodeScratch ds = decode_scratch(hp);
  Bump bm;
  bm.off = ds.total;
  const size_t o_qmk = bm.take(sizeof(Instr) * hp.decode.size());
  const size_t o_tok = bm.take(sizeof(int32_t) * max_batch);
  const size_t o_pos = bm.take(sizeof(int32_t) * max_batch);
  const size_t o_log = bm.take(sizeof(float) * max_batch * c.vocab);
  // multi-step decode: per step the packed maximum (u64), the finished LM
  // tiles and the chosen token, cleared together before each such launch
  const size_t o_msteps = bm.take(sizeof(unsigned long long) * MAX_DECODE_STEPS * (size_t)p->max_ctas);
  p->scratch_bytes = bm.off;
  p->tagged_bytes = ds.tagged_end;
  if (cudaMalloc(&p->scratch, p->scratch_bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(MK_ERR_CUDA);
  }
  uint8_t* s = (uint8_t*)p->scratch;
  if (cudaMemset(p->scratch, 0, p->scratch_bytes) != cudaSuccess) return fail(MK_ERR_CUDA);
  const size_t o_q = ds.o_q, o_rope = ds.o_rope, o_lw = ds.o_lw;

  std::vector<float2> rope((size_t)max_ctx * (d / 2));
  for (int pos = 0; pos < max_ctx; ++pos)
    for (int i = 0; i < d / 2; ++i) {
      const double inv = std::pow((double)c.rope_theta, -2.0 * i / d);
      const double a = (double)pos * inv;
      rope[(size_t)pos * (d / 2) + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  p->d_queue = (Instr*)(s + o_q);
  p->d_queue_mk = (Instr*)(s + o_qmk);
  p->d_ctl = (uint32_t*)(s + ds.o_ctl);
  p->d_tok = (int32_t*)(s + o_tok);
  p->d_pos = (int32_t*)(s + o_pos);
  p->d_logits = (float*)(s + o_log);
  if (cudaMemcpy(s + o_q, hp.decode.data(), sizeof(Instr) * hp.decode.size(),
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(s + o_qmk, hp.decode.data(), sizeof(Instr) * hp.decode.size(),
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(s + o_rope, rope.data(), sizeof(float2) * rope.size(), cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemcpy(s + o_lw, lw.data(), sizeof(LayerW) * L, cudaMemcpyHostToDevice) != cudaSuccess ||
      (p->lw = lw, false))
    return fail(MK_ERR_CUDA);
  if (cudaStreamCreateWithFlags(&p->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
    return fail(MK_ERR_CUDA);

  KParams& k = p->base;
  std::memset(&k, 0, sizeof(k));
  k.L = L; k.H = H; k.nq = c.n_q_heads; k.nkv = nkv; k.d = d; k.F = F; k.V = c.vocab;
  k.qk_norm = c.qk_norm; k.rep = hp.rep; k.qkv_rows = hp.qkv_rows; k.eps = c.rms_eps;
  k.max_batch = hp.max_batch; k.max_ctx = max_ctx; k.n_splits = hp.n_splits;
  k.r_qkv = hp.r_qkv; k.r_o = hp.r_o; k.r_gu = hp.r_gu; k.r_down = hp.r_down; k.r_lm = hp.r_lm;
  k.n_qkv_tiles = hp.n_qkv_tiles; k.n_o_tiles = hp.n_o_tiles; k.n_gu_tiles = hp.n_gu_tiles;
  k.n_down_tiles = hp.n_down_tiles; k.n_lm_tiles = hp.n_lm_tiles;
  k.embed = (const uint16_t*)w->embed;
  k.lm = (const uint16_t*)(c.tied_embeddings ? w->embed : w->lm_head);
  k.final_norm = (const uint16_t*)w->final_norm;
  k.layers = (const LayerW*)(s + o_lw);
  k.resid = (u64*)(s + ds.o_resid);
  k.qkv = (u64*)(s + ds.o_qkv);
  k.part = (u64*)(s + ds.o_part);
  k.attn_out = (u64*)(s + ds.o_attn);
  k.act = (u64*)(s + ds.o_act);
  k.kps = hp.kps;
  k.comb_per = (hp.rep * c.head_dim + hp.n_comb - 1) / hp.n_comb;
  k.bars = (uint32_t*)(s + ds.o_bars);
  k.rope = (const float2*)(s + o_rope);
  k.ctl = p->d_ctl;
  k.queue = p->d_queue_mk;
  k.n_instr = (uint32_t)hp.decode.size();
  k.n_steps = 1;
  p->d_msteps = s + o_msteps;
  std::memcpy(k.xw, hp.expr.data(), sizeof(k.xw));
  k.bl = hp.bl;
  p->kv_bytes = (size_t)L * 2 * max_batch * nkv * (size_t)max_ctx * d * 2;
  if (p->bd.on && (rc = bd_init(p, w)) != MK_OK) return fail(rc);
  *out = p;
  return MK_OK;
}

void mk_plan_destroy(mk_plan* p) {
  if (!p) return;
  if (p->graph) cudaGraphExecDestroy(p->graph);
  if (p->cap_stream) cudaStreamDestroy(p->cap_stream);
  if (p->d_trace) cudaFree(p->d_trace);
  if (p->scratch) cudaFree(p->scratch);
  if (p->pf.mem) cudaFree(p->pf.mem);
  if (p->bd.mem) cudaFree(p->bd.mem);
  delete p;
}

size_t mk_kv_cache_bytes(const mk_plan* p) { return p ? p->kv_bytes : 0; }

int mk_plan_get_stats(const mk_plan* p, mk_plan_stats* out) {
  if (!p || !out) return MK_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->n_instr_decode = (uint32_t)p->hp.decode.size();
  {
    PrefillPlan pp;
    std::string why;
    out->n_instr_prefill = p->pf.built ? (uint32_t)p->pf.pp.queue.size()
                           : build_prefill(p->hp.cfg, p->hp.max_ctx, &pp, &why) == MK_OK
                               ? (uint32_t)pp.queue.size()
                               : 0u;
  }
  out->n_barriers = p->hp.bl.total;
  out->n_launches_per_op_decode = (uint32_t)p->hp.perop_decode.size();
  out->n_ctas = (uint32_t)(p->force_ctas ? p->force_ctas : p->max_ctas);
  {
    // FNV-1a over the decode queue as the device holds it (the order the
    // persistent kernel pops)
    const Instr* dq = p->bd.on ? p->bd.base.queue : p->d_queue_mk;
    const size_t n = p->bd.on ? p->bd.bp.queue.size() : p->hp.decode.size();
    std::vector<uint8_t> q(n * sizeof(Instr));
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(q.data(), dq, q.size(), cudaMemcpyDeviceToHost) != cudaSuccess)
      return MK_ERR_CUDA;
    uint64_t h = 1469598103934665603ull;
    for (uint8_t v : q) h = (h ^ v) * 1099511628211ull;
    out->queue_hash = h;
  }
  out->n_splits = (uint32_t)p->hp.n_splits;
  out->weight_bytes = p->hp.weight_bytes;
  out->scratch_bytes = p->scratch_bytes;
  if (p->bd.on) {
    out->n_instr_decode = (uint32_t)p->bd.bp.queue.size();
    out->n_barriers = p->bd.bp.bl.total;
    out->n_launches_per_op_decode = (uint32_t)p->bd.bp.perop.size();
    out->n_splits = (uint32_t)p->bd.bp.nsplit;
    out->decode_path = 1;
  }
  return MK_OK;
}

static int check_step(mk_plan* p, const void* tokens, const void* positions, int batch,
                      const void* kv, const void* logits) {
  if (!p || !tokens || !positions || !kv || !logits) return MK_ERR_INVALID_ARG;
  if (batch < 1 || batch > p->max_batch) return MK_ERR_INVALID_ARG;
  if (!aligned16(kv)) return MK_ERR_INVALID_ARG;
  if (p->latched) return p->latched;
  return MK_OK;
}

static KParams step_params(mk_plan* p, const int32_t* tokens, const int32_t* positions, int batch,
                           void* kv, float* logits) {
  KParams k = p->base;
  k.tokens = tokens;
  k.positions = positions;
  k.B = batch;
  k.S = 0;
  k.kv = (uint16_t*)kv;
  k.logits = logits;
  k.mode = MODE_MEGA;
  k.trace = p->trace ? p->d_trace : nullptr;
  k.wait_limit_ns = p->wait_limit_ns;
  return k;
}

int mk_decode_step(mk_plan* p, const int32_t* tokens, const int32_t* positions, int batch,
                   void* kv, float* logits, void* stream) {
  int rc = check_step(p, tokens, positions, batch, kv, logits);
  if (rc != MK_OK) return rc;
  const int ctas = p->force_ctas ? p->force_ctas : p->max_ctas;
  cudaStream_t st = (cudaStream_t)stream;
  // MK_LM_SEPARATE: the persistent launch stops before the LM-head tiles (the
  // last instructions of every topological order: each waits on all of the
  // last down projection), which then run as one kernel-per-operator launch.
  if (p->bd.on) {
    if ((rc = bd_bind_kv(p, kv, st)) != MK_OK) return rc;
    BdParams k = bd_params(p, tokens, positions, batch, kv, logits);
    if (!p->lm_separate) return cuda_err(bd_launch_mega(k, ctas, st));
    const auto& r = p->bd.bp.perop.back();  // the LM-head tiles
    k.n_instr -= r.second;
    MK_CUDA(bd_launch_mega(k, ctas, st));
    k.n_instr += r.second;
    k.queue = p->bd.d_queue;  // per-operator ranges index the default order
    k.trace = nullptr;
    return cuda_err(bd_launch_perop(k, r.first, r.second, st));
  }
  KParams k = step_params(p, tokens, positions, batch, kv, logits);
  if (!p->lm_separate) return cuda_err(p->kv.mega(k, ctas, st));
  const auto& r = p->hp.perop_decode.back();  // the LM-head tiles
  k.n_instr -= r.second;
  MK_CUDA(p->kv.mega(k, ctas, st));
  k.n_instr += r.second;
  k.queue = p->d_queue;
  k.trace = nullptr;
  return cuda_err(p->kv.perop(k, r.first, r.second, p->max_ctas, st));
}

int mk_decode_steps(mk_plan* p, const int32_t* token, const int32_t* position, int n_steps,
                    void* kv, int32_t* out_tokens, float* logits, void* stream) {
  int rc = check_step(p, token, position, 1, kv, logits);
  if (rc != MK_OK) return rc;
  if (!out_tokens || n_steps < 1 || n_steps > (int)MAX_DECODE_STEPS) return MK_ERR_INVALID_ARG;
  if (p->bd.on || !p->hp.fast_b1) return MK_ERR_UNSUPPORTED;
  if (p->hp.cfg.vocab >= (1 << 18)) return MK_ERR_UNSUPPORTED;  // rows packed in 18 bits
  cudaStream_t st = (cudaStream_t)stream;
  const int ctas = p->force_ctas ? p->force_ctas : p->max_ctas;
  KParams k = step_params(p, token, position, 1, kv, logits);
  k.n_steps = (uint32_t)n_steps;
  k.lm_slot = reinterpret_cast<unsigned long long*>(p->d_msteps);
  k.out_tokens = out_tokens;
  MK_CUDA(cudaMemsetAsync(p->d_msteps, 0, sizeof(unsigned long long) * (size_t)n_steps * ctas, st));
  return cuda_err(p->kv.mega_steps(k, ctas, st));
}

int mk_decode_step_slots(mk_plan* p, const int32_t* tokens, const int32_t* positions,
                         const int32_t* slots, int batch, void* kv, float* logits, void* stream) {
  int rc = check_step(p, tokens, positions, batch, kv, logits);
  if (rc != MK_OK) return rc;
  if (!slots) return MK_ERR_INVALID_ARG;
  if (!p->bd.on) return MK_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const int ctas = p->force_ctas ? p->force_ctas : p->max_ctas;
  if ((rc = bd_bind_kv(p, kv, st)) != MK_OK) return rc;
  BdParams k = bd_params(p, tokens, positions, batch, kv, logits);
  k.slots = slots;
  return cuda_err(bd_launch_mega(k, ctas, st));
}

int mk_plan_set_lm_mode(mk_plan* p, int mode) {
  if (!p || (mode != MK_LM_FUSED && mode != MK_LM_SEPARATE)) return MK_ERR_INVALID_ARG;
  p->lm_separate = mode == MK_LM_SEPARATE;
  return MK_OK;
}

int mk_decode_step_host(mk_plan* p, const int32_t* tokens_host, const int32_t* positions_host,
                        int batch, void* kv, float* logits_host, void* stream) {
  int rc = check_step(p, tokens_host, positions_host, batch, kv, logits_host);
  if (rc != MK_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  MK_CUDA(cudaMemcpyAsync(p->d_tok, tokens_host, sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
  MK_CUDA(cudaMemcpyAsync(p->d_pos, positions_host, sizeof(int32_t) * batch, cudaMemcpyHostToDevice,
                          st));
  rc = mk_decode_step(p, p->d_tok, p->d_pos, batch, kv, p->d_logits, stream);
  if (rc != MK_OK) return rc;
  uint32_t status = 0;
  MK_CUDA(cudaMemcpyAsync(logits_host, p->d_logits, sizeof(float) * batch * p->hp.cfg.vocab,
                          cudaMemcpyDeviceToHost, st));
  MK_CUDA(cudaMemcpyAsync(&status, (p->bd.on ? p->bd.base.ctl : p->d_ctl) + CTL_STATUS,
                          sizeof(uint32_t), cudaMemcpyDeviceToHost, st));
  MK_CUDA(cudaStreamSynchronize(st));
  if (status) p->latched = (int)status;
  return (int)status;
}

// ---------------------------------------------------------------- prefill
// Build the prefill queue, its buffers and the tensor-map table (first call).
static int prefill_init(mk_plan* p) {
  PrefillState& s = p->pf;
  if (s.built) return MK_OK;
  std::string why;
  int rc = build_prefill(p->hp.cfg, p->hp.max_ctx, &s.pp, &why);
  if (rc != MK_OK) return rc;
  if (pf_setup() != cudaSuccess) return MK_ERR_CUDA;
  const mk_model_cfg& c = p->hp.cfg;
  const PrefillPlan& pp = s.pp;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, F = c.ffn;
  const int qd = c.n_q_heads * d, kd = c.n_kv_heads * d;
  const size_t rows = (size_t)pp.n_blocks * PF_BM;
  const int n_maps = L * TM_PER_LAYER + AM_COUNT;
  Bump bm;
  const size_t o_bars = bm.take(sizeof(uint32_t) * pp.bl.total);
  const size_t o_ctl = bm.take(sizeof(uint32_t) * CTL_WORDS);
  const size_t o_q = bm.take(sizeof(Instr) * pp.queue.size());
  const size_t o_tm = bm.take(sizeof(CUtensorMap) * n_maps);
  const size_t o_xa = bm.take(sizeof(float) * rows * H);
  const size_t o_xb = bm.take(sizeof(float) * rows * H);
  // hi and lo bf16 planes of each tensor-core activation operand
  const size_t o_hn1 = bm.take(4 * rows * H);
  const size_t o_hn2 = bm.take(4 * rows * H);
  const size_t o_qb = bm.take(4 * rows * qd);
  const size_t o_ao = bm.take(4 * rows * qd);
  const size_t o_act = bm.take(4 * rows * F);
  const size_t o_blk = bm.take(sizeof(int4) * pp.n_blocks);
  if (cudaMalloc(&s.mem, bm.off) != cudaSuccess) {
    cudaGetLastError();
    s.mem = nullptr;
    return MK_ERR_CUDA;
  }
  s.bytes = bm.off;
  uint8_t* b = (uint8_t*)s.mem;
  MK_CUDA(cudaMemset(s.mem, 0, s.bytes));
  s.d_tm = (CUtensorMap*)(b + o_tm);
  s.d_blk = (int4*)(b + o_blk);
  s.h_tm.assign(n_maps, CUtensorMap{});
  bool ok = true;
  for (int l = 0; l < L && ok; ++l) {
    const LayerW& w = p->lw[l];
    CUtensorMap* t = &s.h_tm[l * TM_PER_LAYER];
    ok = make_tmap_bf16(t + TM_WQ, w.wq, qd, H, pp.bn_qkv) &&
         make_tmap_bf16(t + TM_WK, w.wk, kd, H, pp.bn_qkv) &&
         make_tmap_bf16(t + TM_WV, w.wv, kd, H, pp.bn_qkv) &&
         make_tmap_bf16(t + TM_WO, w.wo, H, qd, PF_BN) &&
         make_tmap_bf16(t + TM_WG, w.wg, F, H, PF_BN_GU) &&
         make_tmap_bf16(t + TM_WU, w.wu, F, H, PF_BN_GU) &&
         make_tmap_bf16(t + TM_WD, w.wd, H, F, PF_BN);
  }
  CUtensorMap* a = &s.h_tm[L * TM_PER_LAYER];
  // each map spans both planes: the lo row of token row r is r + rows
  ok = ok && make_tmap_bf16(a + AM_HN1, b + o_hn1, 2 * rows, H, PF_BM) &&
       make_tmap_bf16(a + AM_HN2, b + o_hn2, 2 * rows, H, PF_BM) &&
       make_tmap_bf16(a + AM_AO, b + o_ao, 2 * rows, qd, PF_BM) &&
       make_tmap_bf16(a + AM_ACT, b + o_act, 2 * rows, F, PF_BM) &&
       make_tmap_bf16(a + AM_LMW, p->base.lm, (uint64_t)c.vocab, H, PF_BN);
  if (!ok) return MK_ERR_CUDA;
  MK_CUDA(cudaMemcpy(b + o_q, pp.queue.data(), sizeof(Instr) * pp.queue.size(), cudaMemcpyHostToDevice));
  MK_CUDA(cudaMemcpy(s.d_tm, s.h_tm.data(), sizeof(CUtensorMap) * n_maps, cudaMemcpyHostToDevice));
  PfParams& k = s.base;
  std::memset(&k, 0, sizeof(k));
  k.L = L; k.H = H; k.nq = c.n_q_heads; k.nkv = c.n_kv_heads; k.d = d; k.F = F; k.V = c.vocab;
  k.qk_norm = c.qk_norm; k.rep = pp.rep; k.qkv_rows = pp.qkv_rows; k.bn_qkv = pp.bn_qkv;
  k.n_blocks = pp.n_blocks; k.max_ctx = p->hp.max_ctx; k.max_batch = p->max_batch;
  k.eps = c.rms_eps;
  k.n_qkv_n = pp.n_qkv_n; k.n_o_n = pp.n_o_n; k.n_gu_n = pp.n_gu_n; k.n_down_n = pp.n_down_n;
  k.embed = p->base.embed;
  k.final_norm = p->base.final_norm;
  k.layers = p->base.layers;
  k.tm = s.d_tm;
  k.xa = (float*)(b + o_xa);
  k.xb = (float*)(b + o_xb);
  k.hn1 = (uint16_t*)(b + o_hn1);
  k.hn2 = (uint16_t*)(b + o_hn2);
  k.qb = (uint16_t*)(b + o_qb);
  k.ao = (uint16_t*)(b + o_ao);
  k.act = (uint16_t*)(b + o_act);
  k.plane_rows = (int)rows;
  k.rope = p->base.rope;
  k.bars = (uint32_t*)(b + o_bars);
  k.ctl = (uint32_t*)(b + o_ctl);
  k.queue = (const Instr*)(b + o_q);
  k.n_instr = pp.n_body;  // the all-token logits entry point runs the rest too
  std::memcpy(k.xw, pp.expr.data(), sizeof(k.xw));
  s.built = true;
  return MK_OK;
}

// Point the table's cache map at this call's KV cache.
static int prefill_bind_kv(mk_plan* p, void* kv, cudaStream_t st) {
  PrefillState& s = p->pf;
  if (s.kv_mapped == kv) return MK_OK;
  const mk_model_cfg& c = p->hp.cfg;
  const int idx = c.n_layers * TM_PER_LAYER + AM_KV;
  const uint64_t rows = (uint64_t)c.n_layers * 2 * p->max_batch * c.n_kv_heads * p->hp.max_ctx;
  if (!make_tmap_bf16(&s.h_tm[idx], kv, rows, (uint64_t)c.head_dim, PF_BM)) return MK_ERR_CUDA;
  MK_CUDA(cudaMemcpyAsync(s.d_tm + idx, &s.h_tm[idx], sizeof(CUtensorMap), cudaMemcpyHostToDevice, st));
  MK_CUDA(cudaStreamSynchronize(st));
  s.kv_mapped = kv;
  return MK_OK;
}

static int prefill_args(mk_plan* p, const int32_t* tokens, int len, void* kv, float* logits) {
  if (!p || !tokens || !kv || !logits || len < 1 || len > p->hp.max_ctx || !aligned16(kv))
    return MK_ERR_INVALID_ARG;
  if (p->latched) return p->latched;
  return MK_OK;
}

// The LM head of the prompt's last token runs as its own per-operator launch
// of the decode tiles after the prefill body ("Lecture 112", Practical
// implications: a megakernel body mixed with a separate LM-head op).
static int prefill_lm(mk_plan* p, const int32_t* tokens, int last_row, void* kv, float* logits,
                      cudaStream_t st) {
  const mk_model_cfg& c = p->hp.cfg;
  const float* last = p->pf.base.xb + (size_t)last_row * c.hidden;
  u64* dst = p->base.resid + (size_t)(2 * c.n_layers) * p->hp.max_batch * c.hidden;
  // the floats into the low halves of the tagged words (the kernel-per-operator
  // LM tiles read them without a tag check; their tags stay stale for any
  // later persistent launch, which waits for its own writes)
  MK_CUDA(cudaMemcpy2DAsync(dst, sizeof(u64), last, sizeof(float), sizeof(float), c.hidden,
                            cudaMemcpyDeviceToDevice, st));
  KParams k = step_params(p, tokens, tokens, 1, kv, logits);
  k.queue = p->d_queue;
  k.trace = nullptr;
  const auto& r = p->hp.perop_decode.back();  // the LM-head tiles
  return cuda_err(p->kv.perop(k, r.first, r.second, p->max_ctas, st));
}

int mk_prefill(mk_plan* p, const int32_t* tokens, int len, void* kv, float* logits, void* stream) {
  int rc = prefill_args(p, tokens, len, kv, logits);
  if (rc != MK_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = prefill_init(p)) != MK_OK || (rc = prefill_bind_kv(p, kv, st)) != MK_OK) return rc;
  PfParams k = p->pf.base;
  k.tokens = tokens;
  k.S = len;
  k.kv = (uint16_t*)kv;
  k.mode = MODE_MEGA;
  k.wait_limit_ns = p->wait_limit_ns;
  MK_CUDA(pf_launch_mega(k, p->n_sms, st));
  return prefill_lm(p, tokens, len - 1, kv, logits, st);
}

// One prefill chunk: `len` tokens of the sequence in cache slot `slot`,
// taking cache positions pos0 .. pos0 + len - 1 (positions below pos0 already
// cached), its tokens at tokens[tok .. tok + len).
struct PfChunk {
  int slot, pos0, len, tok;
};

// The chunks' 128-token blocks go end to end into the launch's activation
// planes (as many chunks per launch as fit the plan's context), so every
// weight tile streams once per launch for all of them; then each chunk's last
// token runs its LM head into logits[i].
static int prefill_chunks(mk_plan* p, const int32_t* tokens, const std::vector<PfChunk>& ch, void* kv,
                          float* logits, cudaStream_t st) {
  int rc;
  if ((rc = prefill_init(p)) != MK_OK || (rc = prefill_bind_kv(p, kv, st)) != MK_OK) return rc;
  const int V = p->hp.cfg.vocab;
  const int cap = p->pf.pp.n_blocks;  // token blocks one launch holds
  const int n = (int)ch.size();
  for (int c0 = 0; c0 < n;) {
    std::vector<int4> tab;
    int c1 = c0;
    while (c1 < n) {
      const int nb = (ch[c1].len + PF_BM - 1) / PF_BM;
      if (!tab.empty() && (int)tab.size() + nb > cap) break;
      const int first = (int)tab.size();
      for (int m = 0; m < nb; ++m)
        tab.push_back(make_int4(ch[c1].slot | (first << 16), ch[c1].pos0, ch[c1].len, ch[c1].tok));
      ++c1;
    }
    // (a pageable source: the copy has read it when the call returns)
    MK_CUDA(cudaMemcpyAsync(p->pf.d_blk, tab.data(), sizeof(int4) * tab.size(), cudaMemcpyHostToDevice,
                            st));
    PfParams k = p->pf.base;
    k.tokens = tokens;
    k.S = (int)tab.size() * PF_BM;
    k.blk = p->pf.d_blk;
    k.kv = (uint16_t*)kv;
    k.mode = MODE_MEGA;
    k.wait_limit_ns = p->wait_limit_ns;
    MK_CUDA(pf_launch_mega(k, p->n_sms, st));
    int blk0 = 0;
    for (int c = c0; c < c1; ++c) {
      const int row = blk0 * PF_BM + ch[c].len - 1;
      if ((rc = prefill_lm(p, tokens, row, kv, logits + (size_t)c * V, st)) != MK_OK) return rc;
      blk0 += (ch[c].len + PF_BM - 1) / PF_BM;
    }
    c0 = c1;
  }
  return MK_OK;
}

int mk_prefill_batch(mk_plan* p, const int32_t* tokens, const int32_t* lens, int batch, int stride,
                     void* kv, float* logits, void* stream) {
  if (!p || !tokens || !lens || !kv || !logits || batch < 1 || batch > p->max_batch ||
      stride < 1 || !aligned16(kv))
    return MK_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b)
    if (lens[b] < 1 || lens[b] > p->hp.max_ctx || lens[b] > stride) return MK_ERR_INVALID_ARG;
  if (p->latched) return p->latched;
  std::vector<PfChunk> ch(batch);
  for (int b = 0; b < batch; ++b) ch[b] = PfChunk{b, 0, lens[b], b * stride};
  return prefill_chunks(p, tokens, ch, kv, logits, (cudaStream_t)stream);
}

int mk_prefill_chunks(mk_plan* p, const int32_t* tokens, const int32_t* chunks, int n, void* kv,
                      float* logits, void* stream) {
  if (!p || !tokens || !chunks || !kv || !logits || n < 1 || !aligned16(kv)) return MK_ERR_INVALID_ARG;
  std::vector<PfChunk> ch(n);
  for (int i = 0; i < n; ++i) {
    ch[i] = PfChunk{chunks[4 * i], chunks[4 * i + 1], chunks[4 * i + 2], chunks[4 * i + 3]};
    const PfChunk& c = ch[i];
    if (c.slot < 0 || c.slot >= p->max_batch || c.pos0 < 0 || c.len < 1 || c.tok < 0 ||
        (long)c.pos0 + c.len > p->hp.max_ctx)
      return MK_ERR_INVALID_ARG;
    // a later chunk of the same slot continues the slot's previous chunk
    for (int j = i - 1; j >= 0; --j)
      if (ch[j].slot == c.slot) {
        if (ch[j].pos0 + ch[j].len != c.pos0) return MK_ERR_INVALID_ARG;
        break;
      }
  }
  if (p->latched) return p->latched;
  return prefill_chunks(p, tokens, ch, kv, logits, (cudaStream_t)stream);
}

int mk_prefill_logits(mk_plan* p, const int32_t* tokens, int len, void* kv, float* logits,
                      void* stream) {
  int rc = prefill_args(p, tokens, len, kv, logits);
  if (rc != MK_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = prefill_init(p)) != MK_OK || (rc = prefill_bind_kv(p, kv, st)) != MK_OK) return rc;
  PfParams k = p->pf.base;
  k.tokens = tokens;
  k.S = len;
  k.kv = (uint16_t*)kv;
  k.logits = logits;
  k.n_instr = (uint32_t)p->pf.pp.queue.size();  // the body, the final norms, the LM head
  const PfBars& bl = p->pf.pp.bl;
  MK_CUDA(cudaMemsetAsync(k.bars + bl.normf, 0, sizeof(uint32_t) * (bl.total - bl.normf), st));
  k.mode = MODE_MEGA;
  k.wait_limit_ns = p->wait_limit_ns;
  return cuda_err(pf_launch_mega(k, p->n_sms, st));
}

static int launch_per_op_seq(mk_plan* p, const KParams& k, cudaStream_t st) {
  for (const auto& r : p->hp.perop_decode) MK_CUDA(p->kv.perop(k, r.first, r.second, p->max_ctas, st));
  return MK_OK;
}

static int launch_per_op_bd(mk_plan* p, const BdParams& k, cudaStream_t st) {
  BdParams kk = k;
  kk.queue = p->bd.d_queue;  // per-operator ranges index the default order
  for (const auto& r : p->bd.bp.perop) MK_CUDA(bd_launch_perop(kk, r.first, r.second, st));
  return MK_OK;
}

static int launch_per_op_prefill(mk_plan* p, const PfParams& k, void* kv, float* logits,
                                 cudaStream_t st) {
  for (uint32_t j = 0; j < p->pf.pp.n_perop_body; ++j) {
    const auto& r = p->pf.pp.perop[j];
    MK_CUDA(pf_launch_perop(k, r.first, r.second, st));
  }
  return prefill_lm(p, k.tokens, k.S - 1, kv, logits, st);
}

int mk_run_per_op(mk_plan* p, int mode, int use_graph, const int32_t* tokens,
                  const int32_t* positions, int batch_or_len, void* kv, float* logits,
                  void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  PfParams pk;
  KParams k;
  BdParams bk;
  if (mode == MK_PREFILL) {
    int rc = prefill_args(p, tokens, batch_or_len, kv, logits);
    if (rc != MK_OK) return rc;
    if ((rc = prefill_init(p)) != MK_OK || (rc = prefill_bind_kv(p, kv, st)) != MK_OK) return rc;
    pk = p->pf.base;
    pk.tokens = tokens;
    pk.S = batch_or_len;
    pk.kv = (uint16_t*)kv;
    pk.wait_limit_ns = p->wait_limit_ns;
    if (!use_graph) return launch_per_op_prefill(p, pk, kv, logits, st);
  } else {
    if (mode != MK_DECODE) return MK_ERR_INVALID_ARG;
    int rc = check_step(p, tokens, positions, batch_or_len, kv, logits);
    if (rc != MK_OK) return rc;
    if (p->bd.on) {
      if ((rc = bd_bind_kv(p, kv, st)) != MK_OK) return rc;
      bk = bd_params(p, tokens, positions, batch_or_len, kv, logits);
      if (!use_graph) return launch_per_op_bd(p, bk, st);
    }
    k = step_params(p, tokens, positions, batch_or_len, kv, logits);
    k.queue = p->d_queue;
    k.trace = nullptr;
    if (!use_graph && !p->bd.on) return launch_per_op_seq(p, k, st);
  }
  const uintptr_t key[6] = {(uintptr_t)tokens, (uintptr_t)positions, (uintptr_t)batch_or_len,
                            (uintptr_t)kv, (uintptr_t)logits, (uintptr_t)mode};
  if (!p->graph || std::memcmp(key, p->graph_key, sizeof(key)) != 0) {
    if (p->graph) {
      cudaGraphExecDestroy(p->graph);
      p->graph = nullptr;
    }
    cudaGraph_t g = nullptr;
    MK_CUDA(cudaStreamBeginCapture(p->cap_stream, cudaStreamCaptureModeThreadLocal));
    int lrc = mode == MK_PREFILL ? launch_per_op_prefill(p, pk, kv, logits, p->cap_stream)
              : p->bd.on        ? launch_per_op_bd(p, bk, p->cap_stream)
                                : launch_per_op_seq(p, k, p->cap_stream);
    cudaError_t e = cudaStreamEndCapture(p->cap_stream, &g);
    if (lrc != MK_OK || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      return MK_ERR_CUDA;
    }
    e = cudaGraphInstantiate(&p->graph, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      p->graph = nullptr;
      return MK_ERR_CUDA;
    }
    std::memcpy(p->graph_key, key, sizeof(key));
  }
  return cuda_err(cudaGraphLaunch(p->graph, st));
}

int mk_status(mk_plan* p, void* stream) {
  if (!p) return MK_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MK_ERR_CUDA;
  uint32_t status = 0;
  if (cudaMemcpy(&status, p->d_ctl + CTL_STATUS, sizeof(status), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return MK_ERR_CUDA;
  if (!status && p->pf.built &&
      cudaMemcpy(&status, p->pf.base.ctl + CTL_STATUS, sizeof(status), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MK_ERR_CUDA;
  if (!status && p->bd.on &&
      cudaMemcpy(&status, p->bd.base.ctl + CTL_STATUS, sizeof(status), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MK_ERR_CUDA;
  if (status) p->latched = (int)status;
  return (int)status;
}

int mk_plan_reset(mk_plan* p, void* stream) {
  if (!p) return MK_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
  MK_CUDA(cudaMemset(p->base.bars, 0, sizeof(uint32_t) * p->hp.bl.total));
  MK_CUDA(cudaMemset(p->d_ctl, 0, sizeof(uint32_t) * CTL_WORDS));
  // the launch counter restarts at 0: clear every tagged word, so that no
  // stale word carries a tag a later launch expects
  MK_CUDA(cudaMemset(p->scratch, 0, p->tagged_bytes));
  if (p->pf.built) {
    MK_CUDA(cudaMemset(p->pf.base.bars, 0, sizeof(uint32_t) * p->pf.pp.bl.total));
    MK_CUDA(cudaMemset(p->pf.base.ctl, 0, sizeof(uint32_t) * CTL_WORDS));
  }
  if (p->bd.on) {
    MK_CUDA(cudaMemset(p->bd.base.bars, 0, sizeof(uint32_t) * p->bd.bp.bl.total));
    MK_CUDA(cudaMemset(p->bd.base.ctl, 0, sizeof(uint32_t) * CTL_WORDS));
    MK_CUDA(cudaMemset(p->bd.base.arrive, 0, sizeof(uint32_t) * p->bd.arrive_words));
  }
  MK_CUDA(cudaDeviceSynchronize());
  p->latched = 0;
  return MK_OK;
}

int mk_plan_set_debug(mk_plan* p, int force_ctas, uint64_t queue_perm_seed, int trace,
                      uint64_t wait_limit_ns) {
  if (!p || force_ctas < 0 || force_ctas > p->max_ctas) return MK_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MK_ERR_CUDA;
  p->force_ctas = force_ctas;
  p->wait_limit_ns = wait_limit_ns ? wait_limit_ns : 2000000000ull;
  int rc = p->bd.on ? bd_upload_queue(p, queue_perm_seed) : upload_mk_queue(p, queue_perm_seed);
  if (rc != MK_OK) return rc;
  const size_t n_rec = p->bd.on ? p->bd.bp.queue.size() : p->hp.decode.size();
  if (trace && !p->d_trace) {
    if (cudaMalloc(&p->d_trace, n_rec * TRACE_WORDS * 8) != cudaSuccess) return MK_ERR_CUDA;
    MK_CUDA(cudaMemset(p->d_trace, 0, n_rec * TRACE_WORDS * 8));
  }
  p->trace = trace ? 1 : 0;
  return MK_OK;
}

int mk_plan_debug_drop_release(mk_plan* p, uint32_t index) {
  if (!p || index >= p->hp.decode.size()) return MK_ERR_INVALID_ARG;
  if (p->bd.on) return MK_ERR_UNSUPPORTED;
  Instr in;
  MK_CUDA(cudaDeviceSynchronize());
  MK_CUDA(cudaMemcpy(&in, p->d_queue_mk + index, sizeof(Instr), cudaMemcpyDeviceToHost));
  in.flags |= IF_NO_PUBLISH;
  MK_CUDA(cudaMemcpy(p->d_queue_mk + index, &in, sizeof(Instr), cudaMemcpyHostToDevice));
  return MK_OK;
}

int mk_trace_copy(mk_plan* p, void* host_buf, size_t bytes, size_t* n_records) {
  if (!p || !host_buf || !n_records) return MK_ERR_INVALID_ARG;
  *n_records = 0;
  if (!p->d_trace) return MK_ERR_INVALID_ARG;
  MK_CUDA(cudaDeviceSynchronize());
  size_t n = p->bd.on ? p->bd.bp.queue.size() : p->hp.decode.size();
  if (bytes / (TRACE_WORDS * 8) < n) n = bytes / (TRACE_WORDS * 8);
  MK_CUDA(cudaMemcpy(host_buf, p->d_trace, n * TRACE_WORDS * 8, cudaMemcpyDeviceToHost));
  *n_records = n;
  return MK_OK;
}

}  // extern "C"
