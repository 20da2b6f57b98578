// mk_decode_step_noalloc: one decode step that never allocates device memory.
//
// Who needs it: callers that cannot call cudaMalloc at the moment they run a
// step -- e.g. a serving process that hands (nearly) all device memory to its
// own pool and KV cache up front, or code running under an external memory
// manager that forbids new device allocations.  They still own and pass the
// weights, the KV cache, tokens, positions and logits; everything else the
// step needs (activations, split-KV partials, barrier counters, the
// instruction queue, the RoPE table) lives in one file-scope device array of
// fixed size that the library image carries.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"
#include "mk_plan.h"
#include "mk_variants.h"

namespace mk {
namespace {

// The static scratch.  Every GPU that loads this library holds it until the
// process exits.  Every call shares it and finds the previous call's contents.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
uint8_t* g_scratch_addr[kMaxDevices] = {nullptr};  // device address of the array, per device

KernelVariant variant_for(const HostPlan& hp) {
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

bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

// The host-side work of a call depends only on (shape, max_batch, max_ctx,
// SM count): the plan build and the RoPE table are kept from the previous call
// with the same key, and the queue, bytecode and RoPE table are copied into
// the static array only when the array does not already hold them (calls are
// serialised by contract, so the last upload per device is what it holds).
struct NoallocKey {
  mk_model_cfg cfg;
  int max_batch, max_ctx, sms;
  bool same(const NoallocKey& o) const {
    return std::memcmp(&cfg, &o.cfg, sizeof(cfg)) == 0 && max_batch == o.max_batch &&
           max_ctx == o.max_ctx && sms == o.sms;
  }
};
struct NoallocHost {
  bool valid = false;
  NoallocKey key{};
  HostPlan hp;
  std::vector<float2> rope;
};
std::mutex g_mu;
NoallocHost g_host;                            // last plan built (any device)
NoallocKey g_resident[kMaxDevices];            // the shape each device's array holds
bool g_resident_valid[kMaxDevices] = {false};
std::vector<LayerW> g_resident_lw[kMaxDevices];  // the layer table it holds

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" int mk_decode_step_noalloc(const mk_model_cfg* cfg, const mk_weight_ptrs* w,
                                      int max_batch, int max_ctx, const int32_t* tokens,
                                      const int32_t* positions, int batch, void* kv_cache,
                                      float* logits, void* stream) {
  if (!cfg || !w || !tokens || !positions || !kv_cache || !logits) return MK_ERR_INVALID_ARG;
  if (batch < 1 || batch > max_batch || !al16(kv_cache)) return MK_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  // The copies below read host memory that this library owns and rewrites: a
  // captured graph would replay them later, so a capturing stream is refused.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return MK_ERR_INVALID_ARG;
  int cur = 0, sms = 0;
  if (cudaGetDevice(&cur) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, cur) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  NoallocKey key;
  std::memset(&key, 0, sizeof(key));
  key.cfg = *cfg;
  key.max_batch = max_batch;
  key.max_ctx = max_ctx;
  key.sms = sms;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_host.valid || !g_host.key.same(key)) {
    g_host.valid = false;
    std::string why;
    const int rc = build_plan(*cfg, max_batch, max_ctx, sms, &g_host.hp, &why);
    if (rc != MK_OK) return rc;
    if (decode_scratch(g_host.hp).total > (size_t)MK_NOALLOC_SCRATCH_BYTES)
      return MK_ERR_UNSUPPORTED;  // before the RoPE table is computed
    const int hd = g_host.hp.cfg.head_dim;
    g_host.rope.assign((size_t)max_ctx * (hd / 2), make_float2(0.f, 0.f));
    for (int pos = 0; pos < max_ctx; ++pos)
      for (int i = 0; i < hd / 2; ++i) {
        const double a = (double)pos * std::pow((double)g_host.hp.cfg.rope_theta, -2.0 * i / hd);
        g_host.rope[(size_t)pos * (hd / 2) + i] =
            make_float2((float)std::cos(a), (float)std::sin(a));
      }
    g_host.key = key;
    g_host.valid = true;
  }
  const HostPlan& hp = g_host.hp;
  const mk_model_cfg& c = hp.cfg;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, F = c.ffn, nkv = c.n_kv_heads;
  std::vector<LayerW> lw(L);
  bool good = al16(w->embed) && al16(w->final_norm) && (c.tied_embeddings || al16(w->lm_head)) &&
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
    good = al16(x.attn_norm) && al16(x.wq) && al16(x.wk) && al16(x.wv) && al16(x.wo) &&
           al16(x.ffn_norm) && al16(x.wg) && al16(x.wu) && al16(x.wd) &&
           (!c.qk_norm || (al16(x.q_norm) && al16(x.k_norm)));
  }
  if (!good) return MK_ERR_INVALID_ARG;

  // Carve the static array: the decode layout a plan allocates (one queue copy).
  const DecodeScratch ds = decode_scratch(hp);
  if (ds.total > (size_t)MK_NOALLOC_SCRATCH_BYTES) return MK_ERR_UNSUPPORTED;
  const size_t o_q = ds.o_q, o_rope = ds.o_rope, o_lw = ds.o_lw;

  // Per-device set-up on the first call with that device current: the array's
  // device address and the kernel's shared-memory attribute.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MK_ERR_CUDA;
  const KernelVariant kv = variant_for(hp);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MK_ERR_CUDA;
    g_scratch_addr[dev] = (uint8_t*)ptr;
  }
  if (kv.setup() != cudaSuccess) return MK_ERR_CUDA;
  int nsm = 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MK_ERR_CUDA;
  uint8_t* s = g_scratch_addr[dev];

  // The queue, bytecode and RoPE table go in only when this device's array
  // holds another shape's (pageable copies return once the source is read),
  // the layer table only when the weights moved.  Every call clears the tagged
  // intermediate tensors, the counters and the control words: the launch
  // counter restarts at 0, so no word left by an earlier call, of any shape,
  // carries a tag this call expects.
  const std::vector<float2>& rope = g_host.rope;
  if (!(g_resident_valid[dev] && g_resident[dev].same(key))) {
    g_resident_valid[dev] = false;
    g_resident_lw[dev].clear();
    if (cudaMemcpyAsync(s + o_q, hp.decode.data(), sizeof(Instr) * hp.decode.size(),
                        cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(s + o_rope, rope.data(), sizeof(float2) * rope.size(),
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MK_ERR_CUDA;
    g_resident[dev] = key;
    g_resident_valid[dev] = true;
  }
  if (g_resident_lw[dev].size() != lw.size() ||
      std::memcmp(g_resident_lw[dev].data(), lw.data(), sizeof(LayerW) * lw.size()) != 0) {
    g_resident_lw[dev].clear();
    if (cudaMemcpyAsync(s + o_lw, lw.data(), sizeof(LayerW) * L, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
      return MK_ERR_CUDA;
    g_resident_lw[dev] = lw;
  }
  if (cudaMemsetAsync(s, 0, ds.zero_end, st) != cudaSuccess) return MK_ERR_CUDA;

  KParams k;
  std::memset(&k, 0, sizeof(k));
  k.L = L; k.H = H; k.nq = c.n_q_heads; k.nkv = nkv; k.d = d; k.F = F; k.V = c.vocab;
  k.qk_norm = c.qk_norm; k.rep = hp.rep; k.qkv_rows = hp.qkv_rows; k.eps = c.rms_eps;
  k.max_batch = max_batch; k.max_ctx = max_ctx; k.n_splits = hp.n_splits;
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
  k.ctl = (uint32_t*)(s + ds.o_ctl);
  k.queue = (const Instr*)(s + o_q);
  k.n_instr = (uint32_t)hp.decode.size();
  std::memcpy(k.xw, hp.expr.data(), sizeof(k.xw));
  k.bl = hp.bl;
  k.tokens = tokens;
  k.positions = positions;
  k.B = batch;
  k.kv = (uint16_t*)kv_cache;
  k.logits = logits;
  k.mode = MODE_MEGA;
  k.wait_limit_ns = 2000000000ull;
  k.n_steps = 1;
  return kv.mega(k, nsm, st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}
