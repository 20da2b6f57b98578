// Batched decode on the tensor cores: one decode step for up to BD_NMAX
// sequences as one persistent launch of tile instructions with tile-level
// dependencies (the MegaOps Abstract's per-tile synchronisation; "Lecture 112:
// Production Megakernels for Real-World Inference", Technical details: an
// on-device interpreter popping instructions from a queue in DRAM).
//
// Per layer:
//   QKV(m, c) -> ATTN(b, g, s) -> O(m, c) -> GU(m, c) -> DOWN(m, c)
// then LM(m) after the last layer (NORM1(r) before layer 0 only).  The RMSNorms
// are folded into the GEMMs next to them: an O or down tile also writes its
// columns of x * gain (the next norm's input times its gain) and the tile's
// sums of x^2 per sequence; the next projection multiplies x * gain by the
// weights and scales its outputs by 1 / rms, which the projection's linearity
// in each row makes equal to projecting the normed row.  GEMM tiles put 128 weight
// rows (m) on the tcgen05 M side and the batch (padded to N = 16 or 32
// columns) on the N side, over one K chunk (c) of at most BD_KC columns; the
// last chunk of a row tile to arrive adds the chunks' partial sums in chunk
// order and runs the epilogue (RoPE + K/V cache write, residual adds, SwiGLU,
// logits).  Activation operands are split into bf16 hi + lo planes (two MMAs
// per k-step), so every product keeps float32-level precision.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"

namespace mk {

enum BdOp : uint8_t {
  BD_NORM1 = 40,  // layer-0 RMSNorm input of sequences [8 r, 8 r + 8)  (a0 = r)
  BD_QKV = 41,    // [q|k|v] rows [128 m, +128) over K chunk c            (a0 = m, a1 = c)
  BD_ATTN = 42,   // split s of (sequence b, kv head g)                   (a0 = b, a1 = g, a2 = s)
  BD_O = 43,      // O rows of row tile m, chunk c; + residual
  BD_NORM2 = 44,  // RMSNorm(ffn)
  BD_GU = 45,     // 64 gate + 64 up rows of tile m, chunk c; SwiGLU
  BD_DOWN = 46,   // down rows; + residual
  BD_NORMF = 47,  // final RMSNorm
  BD_LM = 48,     // LM-head rows
};

constexpr int BD_M = 128;       // weight rows per GEMM tile (tcgen05 M)
constexpr int BD_BK = 64;       // reduction depth per ring stage (one 128-byte swizzle atom)
constexpr int BD_NMAX = 32;     // most sequences per step (tcgen05 N)
constexpr int BD_KC = 1024;     // K chunk of a split-K tile
constexpr int BD_RG = 8;        // sequences per RMSNorm instruction (one compute warp each)
constexpr int BD_KEYS = 128;    // cached keys per attention block (K in one ring stage, V in the next)
constexpr int BD_NSPLIT_MAX = 8;  // attention splits per (sequence, kv head), at most
// a sequence of n keys uses min(nsplit, ceil(n / BD_SPLIT_KEYS)) of its splits
constexpr int BD_SPLIT_KEYS = 512;

// Barrier sub-tensors: one counter per layer and operator.
struct BdBars {
  uint32_t norm1, qkv, attn, o, norm2, gu, down, normf, lm, total;
};

struct BdPlan {
  mk_model_cfg cfg{};
  int max_batch = 0, max_ctx = 0, nb = 0;  // nb: batch columns (16 or 32)
  int nsplit = 0;  // attention splits per (sequence, kv head)
  int rep = 0, qkv_rows = 0, n_rg = 0;
  uint32_t n_qkv_m = 0, n_o_m = 0, n_gu_m = 0, n_down_m = 0, n_lm_m = 0;  // row tiles
  uint32_t c_h = 0, c_q = 0, c_f = 0;  // K chunks for K = H, n_q*d, F
  uint32_t c_g = 0;  // K chunks of the gate/up projection (2048 columns each where H allows)
  uint32_t c_k = 0;  // K chunks of the QKV projection (512 columns each where H allows)
  BdBars bl{};
  std::vector<Instr> queue;                                // topological
  std::vector<std::pair<uint32_t, uint32_t>> perop;        // (first, count) per launch
};

// Tensor maps (device table): per layer l at l * BD_TM_PER_LAYER + TMB_*;
// then the LM head and the activation maps at L * BD_TM_PER_LAYER + TMB_*.
enum BdMap { TMB_WQ = 0, TMB_WK = 1, TMB_WV = 2, TMB_WO = 3, TMB_WG = 4, TMB_WU = 5, TMB_WD = 6,
             BD_TM_PER_LAYER = 8 };
enum BdGlobalMap { TMB_LM = 0, TMB_HN = 1, TMB_AO = 2, TMB_ACT = 3, TMB_KV = 4, TMB_COUNT = 5 };

struct BdParams {
  int L, H, nq, nkv, d, F, V, qk_norm, rep, qkv_rows, max_ctx, max_batch, nb, n_rg, nsplit;
  float eps;
  uint32_t n_qkv_m, n_o_m, n_gu_m, n_down_m, n_lm_m, c_h, c_q, c_f, c_g, c_k;
  const uint16_t* embed;
  const uint16_t* final_norm;
  const LayerW* layers;     // device array [L]
  const void* tm;           // CUtensorMap table (64-byte aligned)
  float* xa;                // residual after attention [nb][H]
  float* xb;                // residual after the FFN [nb][H]
  uint16_t* hn;             // RMSNorm output, hi/lo planes [2][nb][H]
  uint16_t* ao;             // attention output, hi/lo planes [2][nb][n_q d]
  uint16_t* act;            // SwiGLU output, hi/lo planes [2][nb][F]
  float* q;                 // rotated (normed) queries [nb][n_q d]
  float* ss1;               // sums of x^2 per (row tile, sequence) for the next QKV / LM [tiles][BD_NMAX]
  float* ss2;               // the same for the gate/up projection [tiles][BD_NMAX]
  // split-K partial sums [slot = row tile x chunks + chunk][BD_NMAX][128] in
  // two regions that operators alternate between: O and down in the first,
  // QKV and gate/up in the second from slot part_b.  A chunk may start while
  // the previous operator's row tiles are still summing their chunks (its
  // wait covers only the tiles it reads), never while the one before that
  // is, so neighbours must not share a region.
  float* part;
  uint32_t part_b;
  float* apart;             // attention split partials [max_batch][n_kv][nsplit][rep][d + 2]
  // arrival counters: row tiles of the first region's operator, of the
  // second's from arrive_b, then [max_batch * n_kv] attention groups from
  // n_arrive_gemm
  uint32_t* arrive;
  uint32_t arrive_b;
  uint32_t n_arrive_gemm;
  uint16_t* kv;             // caller's KV cache
  const float2* rope;       // (cos, sin) [max_ctx][d / 2]
  uint32_t* bars;
  uint32_t* ctl;
  const Instr* queue;
  uint32_t n_instr;
  const int32_t* tokens;
  const int32_t* positions;
  const int32_t* slots;     // [B] cache slot of each column, or null (column b uses slot b)
  float* logits;            // [B][V]
  int B;
  int mode;
  uint32_t perop_base;
  unsigned long long wait_limit_ns;
  // TRACE_WORDS x u64 per instruction (queue index), or null: [0] smid | (op |
  // layer << 8) << 32, [1] compute warps took it, [2] inputs ready (GEMM:
  // accumulator full; attention / norm: dependencies met), [3] done, [4]
  // producer posted it, [5] producer's dependency wait met, [6] producer
  // issued its last stage, [7] first MMA issued, [8] last MMA committed;
  // attention splits: [9] first key block ready, [10] last key block done.
  unsigned long long* trace;
};

// Shapes the tensor-core batched path takes (MK_OK) or why not.
// n_sms: SMs of the device (not used: the attention split count is fixed).
int build_bdecode(const mk_model_cfg& cfg, int max_batch, int max_ctx, int n_sms, BdPlan* out,
                  std::string* why);
int simulate_bdecode(const BdPlan& bp, const std::vector<Instr>& q, std::string* why);
void random_order_bdecode(const BdPlan& bp, uint64_t seed, std::vector<Instr>* out);

// Device side (mk_bdecode_kernel.cu).
cudaError_t bd_setup();
cudaError_t bd_launch_mega(const BdParams& p, int ctas, cudaStream_t st);
cudaError_t bd_launch_perop(const BdParams& p, uint32_t first, uint32_t count, cudaStream_t st);

}  // namespace mk
