// Prefill: the causal forward pass of one prompt as one persistent launch of
// tensor-core tiles with tile-level dependencies (the MegaOps Abstract's
// per-tile synchronisation, here between GEMM -> attention -> GEMM tiles of
// 128-token blocks; "Lecture 112: Production Megakernels for Real-World
// Inference", Key takeaways: barriers partitioned along the dependency
// dimensions so consumers start before all producers finish).
#pragma once
#include <stdint.h>

#include <string>
#include <utility>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"

namespace mk {

// Prefill opcodes (disjoint from the decode ones).
enum PfOp : uint8_t {
  PF_NORM1 = 16,  // RMSNorm of a 128-token block before attention   (a0 = block)
  PF_QKV = 17,    // [q|k|v] columns n of a block, RoPE, K/V to cache  (a0 = block, a1 = n)
  PF_ATTN = 18,   // causal attention of a block for one kv group      (a0 = block, a1 = kv head)
  PF_O = 19,      // O columns n of a block + residual                  (a0 = block, a1 = n)
  PF_NORM2 = 20,  // RMSNorm of a block before the FFN                  (a0 = block)
  PF_GU = 21,     // gate/up columns n (128 + 128) of a block, SwiGLU   (a0 = block, a1 = n)
  PF_DOWN = 22,   // down columns n of a block + residual               (a0 = block, a1 = n)
  PF_NORMF = 23,  // final RMSNorm of a block (all-token logits only)    (a0 = block)
  PF_LM = 24,     // LM-head columns n of a block -> f32 logits         (a0 = block, a1 = n)
};

constexpr int PF_BM = 128;   // tokens per block (tcgen05 M)
constexpr int PF_BK = 64;    // reduction depth per ring stage (one 128-byte swizzle atom)
constexpr int PF_BN = 256;   // output features per GEMM tile (tcgen05 N)
constexpr int PF_BN_GU = 128;  // gate/up features per tile (x2 matrices = N 256)

// Expression slot of prefill: S - a0 * PF_BM (> 0: the token block is live).
constexpr int PXS_BLOCK_LIVE = 0;
constexpr int PF_BLOCK_GROUP = 8;  // most token blocks that share each weight tile in the queue order
constexpr int PXS_COUNT = 1;

// Barrier sub-tensors, each [L][n_blocks]; normf and lm are [n_blocks].
struct PfBars {
  uint32_t norm1, qkv, attn, o, norm2, gu, down, normf, lm, total;
};

struct PrefillPlan {
  mk_model_cfg cfg{};
  int max_ctx = 0, n_blocks = 0, rep = 0, qkv_rows = 0;
  int bn_qkv = 0;  // 256, or 128 when a head group does not fill 256 columns
  uint32_t n_qkv_n = 0, n_o_n = 0, n_gu_n = 0, n_down_n = 0, n_lm_n = 0;
  PfBars bl{};
  // queue[0, n_body): the prompt's layers; queue[n_body, size): the final
  // norm and the LM head of every token (run only for all-token logits)
  uint32_t n_body = 0, n_perop_body = 0;  // (and the per-operator ranges of the body)
  std::vector<Instr> queue;                                // topological
  std::vector<std::pair<uint32_t, uint32_t>> perop;        // (first, count) per launch
  std::vector<uint32_t> expr;                              // PXS_COUNT * X_MAX_WORDS
};

// Tensor-map table (in device memory): per layer l, 8 maps at l * 8 + TM_*;
// then the activation maps at L * 8 + AM_*.
enum PfWeightMap { TM_WQ = 0, TM_WK = 1, TM_WV = 2, TM_WO = 3, TM_WG = 4, TM_WU = 5, TM_WD = 6,
                   TM_PER_LAYER = 8 };
enum PfActMap { AM_HN1 = 0, AM_HN2 = 1, AM_AO = 2, AM_ACT = 3, AM_KV = 4, AM_LMW = 5, AM_COUNT = 6 };

// Everything one prefill launch needs (passed by value).
struct PfParams {
  int L, H, nq, nkv, d, F, V, qk_norm, rep, qkv_rows, bn_qkv, n_blocks, max_ctx, max_batch;
  float eps;
  uint32_t n_qkv_n, n_o_n, n_gu_n, n_down_n;
  const uint16_t* embed;
  const uint16_t* final_norm;
  float* logits;            // all-token logits [S][V] (PF_LM tiles), or null
  const LayerW* layers;     // device array [L]
  const void* tm;           // CUtensorMap table (64-byte aligned)
  float* xa;                // residual after attention, f32 [rows][H]
  float* xb;                // residual after the FFN, f32 [rows][H]
  // Tensor-core operands carried as two bf16 planes, [2][rows][cols]: the
  // nearest bf16 (hi) and the bf16 of the remainder (lo), so hi + lo holds
  // ~16 significant bits and an MMA pair (hi, lo) against the exact bf16
  // weights keeps the activation's float32 precision.
  uint16_t* hn1;            // RMSNorm outputs [2][rows][H]
  uint16_t* hn2;
  uint16_t* qb;             // rotated queries [2][rows][n_q * d]
  uint16_t* ao;             // attention outputs [2][rows][n_q * d]
  uint16_t* act;            // SwiGLU outputs [2][rows][F]
  int plane_rows;           // rows of one plane (token blocks x 128)
  uint16_t* kv;             // caller's KV cache
  int slot;                 // the sequence slot this prompt's keys and values go to
  // Several prompts or chunks in one launch (mk_prefill_batch,
  // mk_prefill_chunks): their 128-token blocks lie end to end in the
  // activation planes, and block j of the launch is described by
  // blk[j] = {cache slot | the chunk's first block << 16, the chunk's first
  // position, its length, its first token's offset in `tokens`}; S = the
  // blocks x 128.  Null for one prompt (slot `slot`, positions from 0, block j
  // = the prompt's block j, length S).
  const int4* blk;
  const float2* rope;       // (cos, sin) [max_ctx][d / 2]
  uint32_t* bars;
  uint32_t* ctl;
  const Instr* queue;
  uint32_t n_instr;
  // the plan's expressions [PXS_COUNT][X_MAX_WORDS], in the launch's parameter
  // block (read through the constant cache on the producer's path)
  uint32_t xw[PXS_COUNT * X_MAX_WORDS];
  const int32_t* tokens;
  int S;
  int mode;
  uint32_t perop_base;
  unsigned long long wait_limit_ns;
};
static_assert(sizeof(PfParams) <= 4096, "kernel parameter block limit");

int build_prefill(const mk_model_cfg& cfg, int max_ctx, PrefillPlan* out, std::string* why);
int simulate_prefill(const PrefillPlan& pp, const std::vector<Instr>& q, std::string* why);

}  // namespace mk
