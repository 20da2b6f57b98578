// Internal layout shared by the host plan builder and the device interpreter.
//
// The instruction queue, barrier tensor and symbolic-extent expressions follow
// "Lecture 112: Production Megakernels for Real-World Inference" (Technical
// details: an interpreter loop pops fixed-size instructions from a queue in
// DRAM; Key takeaways: barriers are tensors partitioned along the dependency
// dimensions, and extents are expressions in S and P so the queue is built
// once) and the MegaOps Abstract (a consumer waits on the tiles of the
// intermediate tensor it reads, not on the producer kernel).
#pragma once
#include <stdint.h>
#include <vector_types.h>

#ifdef __CUDACC__
#define MK_HD __host__ __device__ __forceinline__
#else
#define MK_HD inline
#endif

namespace mk {

typedef unsigned long long u64;  // a tagged word (mk_device.cuh)

// ---------------------------------------------------------------- opcodes
enum Op : uint8_t {
  OP_NOP = 0,
  OP_QKV = 1,   // rows of [Wq;Wk;Wv] . rmsnorm(x)               (a0 = row0, a1 = rows)
  OP_ATTN = 2,  // split-KV decode attention                      (a0 = seq, a1 = kv head, a2 = split)
  OP_O = 3,     // rows of Wo . attn + residual                  (a0 = row0, a1 = rows)
  OP_GU = 4,    // rows of Wg, Wu . rmsnorm(x), SwiGLU            (a0 = row0, a1 = rows)
  OP_DOWN = 5,  // rows of Wd . act + residual                   (a0 = row0, a1 = rows)
  OP_LM = 6,    // rows of W_lm . rmsnorm(x)                      (a0 = row0, a1 = rows)
  OP_COUNT = 7
};

constexpr uint32_t NO_BAR = 0xffffffffu;
constexpr uint8_t NO_EXPR = 0xff;

// Instruction flags.
// Decode attention: this instruction combines the splits of its (sequence, kv
// head) group (it follows every split of the group in every topological
// order: it waits on their partials).  Alone, the flag marks a group's only
// split, which combines its own partial; with IF_SLICE the instruction holds
// no keys and combines output slice a2 (comb_per outputs each).
constexpr uint8_t IF_COMBINE = 1;
constexpr uint8_t IF_SLICE = 8;
// The waited counter is cleared before every launch that runs this
// instruction (it is not released by every launch): absolute target.
constexpr uint8_t IF_ABS_TARGET = 2;
// Test-only fault injection (decode interpreter): the instruction stores its
// outputs under a tag no reader expects, so its consumers' bounded waits run
// out.
constexpr uint8_t IF_NO_PUBLISH = 4;

// One queue record, 32 bytes.
struct Instr {
  uint8_t op, flags;
  uint16_t layer;
  uint32_t a0, a1;
  uint16_t a2;
  uint8_t x_lo, x_hi;    // symbolic extent [lo, hi) expressions (NO_EXPR: none)
  uint32_t wait_bar;     // first waited barrier, or NO_BAR
  uint32_t wait_target;  // releases per step expected on each waited barrier
  uint16_t wait_n;       // number of barriers waited on
  uint16_t wait_stride;  // index stride between them
  uint32_t rel_bar;      // barrier this instruction releases (+1), or NO_BAR
};
static_assert(sizeof(Instr) == 32, "instruction record must stay 32 bytes");

// ---------------------------------------------------------------- symbolic extents
// Tiny postfix bytecode over the runtime variables.  Word = op << 24 | imm24.
enum XOp : uint32_t {
  X_END = 0, X_CONST = 1, X_ARG0 = 2, X_ARG1 = 3, X_ARG2 = 4,
  X_B = 5,    // runtime batch
  X_S = 6,    // runtime prompt length
  X_POS = 7,  // pop b, push positions[b]
  X_ADD = 8, X_SUB = 9, X_MUL = 10, X_CEILDIV = 11, X_MIN = 12, X_MAX = 13
};
constexpr int X_MAX_WORDS = 32;  // words per expression slot
constexpr int X_STACK = 4;  // evaluation stack depth (x_eval; checked when a plan is built)

MK_HD uint32_t xw(uint32_t op, uint32_t imm = 0) { return (op << 24) | (imm & 0xffffffu); }

// Evaluate expression `e` (X_MAX_WORDS words).  `pos` may be null when the
// expression does not read positions; X_POS reads pos[b] + pos_add (the step
// index of a multi-step launch), or `known_pos` + pos_add without a load when
// b == known_b (a position the caller already holds).  Out-of-range positions
// evaluate as 0; the caller validates them separately.
MK_HD int64_t x_eval(const uint32_t* e, const Instr& in, int B, int S, const int32_t* pos,
                     int n_pos, int pos_add = 0, int known_b = -1, int known_pos = 0) {
  // 32-bit values (extents and positions stay below 2^24) in X_STACK
  // registers (a shift register) rather than a local array: on the device a
  // dynamically indexed array goes to local memory, whose round trips under
  // load made an evaluation take microseconds.
  int32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
  int sp = 0;
  for (int i = 0; i < X_MAX_WORDS; ++i) {
    const uint32_t w = e[i];
    const uint32_t op = w >> 24;
    const int32_t imm = (int32_t)(w & 0xffffffu);
    if (op == X_END) break;
    if (op <= X_S) {  // a push
      const int32_t v = op == X_CONST  ? imm
                        : op == X_ARG0 ? (int32_t)in.a0
                        : op == X_ARG1 ? (int32_t)in.a1
                        : op == X_ARG2 ? (int32_t)in.a2
                        : op == X_B    ? (int32_t)B
                                       : (int32_t)S;
      s3 = s2; s2 = s1; s1 = s0; s0 = v;
      ++sp;
    } else if (op == X_POS) {  // top b -> positions[b]
      const int32_t b = s0;
      s0 = b == known_b && b >= 0 ? (int32_t)known_pos + pos_add
           : (pos && b >= 0 && b < n_pos) ? (int32_t)pos[b] + pos_add : 0;
    } else {  // a binary operator: second from top (x) op top (y)
      const int32_t y = s0, x = s1;
      int32_t r = 0;
      if (op == X_ADD) r = x + y;
      else if (op == X_SUB) r = x - y;
      else if (op == X_MUL) r = x * y;
      else if (op == X_CEILDIV) r = y > 0 ? (x + y - 1) / y : 0;
      else if (op == X_MIN) r = x < y ? x : y;
      else if (op == X_MAX) r = x > y ? x : y;
      s0 = r; s1 = s2; s2 = s3;
      --sp;
    }
  }
  return sp > 0 ? s0 : 0;
}

// Expression slots used by the plan.
enum XSlot : uint8_t {
  XS_ATTN_LO = 0,  // first key of split a2 of sequence a0: min(a2 * KPS, P + 1)
  XS_ATTN_HI = 1,  // one past its last key: min((a2 + 1) * KPS, P + 1)
  XS_SEQ_LIVE = 2, // B - a0  (> 0: sequence a0 is part of this step)
  XS_COUNT = 3
};

// ---------------------------------------------------------------- barrier tensor layout
// One flat uint32 array.  Decode sub-tensors (all per layer):
//   qkv[L][n_kv]   : QKV row tiles of kv group g (its q heads, k_g, v_g) done
//   split[L][max_batch][n_kv] : the splits of a (sequence, kv group) other
//                    than its combining split done
//   attn[L]        : (sequence, kv group) attention outputs combined
//   o[L]           : O-projection row tiles done (residual x1 complete when full)
//   gu[L]          : gate/up row tiles done (SwiGLU activations complete)
//   down[L]        : down-projection row tiles done (residual x2 complete)
//   lm[1]          : LM-head row tiles done
struct BarLayout {
  uint32_t qkv, split, attn, o, gu, down, lm, total;
};

// Control words (device uint32 array).
enum Ctl : int {
  CTL_HEAD = 0,     // next queue index to pop
  CTL_EXIT = 1,     // CTAs that left the loop this launch
  CTL_GEN = 2,      // completed persistent launches (barrier generation)
  CTL_ABORT = 3,    // nonzero: every CTA stops popping
  CTL_STATUS = 4,   // first latched error code
  CTL_DETAIL = 5,   // instruction index / value that raised it
  CTL_WORDS = 8
};

// Per-layer weight pointers as the device sees them.
struct LayerW {
  const uint16_t *attn_norm, *wq, *wk, *wv, *wo, *q_norm, *k_norm, *ffn_norm, *wg, *wu, *wd;
};

enum Mode : int { MODE_MEGA = 0, MODE_PEROP = 1 };

// Trace record (u64 words) per instruction, indexed by queue position:
// [0] smid | (op | layer << 8) << 32, [1] consumer took it, [2] its waits were
// satisfied, [3] done (released), [4] producer posted it, [5] ns the consumer
// spent waiting for ring stages, [6] first stage available, [7] ns the producer
// spent waiting for free ring stages while streaming it, [8] (batch-1 GEMV)
// last stage consumed and the tile handed to the finisher warp, [9] (batch-1
// GEMV) the finisher took it; for attention tiles [8]..[11] mark its phases
// (inputs rotated, scores, softmax and P V, split arrival).  For handed-off
// tiles [3] is written by the finisher after its release.
constexpr int TRACE_WORDS = 16;

// Everything one launch needs, passed by value as a __grid_constant__ parameter.
struct KParams {
  // shape
  int L, H, nq, nkv, d, F, V, qk_norm, rep, qkv_rows;
  float eps;
  int max_batch, max_ctx, n_splits;
  // tiling
  int r_qkv, r_o, r_gu, r_down, r_lm;
  uint32_t n_qkv_tiles, n_o_tiles, n_gu_tiles, n_down_tiles, n_lm_tiles;
  // weights
  const uint16_t *embed, *lm, *final_norm;
  const LayerW* layers;
  // plan-owned scratch: the intermediate tensors are tagged words (the float
  // and the tag of the launch step that wrote it; see mk_device.cuh)
  u64* resid;     // [2L+1][max_batch][H]
  u64* qkv;       // [L][max_batch][qkv_rows]
  u64* part;      // [L][max_batch][nkv][n_splits][rep][d+2]
  u64* attn_out;  // [L][max_batch][nq*d]
  u64* act;       // [L][max_batch][F]
  int kps;          // keys per attention split (a model constant)
  int comb_per;     // outputs per combine slice (rep * d / the plan's slices, rounded up)
  uint32_t* bars;   // barrier tensor (host simulation; the kernel reads tags)
  const float2* rope;  // [max_ctx][d/2] (cos, sin)
  uint32_t* ctl;
  const Instr* queue;
  uint32_t n_instr;
  // the plan's expressions [XS_COUNT][X_MAX_WORDS], held in the launch's
  // parameter block: the producer evaluates them for every attention
  // instruction it pops, and reads from the constant cache keep that
  // evaluation off the memory system (from global memory its dependent word
  // loads took several microseconds per instruction under the weight stream)
  uint32_t xw[XS_COUNT * X_MAX_WORDS];
  unsigned long long* trace;  // TRACE_WORDS x u64 per instruction, or null
  BarLayout bl;
  // step
  const int32_t* tokens;
  const int32_t* positions;
  int B, S;
  uint16_t* kv;
  float* logits;
  int mode;
  uint32_t perop_base, perop_count;  // kernel-per-operator: the operator's queue range
  unsigned long long wait_limit_ns;
  // Multi-step greedy decode (batch 1): the queue runs n_steps times in one
  // launch; step s reads positions + s and, for s > 0, the token step s - 1
  // chose.  Per step: the packed (ordered logit, inverted index) maximum over
  // the LM-head tiles, the count of finished LM tiles, the chosen token.
  // n_steps = 1 and null pointers for a single step.
  uint32_t n_steps;
  // [n_steps][gridDim.x], zero before the launch: each CTA's packed running
  // greedy choice over the LM-head tiles it finished in that step (see
  // lm_pack in mk_kernel.cuh)
  unsigned long long* lm_slot;
  int32_t* out_tokens;         // [n_steps]
};
static_assert(sizeof(KParams) <= 4096, "kernel parameter block limit");

// Slot words carry the queue index in the low 24 bits and the step of a
// multi-step launch above them.
constexpr uint32_t SLOT_INDEX_BITS = 24;
constexpr uint32_t MAX_DECODE_STEPS = 64;

}  // namespace mk
