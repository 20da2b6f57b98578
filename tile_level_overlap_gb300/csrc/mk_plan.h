// Host plan builder: tile DAG -> instruction queue + barrier tensor + symbolic
// extents, plus a sequential simulator used by the host-only checks.
#pragma once
#include <stdint.h>

#include <string>
#include <utility>
#include <vector>

#include "../../include/mk.h"
#include "mk_internal.h"

namespace mk {

// Kernel geometry shared by the plan builder and the kernel.
constexpr int NW = 8;                 // consumer warps per CTA
constexpr int NT = NW * 32;           // consumer threads
constexpr int NTHREADS = NT + 128;    // + producer warp, finisher warp, two idle warps
// Registers per thread after the kernel's setmaxnreg split (the launch gives
// 168 to each of the 12 warps: 65536 / (3 warps per SM sub-partition x 32 x
// 4), rounded down to 8).  The two consumer warpgroups take 224, the
// producer/finisher warpgroup keeps 56: 8 x 224 + 4 x 56 = 12 x 168.
constexpr int LAUNCH_REGS = 168;
constexpr int SPLIT_REGS_CONSUMER = 224;
constexpr int SPLIT_REGS_SIDE = 56;
static_assert(8 * SPLIT_REGS_CONSUMER + 4 * SPLIT_REGS_SIDE == 12 * LAUNCH_REGS,
              "register split must add up to the launch's registers");
constexpr int NSTAGE = 6;             // weight/KV ring stages
constexpr int STAGE_BYTES = 32768;    // bytes per ring stage
// Copies the producer keeps in flight (issued, not yet landed): PACE_STAGES
// while the consumers compute, PACE_POLL_STAGES while they poll a tile's
// input words.  A poll's read returns behind the copies its SM already has in
// flight, so a full ring of requests (6 x 32 KB) delayed the first tile of
// each all-to-all operator by a whole ring's worth of HBM time.
constexpr int PACE_STAGES = 3;
constexpr int PACE_POLL_STAGES = 2;
constexpr int NISLOT = 8;             // instruction slots between producer and consumers
constexpr int RMAX = 32;              // GEMV rows per tile (both matrices of a gate/up tile)
constexpr int MAX_LAYERS = 64;        // layer pointer table kept in shared memory
constexpr int BMAX_CC = 8;            // CUDA-core GEMV batch limit
constexpr int XBUF_BYTES = 24576;     // activation / attention scratch in shared memory
constexpr int XBUF_FLOATS = XBUF_BYTES / 4;
constexpr int SCORE_FLOATS = 4096;    // attention scores per split (all q heads of a group)
constexpr int FAST_K_UNIT = 8 * NT;   // K must be a multiple of this for the batch-1 fast path
// Batch-1 fast path at K = m * FAST_K_UNIT: whole weight rows per ring stage.
MK_HD constexpr int fast_rps(int m) { return m >= 8 ? 1 : 8 / m; }

constexpr int DEFAULT_SMS = 152;  // SMs of a GB300

// Keys per decode-attention split, a constant of the model shape (head_dim):
// 216 keys at head_dim 128 and 64 keys at head_dim 64, so that 4096 and 1024
// cached keys with 8 kv heads (the Llama-3-8B and Llama-3.2-1B decode shapes)
// give about one attention tile per SM of a 152-SM GB300 (the phase is
// latency-bound: a second round of tiles doubles it).  Multiples of 8 (one
// tensor-core score product).
MK_HD constexpr int keys_per_split(int head_dim) { return head_dim >= 128 ? 216 : 64; }
// Combine instructions per (sequence, kv head) group when it has several
// splits: each reads every split's partial for its slice of the group's
// outputs, so the partials' round trip is spread over several SMs.  One slice
// per COMBINE_SLICE_BYTES of partial words at max_ctx, at most
// COMBINE_SLICES_MAX; a group whose partials fit one slice is combined by its
// last split instead (no extra instruction).  Measured: Llama-3-8B shape at
// 4096 keys, 4 slices: 2.768 -> 2.709 ms per step; Llama-3.2-1B at 1024 keys,
// one slice by the last split 0.695 ms against 0.707 with two slices.
constexpr int COMBINE_SLICE_BYTES = 20480;
constexpr int COMBINE_SLICES_MAX = 8;
inline int combine_slices(int n_splits, int rep, int head_dim) {
  if (n_splits <= 1) return 1;
  const long n = (long)n_splits * rep * head_dim * 8 / COMBINE_SLICE_BYTES;
  return (int)(n < 1 ? 1 : n > COMBINE_SLICES_MAX ? COMBINE_SLICES_MAX : n);
}

struct HostPlan {
  mk_model_cfg cfg{};
  int max_batch = 0, max_ctx = 0;
  int rep = 0, qkv_rows = 0, n_splits = 0, split_max = 0, kps = 0;
  int n_comb = 1;  // combine instructions per (sequence, kv head) group
  int r_qkv = 0, r_o = 0, r_gu = 0, r_down = 0, r_lm = 0;
  uint32_t n_qkv_tiles = 0, n_o_tiles = 0, n_gu_tiles = 0, n_down_tiles = 0, n_lm_tiles = 0;
  bool fast_b1 = false;     // every GEMV K allows the batch-1 register path
  BarLayout bl{};
  std::vector<Instr> decode;                               // default topological order
  std::vector<std::pair<uint32_t, uint32_t>> perop_decode;  // (first, count) per launch
  std::vector<uint32_t> expr;                               // XS_COUNT * X_MAX_WORDS
  uint64_t weight_bytes = 0;
};

// Validate the shape and build the plan.  Returns MK_OK or an MK_ERR_* code
// with a reason in *why.
// n_sms: SMs of the device the plan runs on (sets the row tiling of the
// projections in whole rounds over the SMs; results do not depend on it);
// 0 = DEFAULT_SMS.
int build_plan(const mk_model_cfg& cfg, int max_batch, int max_ctx, int n_sms, HostPlan* out,
               std::string* why);

// Device scratch of a decode plan: offsets into one allocation (256-byte
// aligned), shared by mk_plan_create and mk_decode_step_noalloc.  The tagged
// intermediate tensors ([o_resid, tagged_end)) must be zero before the first
// launch and whenever the launch counter (CTL_GEN) is cleared, so that no
// stale word carries a tag a later launch expects; the barrier counters and
// control words follow them ([o_bars, zero_end) must start at zero too).
struct DecodeScratch {
  size_t o_resid, o_qkv, o_part, o_attn, o_act, tagged_end;
  size_t o_bars, o_ctl, zero_end;
  size_t o_q, o_rope, o_lw;
  size_t total;
};
DecodeScratch decode_scratch(const HostPlan& hp);

// A seeded random topological order of queue `q` (Kahn's algorithm on the
// barrier counters).  Any topological order is a valid pop order.
void random_topological(const HostPlan& hp, const std::vector<Instr>& q, uint64_t seed,
                        std::vector<Instr>* out);

// Run `q` in order on a host model of the barrier counters.  Returns MK_OK when
// every wait is satisfied on arrival and every waited barrier ends with exactly
// the count its waiters expect.
int simulate(const HostPlan& hp, const std::vector<Instr>& q, std::string* why);

}  // namespace mk
