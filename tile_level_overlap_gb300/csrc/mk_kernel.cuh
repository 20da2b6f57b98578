// The persistent interpreter and its tile routines (sm_103a).
//
// One CTA per SM (12 warps: 8 consumer warps, a producer warp, a finisher warp
// and two idle warps that complete the third warpgroup, whose registers go to
// the consumers): a producer warp pops instructions from the global queue
// (one atomic per instruction) and streams each instruction's dependency-free
// operand bytes -- weight rows, or cached K/V rows -- into a shared-memory ring
// with bulk async copies, running ahead of the consumers by up to NSTAGE
// stages and NISLOT instructions.  Eight consumer warps take instructions in
// pop order, compute from the ring, and read their other inputs with a
// bounded poll on the tag each element of an intermediate tensor carries (the
// launch step that wrote it), so a tile waits on exactly the elements it
// reads; a finisher warp adds the consumers' partial sums of a batch-1 GEMV
// tile and stores its outputs under the step's tag, which publishes them
// without a fence or counter.  This is the on-device interpreter of "Lecture 112: Production
// Megakernels for Real-World Inference" (Technical details: a loop with a
// switch, instructions popped atomically from a queue in DRAM; memory
// pipelining across output tiles) with the tile-level dependencies and the
// weight prefetch across operator boundaries of the MegaOps Abstract.
//
// The same kernel runs kernel-per-operator (MODE_PEROP): one launch per
// operator, its tiles split statically over at most one CTA per SM, no tag
// checks; stream order replaces them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mk_device.cuh"
#include "mk_internal.h"
#include "mk_plan.h"
#include "mk_variants.h"

namespace mk {
// Everything below except make_variant() has internal linkage: this header is
// compiled once per kernel specialisation.
namespace {

constexpr uint32_t END_SLOT = 0xffffffffu;
constexpr int CONSUMER_BAR = 1;

// Shared-memory layout (dynamic).
struct SmemLayout {
  static constexpr int ring = 0;
  static constexpr int xbuf = ring + NSTAGE * STAGE_BYTES;
  static constexpr int red = xbuf + XBUF_BYTES;            // [RMAX][BMAX_CC] floats
  static constexpr int redw = red + RMAX * BMAX_CC * 4;    // [2][NW][RMAX] floats (hand-off buffers)
  static constexpr int hpre = redw + 2 * NW * RMAX * 4;    // [2][RMAX] floats (hand-off residual inputs)
  static constexpr int fin = hpre + 2 * RMAX * 4;          // [RMAX][BMAX_CC] floats (finisher)
  static constexpr int ssw = fin + RMAX * BMAX_CC * 4;     // [NW][BMAX_CC] floats
  static constexpr int bars = ssw + NW * BMAX_CC * 4;      // mbarriers
  // full, empty [NSTAGE]; ifull, iempty [NISLOT]; hfull, hempty [2]
  static constexpr int n_mbar = 2 * NSTAGE + 2 * NISLOT + 4;
  static constexpr int islot = bars + n_mbar * 8;          // [NISLOT] x {u32 index, pad, Instr}
  static constexpr int islot_bytes = 48;
  static constexpr int hrec = islot + NISLOT * islot_bytes;  // [2] x {u32 index, pad, Instr}
  static constexpr int flags = hrec + 2 * islot_bytes;     // [16] u32
  static constexpr int layers = flags + 16 * 4;             // [MAX_LAYERS] LayerW
  static constexpr int total = layers + MAX_LAYERS * (int)sizeof(LayerW);
};
static_assert(SmemLayout::total <= 227 * 1024, "shared memory budget");

// F_STOP: set by a consumer that saw the abort word, read by the producer
// before each pop (a shared-memory load instead of a global one).
// F_POLL: set while the consumers poll a GEMV tile's input words; the
// producer then keeps fewer copies in flight (PACE_POLL_STAGES).
enum Flag { F_GEN = 0, F_ABORT = 1, F_LAST = 2, F_SLOT = 3, F_STOP = 4, F_SLOT_B = 5, F_ABORT_B = 6,
            F_TOKEN = 7, F_POLL = 8 };

struct Sh {
  uint8_t* ring;
  float* xbuf;
  float* red;
  float* redw;
  float* hpre;
  float* fin;
  float* ssw;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* ifull;
  uint64_t* iempty;
  uint64_t* hfull;   // a batch-1 GEMV tile's per-warp sums are ready (NW arrivals)
  uint64_t* hempty;  // the finisher has read them (1 arrival)
  uint8_t* islot;
  uint8_t* hrec;     // the handed-off instruction (index + record) per buffer
  volatile uint32_t* flags;
  const LayerW* layers;  // copy of the per-layer weight pointers
};

__device__ __forceinline__ volatile uint32_t* slot_index(const Sh& S, int si) {
  return reinterpret_cast<volatile uint32_t*>(S.islot + si * SmemLayout::islot_bytes);
}
__device__ __forceinline__ Instr* slot_instr(const Sh& S, int si) {
  return reinterpret_cast<Instr*>(S.islot + si * SmemLayout::islot_bytes + 16);
}

__device__ __forceinline__ Sh sh_map(uint8_t* base) {
  Sh s;
  s.ring = base + SmemLayout::ring;
  s.xbuf = reinterpret_cast<float*>(base + SmemLayout::xbuf);
  s.red = reinterpret_cast<float*>(base + SmemLayout::red);
  s.redw = reinterpret_cast<float*>(base + SmemLayout::redw);
  s.hpre = reinterpret_cast<float*>(base + SmemLayout::hpre);
  s.fin = reinterpret_cast<float*>(base + SmemLayout::fin);
  s.ssw = reinterpret_cast<float*>(base + SmemLayout::ssw);
  uint64_t* b = reinterpret_cast<uint64_t*>(base + SmemLayout::bars);
  s.full = b;
  s.empty = b + NSTAGE;
  s.ifull = b + 2 * NSTAGE;
  s.iempty = b + 2 * NSTAGE + NISLOT;
  s.hfull = b + 2 * NSTAGE + 2 * NISLOT;
  s.hempty = s.hfull + 2;
  s.islot = base + SmemLayout::islot;
  s.hrec = base + SmemLayout::hrec;
  s.layers = reinterpret_cast<const LayerW*>(base + SmemLayout::layers);
  s.flags = reinterpret_cast<volatile uint32_t*>(base + SmemLayout::flags);
  return s;
}

// ---------------------------------------------------------------- errors
__device__ void set_error(const KParams& P, uint32_t code, uint32_t detail) {
  if (atomicCAS(&P.ctl[CTL_STATUS], 0u, code) == 0u) atomicExch(&P.ctl[CTL_DETAIL], detail);
  atomicExch(&P.ctl[CTL_ABORT], 1u);
}

// Bounded mbarrier wait.  Gives up (error + false) after `limit_ns`.
__device__ __forceinline__ bool mbar_wait(const KParams& P, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit = P.wait_limit_ns * 4ull;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit) {
      set_error(P, MK_ERR_TIMEOUT, 0xfffffff0u);
      return false;
    }
  }
}

// Bounded poll on tagged words.  `load` reads this thread's words and returns
// true once every tag it read is the expected one (always true for tag 0:
// kernel-per-operator launches, where stream order makes every input ready).
// Retries until it succeeds, the launch is aborted (abort word, or a local
// stop), or the wait limit passes (MK_ERR_TIMEOUT, detail = `detail`).  On
// failure it raises the CTA's stop flag and returns false; the caller still
// finishes its tile on whatever it read, so the ring protocol stays intact,
// and the next instruction is drained.
template <class F>
__device__ __forceinline__ bool poll_until(const KParams& P, const Sh& S, F&& load, uint32_t detail) {
  if (load()) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    __nanosleep(32);
    const uint32_t ab = ld_volatile(&P.ctl[CTL_ABORT]);  // in flight with the loads
    if (load()) return true;
    if (ab != 0u || S.flags[F_STOP] != 0u) {
      S.flags[F_STOP] = 1u;
      return false;
    }
    if (globaltimer() - t0 > P.wait_limit_ns) {
      set_error(P, MK_ERR_TIMEOUT, detail);
      S.flags[F_STOP] = 1u;
      return false;
    }
  }
}

// Tag a launch step expects on its inputs and writes on its outputs: a fresh
// value per (launch, step) in the persistent mode, 0 (no checks) in the
// kernel-per-operator mode.  IF_NO_PUBLISH (test-only) stores under 0, which no
// persistent reader expects.
__device__ __forceinline__ uint32_t step_tag(const KParams& P, uint32_t gen, uint32_t step) {
  return P.mode == MODE_MEGA ? gen + step + 1u : 0u;
}
__device__ __forceinline__ uint32_t pub_tag(const Instr& in, uint32_t tag) {
  return (in.flags & IF_NO_PUBLISH) ? 0u : tag;
}

// ---------------------------------------------------------------- operand sources
// A tile's streamed operand: up to two regions of whole rows, each split into
// ring stages of `rps` rows.
struct Src {
  const uint8_t* ptr[2];
  uint32_t rows[2];
  uint32_t row_bytes;
  uint32_t rps;
  int nreg;
};

// The kernel's dynamic shared memory (every extern __shared__ array aliases it).
extern __shared__ __align__(1024) uint8_t mk_dyn_smem[];

// Per-layer weight pointers, from the copy the kernel prologue puts in shared
// memory (no dependent global load on the producer's issue path).
__device__ __forceinline__ const LayerW& layer_w(const KParams& P, int l) {
  (void)P;
  return reinterpret_cast<const LayerW*>(mk_dyn_smem + SmemLayout::layers)[l];
}

struct AttnExt {
  bool live;
  int pos, lo, hi, nc;  // keys [lo, hi); cached keys [lo, lo + nc)
  bool has_new;         // this split holds the new token's key (index pos)
};

__device__ __forceinline__ AttnExt attn_extent(const KParams& P, const Instr& in, uint32_t step = 0) {
  AttnExt e;
  e.live = x_eval(P.xw + XS_SEQ_LIVE * X_MAX_WORDS, in, P.B, P.S, nullptr, 0) > 0;
  e.pos = 0;
  e.lo = e.hi = e.nc = 0;
  e.has_new = false;
  if (!e.live) return e;
  const int p0 = P.positions[in.a0];
  e.pos = p0 + (int)step;
  if (e.pos < 0 || e.pos >= P.max_ctx) {
    e.live = false;
    return e;
  }
  if (in.flags & IF_SLICE) return e;  // a combine slice holds no keys
  e.lo = (int)x_eval(P.xw + XS_ATTN_LO * X_MAX_WORDS, in, P.B, P.S, P.positions, P.B, (int)step,
                     (int)in.a0, p0);
  e.hi = (int)x_eval(P.xw + XS_ATTN_HI * X_MAX_WORDS, in, P.B, P.S, P.positions, P.B, (int)step,
                     (int)in.a0, p0);
  int cend = e.hi < e.pos ? e.hi : e.pos;
  e.nc = cend > e.lo ? cend - e.lo : 0;
  e.has_new = e.lo <= e.pos && e.pos < e.hi;
  return e;
}

__device__ __forceinline__ size_t kv_offset(const KParams& P, int l, int kv, int b, int g, int pos) {
  return ((((size_t)l * 2 + kv) * P.max_batch + b) * P.nkv + g) * (size_t)P.max_ctx * P.d +
         (size_t)pos * P.d;
}

// GEMV tile: weight matrices and K of instruction `in`.
struct GemvDesc {
  const uint16_t* w0;
  const uint16_t* w1;
  int K, rows, row0;
};

__device__ __forceinline__ GemvDesc gemv_desc(const KParams& P, const Instr& in) {
  GemvDesc g;
  g.w1 = nullptr;
  g.row0 = (int)in.a0;
  g.rows = (int)in.a1;
  const int qd = P.nq * P.d;
  const LayerW& W = layer_w(P, in.layer);
  switch (in.op) {
    case OP_QKV: {
      int r = g.row0;
      g.K = P.H;
      if (r < qd) g.w0 = W.wq + (size_t)r * P.H;
      else if (r < qd + P.nkv * P.d) g.w0 = W.wk + (size_t)(r - qd) * P.H;
      else g.w0 = W.wv + (size_t)(r - qd - P.nkv * P.d) * P.H;
      break;
    }
    case OP_O: g.K = qd; g.w0 = W.wo + (size_t)g.row0 * qd; break;
    case OP_GU:
      g.K = P.H;
      g.w0 = W.wg + (size_t)g.row0 * P.H;
      g.w1 = W.wu + (size_t)g.row0 * P.H;
      break;
    case OP_DOWN: g.K = P.F; g.w0 = W.wd + (size_t)g.row0 * P.F; break;
    default: g.K = P.H; g.w0 = P.lm + (size_t)g.row0 * P.H; break;  // OP_LM
  }
  return g;
}

// Operand source of an instruction; `e` is its attention extent (ignored for
// GEMV tiles).
__device__ __forceinline__ Src src_of(const KParams& P, const Instr& in, const AttnExt& e) {
  Src s;
  s.nreg = 0;
  s.rows[0] = s.rows[1] = 0;
  s.ptr[0] = s.ptr[1] = nullptr;
  if (in.op == OP_ATTN) {
    s.row_bytes = P.d * 2;
    s.rps = STAGE_BYTES / s.row_bytes;
    if (e.live && e.nc > 0) {
      s.nreg = 2;
      s.ptr[0] = reinterpret_cast<const uint8_t*>(P.kv + kv_offset(P, in.layer, 0, in.a0, in.a1, e.lo));
      s.ptr[1] = reinterpret_cast<const uint8_t*>(P.kv + kv_offset(P, in.layer, 1, in.a0, in.a1, e.lo));
      s.rows[0] = s.rows[1] = (uint32_t)e.nc;
    }
    return s;
  }
  GemvDesc g = gemv_desc(P, in);
  s.row_bytes = (uint32_t)g.K * 2;
  s.rps = STAGE_BYTES / s.row_bytes;
  s.nreg = g.w1 ? 2 : 1;
  s.ptr[0] = reinterpret_cast<const uint8_t*>(g.w0);
  s.ptr[1] = reinterpret_cast<const uint8_t*>(g.w1);
  s.rows[0] = s.rows[1] = (uint32_t)g.rows;
  return s;
}

__device__ __forceinline__ Src instr_src(const KParams& P, const Instr& in) {
  AttnExt e;
  e.live = false;
  if (in.op == OP_ATTN) e = attn_extent(P, in);
  return src_of(P, in, e);
}

// The attention extent travels from the producer to the consumers in the
// instruction slot (bytes 4..15), so it is evaluated once per instruction.
__device__ __forceinline__ void slot_put_ext(const Sh& S, int si, const AttnExt& e) {
  int32_t* x = reinterpret_cast<int32_t*>(S.islot + si * SmemLayout::islot_bytes + 4);
  x[0] = e.lo;
  x[1] = e.hi;
  x[2] = e.live ? e.pos : -1;
}
__device__ __forceinline__ AttnExt slot_get_ext(const Sh& S, int si) {
  const int32_t* x = reinterpret_cast<const int32_t*>(S.islot + si * SmemLayout::islot_bytes + 4);
  AttnExt e;
  e.lo = x[0];
  e.hi = x[1];
  e.live = x[2] >= 0;
  e.pos = e.live ? x[2] : 0;
  const int cend = e.hi < e.pos ? e.hi : e.pos;
  e.nc = (e.live && cend > e.lo) ? cend - e.lo : 0;
  e.has_new = e.live && e.lo <= e.pos && e.pos < e.hi;
  if (!e.live) e.lo = e.hi = 0;
  return e;
}

__device__ __forceinline__ uint32_t src_stages(const Src& s) {
  uint32_t n = 0;
  for (int r = 0; r < s.nreg; ++r) n += (s.rows[r] + s.rps - 1) / s.rps;
  return n;
}

// ---------------------------------------------------------------- producer
// MS: the multi-step kernel (mk_decode_steps); the single-step kernel keeps
// the step at 0 at compile time.
template <bool MS>
__device__ void producer(const KParams& P, const Sh& S) {
  const int lane = threadIdx.x & 31;
  if (lane != 0) return;
  const uint64_t policy = policy_evict_first();
  uint32_t stage_ctr = 0, islot_ctr = 0;
  // An instruction is popped only once the ring has a free stage for its first
  // operand block, i.e. when this CTA can start streaming it.  A CTA whose
  // consumers wait on a dependency therefore holds at most the one instruction
  // it is prefetching, and the rest of a dependency-gated operator goes to the
  // CTAs that reach it first instead of queueing behind the waiting one.  The
  // pop and record latency overlap the consumers' work on the stages already
  // in the ring.
  // A multi-step launch runs the queue n_steps times: pop g is instruction
  // g % n_instr of step g / n_instr.
  uint32_t npop = 0;
  // multi-step: the step of pop g is g / n_instr; a CTA's pops increase, so
  // the step is tracked by comparison instead of a division per pop
  uint32_t step_cur = 0, step_base = 0;
  auto pop = [&]() -> uint32_t {
    const uint32_t k = npop++;
    if (P.mode == MODE_MEGA) {
      if (S.flags[F_STOP]) return END_SLOT;
      const uint32_t g = atomicAdd(&P.ctl[CTL_HEAD], 1u);
      return g < P.n_instr * (MS ? P.n_steps : 1u) ? g : END_SLOT;
    }
    // kernel-per-operator: CTA c runs tiles c, c + grid, ... of the
    // operator (a static split, no atomics), so a CTA loads the operator's
    // input activations once, as in the persistent launch
    const uint32_t j = k * gridDim.x + blockIdx.x;
    return j < P.perop_count ? P.perop_base + j : END_SLOT;
  };
  for (;;) {
    const bool room = mbar_wait(P, &S.empty[stage_ctr % NSTAGE], ((stage_ctr / NSTAGE) & 1u) ^ 1u);
    const uint32_t g_in = room ? pop() : END_SLOT;
    const bool end = g_in == END_SLOT;
    if (MS && !end) {
      while (g_in - step_base >= P.n_instr) {
        ++step_cur;
        step_base += P.n_instr;
      }
    }
    const uint32_t step = MS ? step_cur : 0u;
    const uint32_t i_in = end ? END_SLOT : g_in - (MS ? step_base : 0u);
    Instr in;
    if (!end) in = P.queue[i_in];
    const int si = islot_ctr % NISLOT;
    bool posted_end = end;
    AttnExt ext;
    ext.live = false;
    if (!end && in.op == OP_ATTN) ext = attn_extent(P, in, step);
    if (!mbar_wait(P, &S.iempty[si], ((islot_ctr / NISLOT) & 1u) ^ 1u)) posted_end = true;
    if (!posted_end) {
      *slot_instr(S, si) = in;
      slot_put_ext(S, si, ext);
    }
    *slot_index(S, si) = posted_end ? END_SLOT : (i_in | (step << SLOT_INDEX_BITS));
    mbar_arrive(&S.ifull[si]);
    if (P.trace && !posted_end) P.trace[(size_t)i_in * TRACE_WORDS + 4] = globaltimer();
    ++islot_ctr;
    if (posted_end) break;

    const Src src = src_of(P, in, ext);
    bool stuck = false;
    uint64_t blocked_ns = 0;  // (tracing) time spent waiting for a free stage
    for (int r = 0; r < src.nreg && !stuck; ++r) {
      for (uint32_t row = 0; row < src.rows[r]; row += src.rps) {
        uint32_t n = src.rows[r] - row < src.rps ? src.rows[r] - row : src.rps;
        uint32_t bytes = n * src.row_bytes;
        const int st = stage_ctr % NSTAGE;
        const uint64_t tw = P.trace ? globaltimer() : 0;
        if (!mbar_wait(P, &S.empty[st], ((stage_ctr / NSTAGE) & 1u) ^ 1u)) {
          // the consumers stopped taking stages: issue nothing more (the
          // consumers' own bounded waits end their loop)
          stuck = true;
          break;
        }
        if (P.trace) blocked_ns += globaltimer() - tw;
        {
          // pace the stream: at most `lim` copies in flight, fewer while the
          // consumers poll, so their reads do not queue behind a full ring
          const uint32_t lim = S.flags[F_POLL] != 0u ? (uint32_t)PACE_POLL_STAGES : (uint32_t)PACE_STAGES;
          if (stage_ctr >= lim) {
            const uint32_t c2 = stage_ctr - lim;  // an earlier stage, not yet reissued
            if (!mbar_wait(P, &S.full[c2 % NSTAGE], (c2 / NSTAGE) & 1u)) {
              stuck = true;
              break;
            }
          }
        }
        mbar_arrive_expect_tx(&S.full[st], bytes);
        bulk_g2s(S.ring + (size_t)st * STAGE_BYTES, src.ptr[r] + (size_t)row * src.row_bytes, bytes,
                 &S.full[st], policy);
        ++stage_ctr;
      }
    }
    if (P.trace) P.trace[(size_t)i_in * TRACE_WORDS + 7] = blocked_ns;
    if (stuck) break;
  }
}

// ---------------------------------------------------------------- consumer helpers
// Tracing (thread 0 only) writes each timestamp into the instruction's record
// when it is taken, so no timestamp stays live in registers across a tile.
struct Ring {
  uint32_t ctr;      // stages consumed so far
  uint32_t hctr;     // batch-1 GEMV tiles handed to the finisher so far
  uint32_t cur;      // (tracing) queue index of the instruction being run
  uint32_t wait_ns;  // (tracing) time spent waiting for stages in this instruction
  bool first_done;   // (tracing) its first stage was recorded
  bool handed;       // a batch-1 GEMV tile went to the finisher (which records "done")
};
__device__ __forceinline__ void trace_mark(const KParams& P, uint32_t ii, int word) {
  P.trace[(size_t)ii * TRACE_WORDS + word] = globaltimer();
}

// Wait for ring stage number `c` (a running count) and return it.
__device__ __forceinline__ const uint8_t* ring_wait(const KParams& P, const Sh& S, Ring& R, uint32_t c) {
  const int st = c % NSTAGE;
  if (P.trace && threadIdx.x == 0) {
    const uint64_t t0 = globaltimer();
    mbar_wait(P, &S.full[st], (c / NSTAGE) & 1u);
    const uint64_t t1 = globaltimer();
    R.wait_ns += (uint32_t)(t1 - t0);
    if (!R.first_done) {
      P.trace[(size_t)R.cur * TRACE_WORDS + 6] = t1;
      R.first_done = true;
    }
  } else {
    mbar_wait(P, &S.full[st], (c / NSTAGE) & 1u);
  }
  return S.ring + (size_t)st * STAGE_BYTES;
}
__device__ __forceinline__ const uint8_t* ring_acquire(const KParams& P, const Sh& S, Ring& R) {
  return ring_wait(P, S, R, R.ctr);
}
__device__ __forceinline__ void ring_release(const Sh& S, Ring& R) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&S.empty[R.ctr % NSTAGE]);
  ++R.ctr;
}

__device__ __forceinline__ void cbar() { named_bar(CONSUMER_BAR, NT); }

// Deterministic sum over the consumer threads (fixed reduction tree).
__device__ __forceinline__ float consumer_sum(float v, float* scratch) {
  const int t = threadIdx.x, w = t >> 5;
  v = warp_sum(v);
  if ((t & 31) == 0) scratch[w] = v;
  cbar();
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < NW; ++k) s += scratch[k];
  cbar();
  return s;
}

// Token id of sequence b from the caller, validated.
__device__ __forceinline__ int token_of(const KParams& P, int b) {
  int t = P.tokens[b];
  if (t < 0 || t >= P.V) {
    if (threadIdx.x == 0) set_error(P, MK_ERR_BOUNDS, (uint32_t)b);
    t = 0;
  }
  return t;
}

// ---------------------------------------------------------------- greedy choice (multi-step)
// A logit and its vocabulary row packed so that the unsigned maximum picks the
// largest logit and, among equal logits, the smallest row: the float's bits
// mapped to an order-preserving word (bits 63..32), the row inverted (bits
// 31..14, rows below 2^18), and bits 13..0 free for a count.  Each CTA's
// finisher keeps the running maximum over the LM-head tiles it finished in a
// step and stores it with their count as one word per (step, CTA): plain
// stores to distinct words, no same-address atomics (8000 of those per step
// queued on one L2 slice and slowed the LM head's weight stream).
constexpr int LM_ROW_BITS = 18, LM_CNT_BITS = 14;
constexpr unsigned long long LM_CNT_MASK = (1ull << LM_CNT_BITS) - 1;
__device__ __forceinline__ unsigned long long lm_pack(float y, uint32_t row) {
  const uint32_t u = __float_as_uint(y);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) |
         ((unsigned long long)(((1u << LM_ROW_BITS) - 1u) - row) << LM_CNT_BITS);
}
__device__ __forceinline__ int lm_row(unsigned long long key) {
  return (int)(((1u << LM_ROW_BITS) - 1u) - (uint32_t)((key >> LM_CNT_BITS) & ((1u << LM_ROW_BITS) - 1u)));
}

// The token step `step - 1` chose (all consumer threads call it): consumer
// warp 0 polls the CTAs' words of that step until their counts add up to the
// LM-head tile count, takes the largest packed maximum and hands the row to
// the others through shared memory.  Validated like a caller's token.
__device__ int ms_chosen_token(const KParams& P, const Sh& S, uint32_t step) {
  const int t = threadIdx.x;
  if (t < 32) {
    const u64* w = reinterpret_cast<const u64*>(P.lm_slot) + (size_t)(step - 1) * gridDim.x;
    const uint64_t t0 = globaltimer();
    unsigned long long best = 0;
    for (;;) {
      unsigned long long m = 0;
      uint32_t cnt = 0;
      for (uint32_t c = (uint32_t)t; c < gridDim.x; c += 32) {
        const unsigned long long v = ld_tagged(w + c);
        cnt += (uint32_t)(v & LM_CNT_MASK);
        m = (v & ~LM_CNT_MASK) > m ? (v & ~LM_CNT_MASK) : m;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        const unsigned long long om = __shfl_xor_sync(0xffffffffu, m, o);
        m = om > m ? om : m;
      }
      best = m;
      if (cnt >= P.n_lm_tiles) break;  // warp-uniform
      // bounded: the lane-0 verdict decides for the whole warp
      int verdict = 0;
      if (t == 0) {
        if (ld_volatile(&P.ctl[CTL_ABORT]) != 0u || S.flags[F_STOP] != 0u) verdict = 1;
        else if (globaltimer() - t0 > P.wait_limit_ns) verdict = 2;
      }
      verdict = __shfl_sync(0xffffffffu, verdict, 0);
      if (verdict) {
        if (t == 0) {
          if (verdict == 2) set_error(P, MK_ERR_TIMEOUT, 0xfffffff5u);
          S.flags[F_STOP] = 1u;
        }
        break;
      }
      __nanosleep(32);
    }
    if (t == 0) {
      int row = lm_row(best);
      if (row < 0 || row >= P.V) {
        if (S.flags[F_STOP] == 0u) set_error(P, MK_ERR_BOUNDS, 0u);
        row = 0;
      }
      S.flags[F_TOKEN] = (uint32_t)row;
    }
  }
  cbar();
  return (int)S.flags[F_TOKEN];
}

// Activation source of a GEMV op (row-major [max_batch][K] tagged words), or
// null when it is the embedding row of the sequence's token (layer-0 QKV).
__device__ __forceinline__ const u64* gemv_x(const KParams& P, const Instr& in) {
  const size_t bh = (size_t)P.max_batch * P.H;
  switch (in.op) {
    case OP_QKV: return in.layer == 0 ? nullptr : P.resid + (size_t)(2 * in.layer) * bh;
    case OP_O: return P.attn_out + (size_t)in.layer * P.max_batch * (P.nq * P.d);
    case OP_GU: return P.resid + (size_t)(2 * in.layer + 1) * bh;
    case OP_DOWN: return P.act + (size_t)in.layer * P.max_batch * P.F;
    default: return P.resid + (size_t)(2 * P.L) * bh;
  }
}
__device__ __forceinline__ const uint16_t* gemv_gain(const KParams& P, const Instr& in) {
  switch (in.op) {
    case OP_QKV: return layer_w(P, in.layer).attn_norm;
    case OP_GU: return layer_w(P, in.layer).ffn_norm;
    case OP_LM: return P.final_norm;
    default: return nullptr;
  }
}

// Read 8 consecutive tagged words (64-byte aligned) into x; true when every
// tag is `tag` (or tag is 0).
__device__ __forceinline__ bool ld_tagged8(const u64* p, uint32_t tag, float (&x)[8]) {
  u64 w[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) ld_tagged2(p + 2 * k, w[2 * k], w[2 * k + 1]);
  uint32_t bad = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[k] = tag_val(w[k]);
    bad |= tag_of(w[k]) ^ tag;
  }
  return tag == 0u || bad == 0u;
}

// Load 8 consecutive activations of sequence b starting at column c (a bounded
// poll on their tags), or widen them from the embedding row.
__device__ __forceinline__ void load_x8(const KParams& P, const Sh& S, const u64* xs,
                                        const uint16_t* emb_row, int b, int K, int c, uint32_t tag,
                                        float (&x)[8]) {
  if (xs) {
    const u64* p = xs + (size_t)b * K + c;
    poll_until(P, S, [&]() { return ld_tagged8(p, tag, x); }, 0xfffffff1u);
  } else {
    uint4 w = __ldg(reinterpret_cast<const uint4*>(emb_row + c));
    widen8(w, x);
  }
}

// ---------------------------------------------------------------- GEMV, batch 1, K = M * 8 * NT
// Thread t owns columns 8*(t + NT*j) .. +8 for j < M and keeps them (normed)
// in registers; each ring stage holds RPS = 8 / M whole rows, whose per-thread
// partial dot products are summed across the warp (multi-value butterfly) into
// a per-warp row slot; one fixed-order sum over warps per tile.
template <int M, bool MS>
__device__ __forceinline__ void load_x_fast(const KParams& P, const Sh& S, const Instr& in,
                                            float (&xr)[M][8], uint32_t step, uint32_t tag) {
  const int t = threadIdx.x;
  constexpr int K = M * FAST_K_UNIT;
  const u64* xs = gemv_x(P, in);
  // a later step of a multi-step launch starts from the token the previous
  // step chose (every CTA's LM-head tiles of that step finished)
  int tok = 0;
  if (!xs) tok = (MS && step > 0) ? ms_chosen_token(P, S, step) : token_of(P, 0);
  const uint16_t* emb_row = xs ? nullptr : P.embed + (size_t)tok * P.H;
  const uint16_t* gain = gemv_gain(P, in);
  uint4 gw[M];
  if (gain) {
#pragma unroll
    for (int j = 0; j < M; ++j) gw[j] = __ldg(reinterpret_cast<const uint4*>(gain + 8 * (t + NT * j)));
  }
  if (xs) {
    if (t == 0) S.flags[F_POLL] = 1u;
    // every word of this thread's columns in flight at once, one tag check
    poll_until(P, S, [&]() {
      bool ok = true;
#pragma unroll
      for (int j = 0; j < M; ++j) ok &= ld_tagged8(xs + 8 * (t + NT * j), tag, xr[j]);
      return ok;
    }, 0xfffffff2u);
    if (t == 0) S.flags[F_POLL] = 0u;
  } else {
#pragma unroll
    for (int j = 0; j < M; ++j) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(emb_row + 8 * (t + NT * j)));
      widen8(w, xr[j]);
    }
  }
  if (gain) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < M; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(xr[j][e], xr[j][e], ss);
    ss = consumer_sum(ss, S.ssw);
    const float inv = 1.0f / sqrtf(ss / (float)K + P.eps);
#pragma unroll
    for (int j = 0; j < M; ++j) {
      float g8[8];
      widen8(gw[j], g8);
#pragma unroll
      for (int e = 0; e < 8; ++e) xr[j][e] = xr[j][e] * inv * g8[e];
    }
  }
}

// The down projection's input (the SwiGLU output: no norm, no gain, never the
// embedding), loaded without the general form's gain registers.
template <int M>
__device__ __forceinline__ void load_x_plain(const KParams& P, const Sh& S, const u64* xs,
                                             float (&xr)[M][8], uint32_t tag) {
  const int t = threadIdx.x;
  // two halves, so that the tag halves of the words in flight do not push
  // the register-resident activations out
  constexpr int MA = (M + 1) / 2;
  if (t == 0) S.flags[F_POLL] = 1u;
  poll_until(P, S, [&]() {
    bool ok = true;
#pragma unroll
    for (int j = 0; j < MA; ++j) ok &= ld_tagged8(xs + 8 * (t + NT * j), tag, xr[j]);
    return ok;
  }, 0xfffffff3u);
  poll_until(P, S, [&]() {
    bool ok = true;
#pragma unroll
    for (int j = MA; j < M; ++j) ok &= ld_tagged8(xs + 8 * (t + NT * j), tag, xr[j]);
    return ok;
  }, 0xfffffff3u);
  if (t == 0) S.flags[F_POLL] = 0u;
}

// The residual input of an O / down tile output element (thread t owns output
// (r, b) = (t / B, t % B)): its word is read before the tile streams, so that
// the read's latency hides behind the stages, and its tag is checked after
// them (epilogue_resolve).  Every (row, sequence) pair of a tile maps to one
// consumer thread (RMAX * BMAX_CC <= NT).
// The tagged word of output (r, b)'s residual input, or null (no residual, or
// the embedding row in layer 0).
__device__ __forceinline__ const u64* residual_src(const KParams& P, const Instr& in, const GemvDesc& g,
                                                   int t) {
  const int B = P.B, l = in.layer;
  if (t >= g.rows * B) return nullptr;
  const int r = t / B, b = t % B, row = g.row0 + r;
  const size_t bh = (size_t)P.max_batch * P.H;
  if (in.op == OP_O && l > 0) return P.resid + (size_t)(2 * l) * bh + (size_t)b * P.H + row;
  if (in.op == OP_DOWN) return P.resid + (size_t)(2 * l + 1) * bh + (size_t)b * P.H + row;
  return nullptr;
}
template <bool MS>
__device__ __forceinline__ u64 epilogue_prefetch(const KParams& P, const Sh& S, const Instr& in,
                                                 const GemvDesc& g, int t, uint32_t step = 0) {
  if (in.op == OP_O && in.layer == 0) {
    // layer 0's residual input is the token's embedding row (all consumer
    // threads take part when the token is a previous step's choice)
    const int tok0 = (MS && step > 0) ? ms_chosen_token(P, S, step) : 0;
    if (t >= g.rows * P.B) return 0ull;
    const int r = t / P.B, b = t % P.B;
    const int tok = (MS && step > 0) ? tok0 : token_of(P, b);
    return (u64)((uint32_t)P.embed[(size_t)tok * P.H + g.row0 + r] << 16);
  }
  const u64* src = residual_src(P, in, g, t);
  return src ? ld_tagged(src) : 0ull;
}
// The residual input's value, once its tag is the expected one (a bounded poll
// when the early read found it stale).
__device__ __forceinline__ float epilogue_resolve(const KParams& P, const Sh& S, const Instr& in,
                                                  const GemvDesc& g, int t, u64 w, uint32_t tag) {
  const u64* src = residual_src(P, in, g, t);
  if (src && tag != 0u && tag_of(w) != tag)
    poll_until(P, S, [&]() {
      w = ld_tagged(src);
      return tag_of(w) == tag;
    }, 0xfffffff4u);
  return tag_val(w);
}

// Hand-off buffers between the consumers and the finisher warp: record `hb`
// holds the instruction whose per-warp sums sit in redw[hb].
__device__ __forceinline__ volatile uint32_t* hrec_index(const Sh& S, int hb) {
  return reinterpret_cast<volatile uint32_t*>(S.hrec + hb * SmemLayout::islot_bytes);
}
__device__ __forceinline__ volatile uint32_t* hrec_step(const Sh& S, int hb) {
  return reinterpret_cast<volatile uint32_t*>(S.hrec + hb * SmemLayout::islot_bytes + 4);
}
__device__ __forceinline__ Instr* hrec_instr(const Sh& S, int hb) {
  return reinterpret_cast<Instr*>(S.hrec + hb * SmemLayout::islot_bytes + 16);
}
// Every consumer warp: wait until the finisher has read buffer R.hctr & 1
// (used two hand-offs ago, so normally long free).
__device__ __forceinline__ int handoff_acquire(const KParams& P, const Sh& S, const Ring& R) {
  const int hb = (int)(R.hctr & 1u);
  if ((threadIdx.x & 31) == 0) mbar_wait(P, &S.hempty[hb], ((R.hctr >> 1) & 1u) ^ 1u);
  __syncwarp();
  return hb;
}
// Every consumer warp, after its sums (and, in warp 0, the record) are written.
__device__ __forceinline__ void handoff_commit(const Sh& S, Ring& R, int hb) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&S.hfull[hb]);
  ++R.hctr;
}

// Batch-1 GEMV tile: streams the tile's rows and leaves one partial sum per
// (warp, row) in a hand-off buffer; the finisher warp adds them up, runs the
// epilogue and releases the tile, so the consumers go straight on to the next
// instruction.  Software-pipelined by one stage: a stage's loads are issued,
// then the warp reduction of the previous stage's row sums, then this stage's
// FMAs, so the shuffle chain overlaps the shared-memory latency instead of
// following it; the loop body stays small (one stage).
template <int M, bool MS>
__device__ __forceinline__ void gemv_fast(const KParams& P, const Sh& S, const Instr& in,
                                          uint32_t ii, uint32_t step, uint32_t tag, const GemvDesc& g,
                                          const Src& src, Ring& R, const float (&xr)[M][8]) {
  constexpr int RPS = fast_rps(M);  // whole rows per 32 KB stage at K = M * 2048
  constexpr int kDup = 32 / RPS;    // lanes holding the same total after the reduction
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int K = g.K;
  const int rows0 = (int)src.rows[0];
  const int nst = ((rows0 + RPS - 1) / RPS) * src.nreg;
  const int hb = handoff_acquire(P, S, R);
  if (P.trace && t == 0) trace_mark(P, ii, 11);
  // the residual input of the tile's outputs (O, down), loaded now so that its
  // latency hides behind the stages; the finisher takes it from the hand-off
  const u64 pre_w = epilogue_prefetch<MS>(P, S, in, g, t, step);
  if (MS && t == 0) *hrec_step(S, hb) = step;  // the buffer is this tile's from here on
  float* redw = S.redw + hb * NW * RMAX;
  // the activations as packed (even, odd) column pairs for fma.rn.f32x2
  u64 xp[M][4];
#pragma unroll
  for (int j = 0; j < M; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) xp[j][k] = pack_f32x2(xr[j][2 * k], xr[j][2 * k + 1]);
  const int idx = warp_multi_index<RPS>(lane);
  const bool writer = (lane & (kDup - 1)) == 0;
  float prev[RPS];
#pragma unroll
  for (int i = 0; i < RPS; ++i) prev[i] = 0.f;
  int prev_row = 0, prev_n = 0;  // tile row and row count of the sums in prev
  int srow = 0, reg = 0;         // first row of the next stage in its region
#pragma unroll 1
  for (int s = 0; s < nst; ++s) {
    const int n = rows0 - srow < RPS ? rows0 - srow : RPS;
    const int st = R.ctr % NSTAGE;
    const uint8_t* stage = ring_acquire(P, S, R);
    uint4 wv[RPS][M];
#pragma unroll
    for (int i = 0; i < RPS; ++i)
#pragma unroll
      for (int j = 0; j < M; ++j)
        wv[i][j] = reinterpret_cast<const uint4*>(stage + (size_t)i * K * 2)[t + NT * j];
    // the previous stage's sums while the loads are in flight
    {
      const float v = warp_reduce_multi<RPS>(prev, lane);
      if (writer && idx < prev_n) redw[w * RMAX + prev_row + idx] = v;
    }
#pragma unroll
    for (int i = 0; i < RPS; ++i) {
      // Packed products: each bf16 pair of a weight word times the matching
      // pair of activations in one fma.rn.f32x2 (even and odd columns in the
      // two lanes of the accumulator pair), per 8-column group; the lanes and
      // the groups are added in a fixed order.  Rows past the region's end
      // read stale stage bytes into sums that are never stored.
      u64 acc = dot8_x2(wv[i][0], xp[0], 0ull);
#pragma unroll
      for (int j = 1; j < M; ++j) acc = dot8_x2(wv[i][j], xp[j], acc);
      prev[i] = pair_sum(acc);
    }
    __syncwarp();
    mbar_arrive_if(&S.empty[st], lane == 0);
    ++R.ctr;
    prev_row = reg * rows0 + srow;
    prev_n = n;
    srow += RPS;
    if (srow >= rows0) {
      srow = 0;
      ++reg;
    }
  }
  {
    const float v = warp_reduce_multi<RPS>(prev, lane);
    if (writer && idx < prev_n) redw[w * RMAX + prev_row + idx] = v;
  }
  if (t < RMAX) S.hpre[hb * RMAX + t] = epilogue_resolve(P, S, in, g, t, pre_w, tag);
  if (t == 0) {
    if (P.trace) trace_mark(P, ii, 8);
    *hrec_instr(S, hb) = in;
    *hrec_index(S, hb) = ii;
  }
  if (P.trace && t == NT - 32) trace_mark(P, ii, 13);
  handoff_commit(S, R, hb);
  R.handed = true;
  if (P.trace && t == 0) trace_mark(P, ii, 15);
}

// ---------------------------------------------------------------- GEMV, any K, batch <= BMAX_CC
// x[B][K] (normed) staged in shared memory; one warp per (row, sequence) pair.
__device__ __forceinline__ void gemv_generic(const KParams& P, const Sh& S, const Instr& in, const GemvDesc& g,
                             const Src& src, Ring& R, uint32_t tag) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int K = g.K, B = P.B, K8 = K / 8;
  const u64* xs = gemv_x(P, in);
  const uint16_t* gain = gemv_gain(P, in);
  float ss[BMAX_CC];
#pragma unroll
  for (int b = 0; b < BMAX_CC; ++b) ss[b] = 0.f;
  for (int idx = t; idx < B * K8; idx += NT) {
    const int b = idx / K8, c = (idx % K8) * 8;
    const uint16_t* emb_row = xs ? nullptr : P.embed + (size_t)token_of(P, b) * P.H;
    float x[8];
    load_x8(P, S, xs, emb_row, b, K, c, tag, x);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      S.xbuf[b * K + c + e] = x[e];
      s = fmaf(x[e], x[e], s);
    }
#pragma unroll
    for (int bb = 0; bb < BMAX_CC; ++bb)
      if (bb == b) ss[bb] += s;
  }
  if (gain) {
    float inv[BMAX_CC];
#pragma unroll
    for (int b = 0; b < BMAX_CC; ++b)
      inv[b] = b < B ? 1.0f / sqrtf(consumer_sum(ss[b], S.ssw) / (float)K + P.eps) : 0.f;
    cbar();
    for (int idx = t; idx < B * K; idx += NT) {
      const int b = idx / K, k = idx % K;
      float iv = 0.f;
#pragma unroll
      for (int bb = 0; bb < BMAX_CC; ++bb)
        if (bb == b) iv = inv[bb];
      const float gw = __uint_as_float((uint32_t)__ldg(gain + k) << 16);
      S.xbuf[idx] = S.xbuf[idx] * iv * gw;
    }
  }
  cbar();

  int tile_row = 0;
  for (int r = 0; r < src.nreg; ++r) {
    for (uint32_t row = 0; row < src.rows[r]; row += src.rps) {
      const int n = (int)(src.rows[r] - row < src.rps ? src.rows[r] - row : src.rps);
      const uint8_t* stage = ring_acquire(P, S, R);
      for (int p = w; p < n * B; p += NW) {
        const int rr = p / B, b = p % B;
        const uint4* wrow = reinterpret_cast<const uint4*>(stage + (size_t)rr * K * 2);
        const float* xb = S.xbuf + b * K;
        float a = 0.f;
        for (int v = lane; v < K8; v += 32) a = dot8(wrow[v], xb + v * 8, a);
        a = warp_sum(a);
        if (lane == 0) S.red[(tile_row + rr) * BMAX_CC + b] = a;
      }
      ring_release(S, R);
      tile_row += n;
    }
  }
  cbar();
}


// Store a finished GEMV tile: y[r][b] is in red[r * BMAX_CC + b]; `t` is the
// (row, sequence) slot of this thread and `pre` its residual input from
// epilogue_prefetch.
// Outputs are stored as tagged words under `ptag` (the logits as plain floats):
// their consumers poll the tags, so no fence or counter release follows.
__device__ void gemv_epilogue(const KParams& P, const float* red, const Instr& in, const GemvDesc& g,
                              float pre, int t, uint32_t ptag) {
  const int B = P.B, l = in.layer;
  if (t >= g.rows * B) return;
  const int r = t / B, b = t % B, row = g.row0 + r;
  const size_t bh = (size_t)P.max_batch * P.H;
  const float y = red[r * BMAX_CC + b];
  switch (in.op) {
    case OP_QKV:
      st_tagged(P.qkv + ((size_t)l * P.max_batch + b) * P.qkv_rows + row, y, ptag);
      break;
    case OP_O:
      st_tagged(P.resid + (size_t)(2 * l + 1) * bh + (size_t)b * P.H + row, pre + y, ptag);
      break;
    case OP_GU: {
      const float u = red[(g.rows + r) * BMAX_CC + b];
      st_tagged(P.act + ((size_t)l * P.max_batch + b) * P.F + row, y / (1.0f + expf(-y)) * u, ptag);
      break;
    }
    case OP_DOWN:
      st_tagged(P.resid + (size_t)(2 * l + 2) * bh + (size_t)b * P.H + row, pre + y, ptag);
      break;
    default:
      P.logits[(size_t)b * P.V + row] = y;
      break;
  }
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------- decode attention (split-KV)
// One (sequence, kv head, split): the split's cached keys stream through the
// ring; the new token's key/value come from the QKV output (normed when q/k
// norm is on, rotated, rounded to bf16 like every cached entry, written to the
// cache by the split that holds slot pos).
// Partial (max, sum, unnormalised o) per q head, stored as tagged words.  The
// group's combine instructions (IF_COMBINE | IF_SLICE, after every split in
// the queue) then poll every live split's partial and combine them in split
// order, each for its slice of the group's outputs; a group's only split
// (IF_COMBINE alone) combines its own partial.  A split past the sequence's
// keys holds none and does nothing.
// (tracing) attention tile phase boundaries: trace words 8 (inputs loaded and
// rotated), 9 (scores), 10 (softmax and P V), 11 (partials of the group ready,
// combining split only)
__device__ __forceinline__ void attn_mark(const KParams& P, uint32_t ii, int word) {
  if (P.trace && threadIdx.x == 0) P.trace[(size_t)ii * TRACE_WORDS + word] = globaltimer();
}

template <int D, int REP>
__device__ __forceinline__ void attn_tile(const KParams& P, const Sh& S, const Instr& in, const AttnExt& e,
                          uint32_t ii, uint32_t tag, Ring& R) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int l = in.layer, b = (int)in.a0, g = (int)in.a1, split = (int)in.a2;
  constexpr int rep = REP;
  const int qd = P.nq * D, NS = P.n_splits;
  constexpr int smax = SCORE_FLOATS / REP;
  const uint32_t ptag = pub_tag(in, tag);
  if (t == 0 && b < P.B && !e.live) set_error(P, MK_ERR_BOUNDS, ii);  // position out of range
  float* qs = S.xbuf;            // [rep][D]
  float* kn = qs + 8 * 128;      // [D]
  float* vn = kn + 128;          // [D]
  float* sc = vn + 128;          // [rep][smax]
  u64* part = P.part + ((((size_t)l * P.max_batch + b) * P.nkv + g) * NS + split) * rep * (D + 2);
  const int n = e.hi - e.lo;     // keys of this split (0: past the sequence's keys)

  if (e.live && n > 0) {
    // RoPE factors of this thread's rotation pairs, fetched together with q/k/v
    const float2* rt = P.rope + (size_t)e.pos * (D / 2);
    constexpr int NROT = ((REP + 1) * (D / 2) + NT - 1) / NT;
    float2 cs[NROT];
#pragma unroll
    for (int j = 0; j < NROT; ++j) {
      const int i = t + j * NT;
      cs[j] = i < (rep + 1) * (D / 2) ? __ldg(rt + i % (D / 2)) : make_float2(0.f, 0.f);
    }
    // q of the group's heads, k and v: a bounded poll on their tags
    {
      const u64* base = P.qkv + ((size_t)l * P.max_batch + b) * P.qkv_rows;
      constexpr int NQ = ((REP + 2) * D + NT - 1) / NT;
      u64 wq[NQ];
      poll_until(P, S, [&]() {
        uint32_t bad = 0;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const int i = t + j * NT;
          if (i < (REP + 2) * D) {
            const u64* src = i < REP * D       ? base + g * REP * D + i
                             : i < (REP + 1) * D ? base + qd + g * D + (i - REP * D)
                                                 : base + qd + P.nkv * D + g * D + (i - (REP + 1) * D);
            wq[j] = ld_tagged(src);
            bad |= tag_of(wq[j]) ^ tag;
          }
        }
        return tag == 0u || bad == 0u;
      }, ii);
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        const int i = t + j * NT;
        if (i < REP * D) qs[i] = tag_val(wq[j]);
        else if (i < (REP + 1) * D) kn[i - REP * D] = tag_val(wq[j]);
        else if (i < (REP + 2) * D) vn[i - (REP + 1) * D] = round_bf16(tag_val(wq[j]));
      }
    }
    cbar();
    if (P.trace && t == 0) trace_mark(P, ii, 2);
    if (P.qk_norm) {
      const LayerW& W = layer_w(P, l);
      if (w <= rep) {
        float* u = w < rep ? qs + w * D : kn;
        const uint16_t* gn = w < rep ? W.q_norm : W.k_norm;
        float s = 0.f;
        for (int i = lane; i < D; i += 32) s = fmaf(u[i], u[i], s);
        s = warp_sum(s);
        const float inv = 1.0f / sqrtf(s / (float)D + P.eps);
        for (int i = lane; i < D; i += 32)
          u[i] = u[i] * inv * __uint_as_float((uint32_t)__ldg(gn + i) << 16);
      }
      cbar();
    }
#pragma unroll
    for (int j = 0; j < NROT; ++j) {
      const int i = t + j * NT;
      if (i < (rep + 1) * (D / 2)) {
        const int h = i / (D / 2), k = i % (D / 2);
        float* u = h < rep ? qs + h * D : kn;
        const float u1 = u[k], u2 = u[k + D / 2];
        const float r1 = u1 * cs[j].x - u2 * cs[j].y, r2 = u2 * cs[j].x + u1 * cs[j].y;
        // the new key enters attention as the bf16 cache stores it
        u[k] = h < rep ? r1 : round_bf16(r1);
        u[k + D / 2] = h < rep ? r2 : round_bf16(r2);
      }
    }
    cbar();
    attn_mark(P, ii, 8);
    if (e.has_new)
      for (int i = t; i < D; i += NT) {
        P.kv[kv_offset(P, l, 0, b, g, e.pos) + i] = __bfloat16_as_ushort(__float2bfloat16_rn(kn[i]));
        P.kv[kv_offset(P, l, 1, b, g, e.pos) + i] = __bfloat16_as_ushort(__float2bfloat16_rn(vn[i]));
      }

    const float scale = 1.0f / sqrtf((float)D);
    const int kps = (int)(STAGE_BYTES / (D * 2));
    if constexpr (REP <= 4) {
      // Scores of cached keys on the tensor cores, 8 keys per m16n8k16 product
      // per warp: A rows r < REP hold q of head r rounded to bf16, rows REP..
      // 2 REP - 1 the bf16 of its remainder (hi + lo keeps q's float32
      // precision against the exact bf16 keys), the other rows zero.  The
      // reduction index is permuted so that lane t's four values of k-step
      // 2 s + u are dimensions 32 s + 8 t + 4 u .. + 3: one 16-byte load per key
      // row gives two k-steps of B.
      constexpr int KSTEPS = D / 16;
      const int g = lane >> 2, tq = lane & 3;
      uint32_t af[KSTEPS][2];
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int base = 32 * (ks >> 1) + 8 * tq + 4 * (ks & 1);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t hv[2];
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const float qf = g < 2 * REP ? qs[(g % REP) * D + base + 2 * r + x] : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(qf);
            const __nv_bfloat16 v = g < REP ? hi : __float2bfloat16_rn(qf - __bfloat162float(hi));
            hv[x] = (uint32_t)__bfloat16_as_ushort(v);
          }
          af[ks][r] = hv[0] | (hv[1] << 16);
        }
      }
      for (int c0 = 0; c0 < e.nc; c0 += kps) {
        const int cnt = e.nc - c0 < kps ? e.nc - c0 : kps;
        const uint8_t* stage = ring_acquire(P, S, R);
        const int nblk = (cnt + 7) >> 3;
        for (int nb = w; nb < nblk; nb += NW) {
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          const uint8_t* row = stage + (size_t)(nb * 8 + g) * D * 2 + tq * 16;
#pragma unroll
          for (int s2 = 0; s2 < KSTEPS / 2; ++s2) {
            const uint4 kk = *reinterpret_cast<const uint4*>(row + s2 * 64);
            mma_bf16_16816(c, af[2 * s2][0], 0u, af[2 * s2][1], 0u, kk.x, kk.y);
            mma_bf16_16816(c, af[2 * s2 + 1][0], 0u, af[2 * s2 + 1][1], 0u, kk.z, kk.w);
          }
          // row g (hi) + row g + REP (lo): lanes 4 REP apart
          const float s0 = c[0] + __shfl_xor_sync(0xffffffffu, c[0], 4 * REP);
          const float s1 = c[1] + __shfl_xor_sync(0xffffffffu, c[1], 4 * REP);
          const int j = nb * 8 + 2 * tq;
          if (g < REP) {
            if (j < cnt) sc[g * smax + c0 + j] = s0 * scale;
            if (j + 1 < cnt) sc[g * smax + c0 + j + 1] = s1 * scale;
          }
        }
        ring_release(S, R);
      }
    } else {
      // scores of cached keys: 8 lanes per key, lane `sub` holds element groups
      // {sub, sub + 8, ...} of 8 (conflict-free 16-byte shared loads)
      constexpr int G = D / 64;  // 8-element groups per lane
      const int sub = lane & 7, quad = lane >> 3;
      float qv[REP][G][8];
#pragma unroll
      for (int h = 0; h < REP; ++h)
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
#pragma unroll
          for (int k = 0; k < 8; ++k) qv[h][gi][k] = qs[h * D + (sub + 8 * gi) * 8 + k];
      for (int c0 = 0; c0 < e.nc; c0 += kps) {
        const int cnt = e.nc - c0 < kps ? e.nc - c0 : kps;
        const uint8_t* stage = ring_acquire(P, S, R);
        for (int j0 = w * 4; j0 < cnt; j0 += NW * 4) {
          const int j = j0 + quad;
          const bool ok = j < cnt;
          const uint4* krow = reinterpret_cast<const uint4*>(stage + (size_t)(ok ? j : 0) * D * 2);
          float kx[G][8];
#pragma unroll
          for (int gi = 0; gi < G; ++gi) widen8(krow[sub + 8 * gi], kx[gi]);
#pragma unroll
          for (int h = 0; h < REP; ++h) {
            float a = 0.f;
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
#pragma unroll
              for (int k = 0; k < 8; ++k) a = fmaf(qv[h][gi][k], kx[gi][k], a);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            if (ok && sub == 0) sc[h * smax + c0 + j] = a * scale;
          }
        }
        ring_release(S, R);
      }
    }
    if (e.has_new && w < rep) {
      float a = 0.f;
      for (int i = lane; i < D; i += 32) a = fmaf(qs[w * D + i], kn[i], a);
      a = warp_sum(a);
      if (lane == 0) sc[w * smax + (e.pos - e.lo)] = a * scale;
    }
    cbar();
    attn_mark(P, ii, 9);
    // (max, sum) of head w stay in lane 0 of warp w until the partial's
    // outputs are stored: they are stored last, so a combining split that
    // sees them finds the outputs written too (normally; it checks their tags)
    float m_h = -INFINITY, s_h = 0.f;
    if (w < rep) {
      float m = -INFINITY;
      for (int j = lane; j < n; j += 32) m = fmaxf(m, sc[w * smax + j]);
      m = warp_max(m);
      float s = 0.f;
      for (int j = lane; j < n; j += 32) {
        const float p = expf(sc[w * smax + j] - m);
        sc[w * smax + j] = p;
        s += p;
      }
      s = warp_sum(s);
      m_h = m;
      s_h = s;
    }
    cbar();
    // o = sum_j p_j v_j.  Lane owns DPL consecutive columns, warp w a head
    // group (HPW heads) and the keys j = kw, kw + KS, ... of each stage, so
    // each V element is widened once for HPW heads; the KS key subsets of a
    // head group are then added in warp order through shared memory.
    constexpr int DPL = D / 32;                          // columns per lane
    constexpr int HPW = REP < 4 ? REP : 4;               // heads per warp
    constexpr int KS = NW / (REP / HPW);                 // key subsets per head group
    static_assert(NW * HPW * D <= SCORE_FLOATS, "P V reduction buffer");
    const int hg = w / KS, kw = w % KS;
    float acc[HPW][DPL];
#pragma unroll
    for (int h = 0; h < HPW; ++h)
#pragma unroll
      for (int k = 0; k < DPL; ++k) acc[h][k] = 0.f;
    for (int c0 = 0; c0 < e.nc; c0 += kps) {
      const int cnt = e.nc - c0 < kps ? e.nc - c0 : kps;
      const uint8_t* stage = ring_acquire(P, S, R);
      const float* ph = sc + (hg * HPW) * smax + c0;
#pragma unroll 4
      for (int j = kw; j < cnt; j += KS) {
        float vx[DPL];
        if constexpr (DPL == 4) {
          const uint2 u = *reinterpret_cast<const uint2*>(stage + (size_t)j * D * 2 + lane * 8);
          vx[0] = bf_lo(u.x); vx[1] = bf_hi(u.x); vx[2] = bf_lo(u.y); vx[3] = bf_hi(u.y);
        } else {
          const uint32_t u = *reinterpret_cast<const uint32_t*>(stage + (size_t)j * D * 2 + lane * 4);
          vx[0] = bf_lo(u); vx[1] = bf_hi(u);
        }
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const float p = ph[h * smax + j];
#pragma unroll
          for (int k = 0; k < DPL; ++k) acc[h][k] = fmaf(p, vx[k], acc[h][k]);
        }
      }
      ring_release(S, R);
    }
    // the new key's probability for this thread's outputs, read before sc is reused
    const float p_new0 = (e.has_new && t < rep * D) ? sc[(t / D) * smax + (e.pos - e.lo)] : 0.f;
    const float p_new1 = (e.has_new && t + NT < rep * D) ? sc[((t + NT) / D) * smax + (e.pos - e.lo)] : 0.f;
    const float p_new2 = (e.has_new && t + 2 * NT < rep * D) ? sc[((t + 2 * NT) / D) * smax + (e.pos - e.lo)] : 0.f;
    const float p_new3 = (e.has_new && t + 3 * NT < rep * D) ? sc[((t + 3 * NT) / D) * smax + (e.pos - e.lo)] : 0.f;
    cbar();  // every warp is done reading the probabilities: reuse sc
    float* red = sc;  // [NW][HPW][D]
#pragma unroll
    for (int h = 0; h < HPW; ++h)
#pragma unroll
      for (int k = 0; k < DPL; ++k) red[(w * HPW + h) * D + lane * DPL + k] = acc[h][k];
    cbar();
    for (int i = t, k = 0; i < rep * D; i += NT, ++k) {
      const int h = i / D, c = i % D;
      const int g2 = h / HPW, hh = h % HPW;
      float o = 0.f;
#pragma unroll
      for (int q = 0; q < KS; ++q) o += red[((g2 * KS + q) * HPW + hh) * D + c];
      if (e.has_new) {
        const float pn = k == 0 ? p_new0 : k == 1 ? p_new1 : k == 2 ? p_new2 : p_new3;
        o = fmaf(pn, vn[c], o);
      }
      st_tagged(part + h * (D + 2) + c, o, ptag);
    }
    cbar();  // every output of the partial is stored
    if (w < rep && lane == 0) {
      st_tagged(part + w * (D + 2) + D, m_h, ptag);
      st_tagged(part + w * (D + 2) + D + 1, s_h, ptag);
    }
    attn_mark(P, ii, 10);
  } else if (P.trace && t == 0) {
    trace_mark(P, ii, 2);
  }
  if ((in.flags & IF_COMBINE) && e.live) {
    // Combine the group's live splits (those holding keys: ceil((pos + 1) /
    // KPS) of them) in split order: weights f_s = exp(m_s - max_s m_s) per
    // head (staged in shared memory), o = sum_s f_s o_s / sum_s f_s l_s.  Every
    // partial is a bounded poll on its tags.  A slice instruction combines
    // outputs [o0, o1) of the group's rep * D (every slice reads all splits'
    // max and sum, and only its own outputs' partial values).
    const int nl = (e.pos + P.kps) / P.kps;  // ceil((pos + 1) / KPS)
    const int per = (in.flags & IF_SLICE) ? P.comb_per : rep * D;
    const int o0 = (in.flags & IF_SLICE) ? split * per : 0;
    const int o1 = o0 + per < rep * D ? o0 + per : rep * D;
    const u64* gp = P.part + (((size_t)l * P.max_batch + b) * P.nkv + g) * NS * rep * (D + 2);
    cbar();  // the scratch in xbuf is free (this split's own work is done)
    float* fw = S.xbuf;                 // [nl][rep] weights
    float* lw = S.xbuf + NS * rep;      // [nl][rep] partial sums
    float* linv = lw + NS * rep;        // [rep]
    // This thread's (head, column) outputs: their partial values are read CB
    // splits at a time (every load of a batch in flight together); the first
    // batch goes out once every split's (max, sum) is in, so its round trip
    // overlaps the weights' computation, and is checked afterwards.
    constexpr int NO = (REP * D + NT - 1) / NT;
    constexpr int CB = NO <= 2 ? 20 : 8;
    float v[NO][CB];
    // Every load of a batch is issued before any result is used: lanes past
    // the slice or splits past nl read a valid word of the slice (clamped
    // indices) whose value is then dropped, so no load sits behind a branch
    // (predicated loads measured slower: the compiler no longer kept them in
    // flight together); a warp whose outputs all lie past the slice issues
    // none.
    auto load_batch = [&](int s0) {
      uint32_t bad = 0;
      u64 wv[NO][CB];
#pragma unroll
      for (int k = 0; k < NO; ++k) {
        const int i = o0 + t + k * NT;
        const int ic = i < o1 ? i : o1 - 1;
        const u64* pc = gp + (size_t)(ic / D) * (D + 2) + (ic % D);
        if (o0 + (t & ~31) + k * NT < o1) {  // warp-uniform
#pragma unroll
          for (int u = 0; u < CB; ++u) {
            const int sc = s0 + u < nl ? s0 + u : nl - 1;
            wv[k][u] = ld_tagged(pc + (size_t)sc * rep * (D + 2));
          }
        } else {
#pragma unroll
          for (int u = 0; u < CB; ++u) wv[k][u] = 0ull;
        }
      }
#pragma unroll
      for (int k = 0; k < NO; ++k) {
        const int i = o0 + t + k * NT;
#pragma unroll
        for (int u = 0; u < CB; ++u) {
          const bool use = i < o1 && s0 + u < nl;
          v[k][u] = use ? tag_val(wv[k][u]) : 0.f;
          bad |= use ? (tag_of(wv[k][u]) ^ tag) : 0u;
        }
      }
      return bad;
    };
    for (int i = t; i < nl * rep; i += NT) {
      const u64* ps = gp + (size_t)i * (D + 2) + D;
      u64 mw = 0, lw2 = 0;
      poll_until(P, S, [&]() {
        ld_tagged2(ps, mw, lw2);
        return tag == 0u || ((tag_of(mw) ^ tag) | (tag_of(lw2) ^ tag)) == 0u;
      }, ii);
      fw[i] = tag_val(mw);
      lw[i] = tag_val(lw2);
    }
    cbar();
    attn_mark(P, ii, 11);
    const uint32_t bad0 = load_batch(0);
    if (w < rep) {
      float M = -INFINITY;
      for (int s = lane; s < nl; s += 32) M = fmaxf(M, fw[s * rep + w]);
      M = warp_max(M);
      float Ls = 0.f;
      for (int s = lane; s < nl; s += 32) {
        const float ms = fw[s * rep + w];
        const float f = ms == -INFINITY ? 0.f : expf(ms - M);
        fw[s * rep + w] = f;
        Ls = fmaf(lw[s * rep + w], f, Ls);
      }
      Ls = warp_sum(Ls);
      if (lane == 0) linv[w] = 1.0f / Ls;
    }
    cbar();
    // o = sum_s f_s o_s in split order
    float O[NO];
#pragma unroll
    for (int k = 0; k < NO; ++k) O[k] = 0.f;
    for (int s0 = 0; s0 < nl; s0 += CB) {
      if (s0 > 0 || (tag != 0u && bad0 != 0u))
        poll_until(P, S, [&]() { return load_batch(s0) == 0u || tag == 0u; }, ii);
#pragma unroll
      for (int k = 0; k < NO; ++k) {
        const int h = (o0 + t + k * NT) / D;
#pragma unroll
        for (int u = 0; u < CB; ++u)
          if (s0 + u < nl) O[k] = fmaf(v[k][u], fw[(s0 + u) * rep + h], O[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < NO; ++k) {
      const int i = o0 + t + k * NT;
      if (i < o1) {
        const int h = i / D, c = i % D;
        st_tagged(P.attn_out + ((size_t)l * P.max_batch + b) * qd + (size_t)(g * rep + h) * D + c,
                  O[k] * linv[h], ptag);
      }
    }
  }
  // no barrier here: the next instruction's slot hand-off orders every reuse
  // of the shared scratch
}

template <int AD, int AREP>
__device__ __forceinline__ void attn_dispatch(const KParams& P, const Sh& S, const Instr& in, const AttnExt& e,
                              uint32_t ii, uint32_t tag, Ring& R) {
  if constexpr (AD != 0) {
    attn_tile<AD, AREP>(P, S, in, e, ii, tag, R);
  } else if (P.d == 128) {
    switch (P.rep) {
      case 1: attn_tile<128, 1>(P, S, in, e, ii, tag, R); break;
      case 2: attn_tile<128, 2>(P, S, in, e, ii, tag, R); break;
      case 4: attn_tile<128, 4>(P, S, in, e, ii, tag, R); break;
      default: attn_tile<128, 8>(P, S, in, e, ii, tag, R); break;
    }
  } else {
    switch (P.rep) {
      case 1: attn_tile<64, 1>(P, S, in, e, ii, tag, R); break;
      case 2: attn_tile<64, 2>(P, S, in, e, ii, tag, R); break;
      case 4: attn_tile<64, 4>(P, S, in, e, ii, tag, R); break;
      default: attn_tile<64, 8>(P, S, in, e, ii, tag, R); break;
    }
  }
}

// Drain an instruction's stages without computing (after an abort).
__device__ __forceinline__ void drain(const KParams& P, const Sh& S, const Instr& in, const AttnExt& e,
                                      Ring& R) {
  const uint32_t n = src_stages(src_of(P, in, e));
  for (uint32_t k = 0; k < n; ++k) {
    ring_acquire(P, S, R);
    ring_release(S, R);
  }
}

// ---------------------------------------------------------------- consumer loop
// MH, MF: K / FAST_K_UNIT of the hidden size and of the FFN size for the
// batch-1 register path (0: the shared-memory path only).  AD, AREP: head_dim
// and q heads per kv head of the attention tile (0: chosen at run time).
template <int MH, int MF, int AD, int AREP, bool MS>
__device__ void consumer(const KParams& P, const Sh& S) {
  const int t = threadIdx.x;
  Ring R{0, 0, 0, 0, false, false};
  uint32_t islot_ctr = 0;
  const uint32_t gen = S.flags[F_GEN];
  constexpr int XH = MH > 0 ? MH : 1, XF = MF > 0 ? MF : 1;
  constexpr int XM = XH > XF ? XH : XF;
  // The activation vector stays in registers while consecutive tiles read it
  // (same operator and layer): the tag names what it holds.  One array serves
  // both widths (every operator change reloads it anyway).
  float xr[XM][8];
  uint32_t tag_x = 0xffffffffu;
  for (;;) {
    const int si = islot_ctr % NISLOT;
    // The broadcast words are double-buffered by instruction parity: warps
    // 1..7 may still be reading this instruction's words while warp 0 (which
    // finishes every batch-1 tile) already fills in the next instruction's.
    const int f_slot = (islot_ctr & 1u) ? F_SLOT_B : F_SLOT;
    const int f_abort = (islot_ctr & 1u) ? F_ABORT_B : F_ABORT;
    const uint64_t t_top = (P.trace && t == 0) ? globaltimer() : 0;
    // One thread takes the slot (a bounded wait) and hands it, with the stop
    // verdict, to every consumer thread through one consumer barrier (which
    // also keeps the warps of a tile in step, so the ring's stages are freed
    // together).  The tiles' dependencies are not waited on here: each tile
    // polls the tags of the words it reads (poll_until).
    if (t == 0) {
      uint32_t v = 0xffffffffu;
      if (mbar_wait(P, &S.ifull[si], (islot_ctr / NISLOT) & 1u)) v = *slot_index(S, si);
      S.flags[f_slot] = v;
      const uint32_t iv = (!MS || v == END_SLOT) ? v : v & ((1u << SLOT_INDEX_BITS) - 1u);
      const uint32_t aborted = S.flags[F_STOP];
      const uint64_t t_begin = P.trace ? globaltimer() : 0;
      S.flags[f_abort] = aborted;
      if (aborted) S.flags[F_STOP] = 1u;  // the producer stops popping
      if (P.trace && iv != END_SLOT) {
        unsigned long long* tr = P.trace + (size_t)iv * TRACE_WORDS;
        tr[12] = t_top;
        tr[1] = t_begin;
        R.cur = iv;
      }
    }
    cbar();
    if (P.trace && t == 0 && S.flags[f_slot] != END_SLOT) trace_mark(P, R.cur, 10);
    const uint32_t slotv = S.flags[f_slot];
    const uint32_t i = (!MS || slotv == END_SLOT) ? slotv : slotv & ((1u << SLOT_INDEX_BITS) - 1u);
    const uint32_t step = (!MS || slotv == END_SLOT) ? 0u : slotv >> SLOT_INDEX_BITS;
    Instr in;
    AttnExt ext;
    ext.live = false;
    if (i != END_SLOT) {
      in = *slot_instr(S, si);
      if (in.op == OP_ATTN) ext = slot_get_ext(S, si);
    }
    const bool aborted_now = S.flags[f_abort] != 0u;
    __syncwarp();
    if ((t & 31) == 0) mbar_arrive(&S.iempty[si]);
    ++islot_ctr;
    if (i == END_SLOT) break;
    if (aborted_now) {
      drain(P, S, in, ext, R);
      continue;
    }
    const uint32_t tag = step_tag(P, gen, step);
    // The batch-1 GEMV tiles (most instructions) come first in the code, so
    // their dispatch path stays short and contiguous; the finisher stores and
    // publishes them.
    if (MH > 0 && P.B == 1 && in.op != OP_ATTN) {
      const GemvDesc g = gemv_desc(P, in);
      const Src src = instr_src(P, in);
      const uint32_t xtag = (uint32_t)in.op | ((uint32_t)in.layer << 8) | (step << 24);
      if (in.op != OP_DOWN) {
        auto& xh = *reinterpret_cast<float(*)[XH][8]>(&xr);
        if (xtag != tag_x) {
          load_x_fast<XH, MS>(P, S, in, xh, step, tag);
          tag_x = xtag;
        }
        if (P.trace && t == 0) trace_mark(P, i, 2);
        gemv_fast<XH, MS>(P, S, in, i, step, tag, g, src, R, xh);
      } else {
        auto& xf = *reinterpret_cast<float(*)[XF][8]>(&xr);
        if (xtag != tag_x) {
          load_x_plain<XF>(P, S, gemv_x(P, in), xf, tag);
          tag_x = xtag;
        }
        if (P.trace && t == 0) trace_mark(P, i, 2);
        gemv_fast<XF, MS>(P, S, in, i, step, tag, g, src, R, xf);
      }
    } else if (in.op == OP_ATTN) {
      attn_dispatch<AD, AREP>(P, S, in, ext, i, tag, R);
      // Every GEMV after attention reloads its activations; overwriting the
      // register copies here makes them dead during the attention tile, so
      // attention does not have to spill around them.
#pragma unroll
      for (int j = 0; j < XM; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) xr[j][e] = 0.f;
      tag_x = 0xffffffffu;
    } else {
      const GemvDesc g = gemv_desc(P, in);
      const Src src = instr_src(P, in);
      const u64 pre_w = epilogue_prefetch<false>(P, S, in, g, t);
      gemv_generic(P, S, in, g, src, R, tag);
      if (P.trace && t == 0) trace_mark(P, i, 2);
      gemv_epilogue(P, S.red, in, g, epilogue_resolve(P, S, in, g, t, pre_w, tag), t, pub_tag(in, tag));
    }
    if (P.trace && t == 0) {
      unsigned long long* tr = P.trace + (size_t)i * TRACE_WORDS;
      tr[0] = (unsigned long long)smid() | ((unsigned long long)(in.op | (in.layer << 8)) << 32);
      if (!R.handed) tr[3] = globaltimer();  // handed-off tiles: the finisher writes it
      tr[5] = R.wait_ns;
    }
    R.wait_ns = 0;
    R.first_done = false;
    R.handed = false;
    // no barrier here: the next instruction's slot and the tiles' own barriers
    // order every reuse of the shared scratch
  }
  // tell the finisher that no more tiles come
  const int hb = handoff_acquire(P, S, R);
  if (t == 0) *hrec_index(S, hb) = END_SLOT;
  handoff_commit(S, R, hb);
}

// One LM-head tile of a multi-step launch (finisher warp, batch 1): the
// tile's largest logit (lane r holds row r's in `y`) folded into this CTA's
// running choice for the step, stored with the CTA's tile count.  Runs before
// the tile's logits are stored (only the launch's last step stores them).
__device__ __forceinline__ void lm_tile_choose(const KParams& P, const GemvDesc& g, uint32_t step, int lane,
                                               float y, uint32_t& cur_step, unsigned long long& run) {
  unsigned long long key = 0;
  if (lane < g.rows) key = lm_pack(y, (uint32_t)(g.row0 + lane));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
    key = other > key ? other : key;
  }
  if (lane == 0) {
    if (step != cur_step) {  // a CTA meets the steps in order
      cur_step = step;
      run = 0;
    }
    const unsigned long long cnt = (run & LM_CNT_MASK) + 1;
    const unsigned long long m = (run & ~LM_CNT_MASK) > key ? (run & ~LM_CNT_MASK) : key;
    run = m | cnt;
    unsigned long long* slot = P.lm_slot + (size_t)step * gridDim.x + blockIdx.x;
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(slot), "l"(run) : "memory");
  }
}

// The tokens a multi-step launch chose, into out_tokens (the last CTA to
// leave the launch, all its threads): every CTA's words are final by then.
__device__ void lm_write_tokens(const KParams& P) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  for (uint32_t s = (uint32_t)w; s < P.n_steps; s += NTHREADS / 32) {
    const unsigned long long* words = P.lm_slot + (size_t)s * gridDim.x;
    unsigned long long m = 0;
    for (uint32_t c = (uint32_t)lane; c < gridDim.x; c += 32) {
      const unsigned long long v = __ldcg(words + c) & ~LM_CNT_MASK;
      m = v > m ? v : m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long om = __shfl_xor_sync(0xffffffffu, m, o);
      m = om > m ? om : m;
    }
    if (lane == 0) {
      const int row = lm_row(m);
      P.out_tokens[s] = row < P.V ? row : 0;
    }
  }
}

// ---------------------------------------------------------------- finisher warp
// Takes the batch-1 GEMV tiles in hand-off order: adds up the consumer warps'
// partial sums (fixed order), frees the buffer and stores the outputs
// (residual adds, SwiGLU) as tagged words, which publishes them: the
// consumers poll the tags, so no fence or counter release follows and the
// store latency stays off the consumers' path.
template <bool MS>
__device__ void finisher(const KParams& P, const Sh& S) {
  const int lane = threadIdx.x & 31;
  const uint32_t gen = S.flags[F_GEN];
  uint32_t lm_step = 0xffffffffu;  // multi-step: the step of this CTA's running choice
  unsigned long long lm_run = 0;
  for (uint32_t h = 0;; ++h) {
    const int hb = (int)(h & 1u);
    if (!mbar_wait(P, &S.hfull[hb], (h >> 1) & 1u)) break;
    const uint32_t ii = *hrec_index(S, hb);
    if (ii == END_SLOT) break;
    const Instr in = *hrec_instr(S, hb);
    const uint64_t t_take = P.trace ? globaltimer() : 0;
    const GemvDesc g = gemv_desc(P, in);
    const int ntot = g.w1 ? 2 * g.rows : g.rows;
    const float* redw = S.redw + hb * NW * RMAX;
    if (lane < ntot) {
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < NW; ++k) s += redw[k * RMAX + lane];
      S.fin[lane * BMAX_CC] = s;
    }
    const float pre = S.hpre[hb * RMAX + lane];
    const uint32_t step = MS ? *hrec_step(S, hb) : 0u;
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.hempty[hb]);
    if (P.trace && lane == 0) P.trace[(size_t)ii * TRACE_WORDS + 14] = globaltimer();
    if (MS && in.op == OP_LM) {
      // greedy choice from the registers; the logits of steps before the
      // launch's last are not returned, so they are not stored
      lm_tile_choose(P, g, step, lane, S.fin[lane * BMAX_CC], lm_step, lm_run);
      if (step + 1u == P.n_steps) gemv_epilogue(P, S.fin, in, g, pre, lane, 0u);
    } else {
      gemv_epilogue(P, S.fin, in, g, pre, lane, pub_tag(in, step_tag(P, gen, step)));
    }
    __syncwarp();
    if (lane == 0) {
      if (P.trace) {
        unsigned long long* tr = P.trace + (size_t)ii * TRACE_WORDS;
        tr[9] = t_take;
        tr[3] = globaltimer();
      }
    }
  }
  // this CTA's choice words are visible before the launch's last CTA reads
  // them to write the chosen tokens
  if (MS && lane == 0) __threadfence();
}

template <int MH, int MF, int AD, int AREP, bool MS>
__global__ void __launch_bounds__(NTHREADS, 1) mk_interpreter(const __grid_constant__ KParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Sh S = sh_map(smem);
  const int t = threadIdx.x;
  if (t == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], NW);
    }
    for (int s = 0; s < NISLOT; ++s) {
      mbar_init(&S.ifull[s], 1);
      mbar_init(&S.iempty[s], NW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.hfull[b], NW);
      mbar_init(&S.hempty[b], 1);
    }

    fence_mbar_init();
    fence_proxy_async_smem();
    S.flags[F_GEN] = P.mode == MODE_MEGA ? ld_volatile(&P.ctl[CTL_GEN]) : 0u;
    S.flags[F_STOP] = 0u;
    S.flags[F_POLL] = 0u;
  }
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(P.layers);
    uint32_t* dst = reinterpret_cast<uint32_t*>(smem + SmemLayout::layers);
    const int words = P.L * (int)(sizeof(LayerW) / 4);
    for (int i = t; i < words; i += NTHREADS) dst[i] = src[i];
  }
  __syncthreads();
  // Register split: the launch gives every thread the same count (168 at 12
  // warps); the producer/finisher warpgroup (warps 8-11: producer, finisher,
  // two idle warps) gives most of its share to the two consumer warpgroups.
  // Shares: 8 consumer warps x 224 + 4 warps x 56 = 12 warps x 168 per thread.
  if (t >= NT) {
    setmaxnreg_dec<SPLIT_REGS_SIDE>();
    if (t < NT + 32) producer<MS>(P, S);
    else if (t < NT + 64) finisher<MS>(P, S);

  } else {
    setmaxnreg_inc<SPLIT_REGS_CONSUMER>();
    consumer<MH, MF, AD, AREP, MS>(P, S);
  }
  __syncthreads();
  if (t == 0 && P.mode == MODE_MEGA) {
    __threadfence();
    const uint32_t old = atomicAdd(&P.ctl[CTL_EXIT], 1u);
    S.flags[F_LAST] = old == gridDim.x - 1 ? 1u : 0u;
    if (old == gridDim.x - 1) {
      // every CTA has left its loop: rewind the queue head for the next launch
      P.ctl[CTL_HEAD] = 0u;
      P.ctl[CTL_EXIT] = 0u;
      P.ctl[CTL_GEN] = S.flags[F_GEN] + (MS ? P.n_steps : 1u);
      __threadfence();
    }
  }
  if (MS && P.mode == MODE_MEGA) {
    __syncthreads();
    if (S.flags[F_LAST]) {
      __threadfence();
      lm_write_tokens(P);
    }
  }
}

// ---------------------------------------------------------------- host-side launch helpers
// The register split (setmaxnreg) adds up only if the launch gives each thread
// exactly LAUNCH_REGS registers; with fewer, the consumer warps' increase
// could never be granted, so such a build is refused instead of launched.
template <class K>
cudaError_t check_launch_regs(K kernel) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, kernel);
  if (e != cudaSuccess) return e;
  return a.numRegs == LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int MH, int MF, int AD, int AREP>
struct VariantImpl {
  static cudaError_t setup() {
    cudaError_t e = cudaFuncSetAttribute(mk_interpreter<MH, MF, AD, AREP, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SmemLayout::total);
    if (e == cudaSuccess) e = check_launch_regs(mk_interpreter<MH, MF, AD, AREP, false>);
    if (e != cudaSuccess || MH == 0) return e;
    e = cudaFuncSetAttribute(mk_interpreter<MH, MF, AD, AREP, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SmemLayout::total);
    if (e == cudaSuccess) e = check_launch_regs(mk_interpreter<MH, MF, AD, AREP, true>);
    return e;
  }
  static cudaError_t occupancy(int* per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, mk_interpreter<MH, MF, AD, AREP, false>,
                                                         NTHREADS, SmemLayout::total);
  }
  static cudaError_t mega(const KParams& p, int ctas, cudaStream_t st) {
    KParams pp = p;
    void* args[] = {(void*)&pp};
    return cudaLaunchCooperativeKernel((const void*)mk_interpreter<MH, MF, AD, AREP, false>, dim3(ctas),
                                       dim3(NTHREADS), args, (size_t)SmemLayout::total, st);
  }
  // the multi-step kernel (mk_decode_steps; batch-1 register path only)
  static cudaError_t mega_steps(const KParams& p, int ctas, cudaStream_t st) {
    if (MH == 0) return cudaErrorNotSupported;
    KParams pp = p;
    void* args[] = {(void*)&pp};
    return cudaLaunchCooperativeKernel((const void*)mk_interpreter<MH, MF, AD, AREP, MH != 0>, dim3(ctas),
                                       dim3(NTHREADS), args, (size_t)SmemLayout::total, st);
  }
  // one launch of an operator's `count` tiles on at most `ctas` CTAs
  static cudaError_t perop(const KParams& p, uint32_t first, uint32_t count, int ctas, cudaStream_t st) {
    KParams pp = p;
    pp.mode = MODE_PEROP;
    pp.perop_base = first;
    pp.perop_count = count;
    const uint32_t grid = count < (uint32_t)ctas ? count : (uint32_t)ctas;
    mk_interpreter<MH, MF, AD, AREP, false><<<grid, NTHREADS, SmemLayout::total, st>>>(pp);
    return cudaGetLastError();
  }
};

}  // namespace

template <int MH, int MF, int AD, int AREP>
KernelVariant make_variant() {
  using V = VariantImpl<MH, MF, AD, AREP>;
  KernelVariant k;
  k.mh = MH;
  k.mf = MF;
  k.ad = AD;
  k.arep = AREP;
  k.setup = &V::setup;
  k.occupancy = &V::occupancy;
  k.mega = &V::mega;
  k.mega_steps = &V::mega_steps;
  k.perop = &V::perop;
  return k;
}

}  // namespace mk
