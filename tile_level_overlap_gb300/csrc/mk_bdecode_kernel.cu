// Batched decode interpreter (sm_103a): tensor-core GEMM tiles, CUDA-core
// split-KV attention, RMSNorm blocks; one persistent CTA per SM, tile-level
// dependencies through barrier counters (see mk_bdecode.h).
//
//  warp 0      producer: pops instructions (one atomic each), streams the
//              weight k-blocks of a GEMM tile ahead of its dependencies and
//              the activation k-blocks (hi and lo planes) once they are
//              satisfied, or the K/V blocks of an attention split, with 2D TMA
//              loads into a 6 x 32 KB ring.
//  warp 1      tensor-core issuer: D[128 weight rows][N batch columns] +=
//              W_tile * x_hi^T, then * x_lo^T, per k-step (tcgen05.mma,
//              accumulators in TMEM, two 32-column accumulators).
//  warps 2-9   compute: split-K partial sums, the last chunk's reduction and
//              epilogue (the two warps of a TMEM lane quarter take 16 batch
//              columns each), the layer-0 RMSNorm, the attention splits and
//              their combine.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mk.h"
#include "mk_bdecode.h"
#include "mk_device.cuh"
#include "mk_internal.h"
#include "mk_plan.h"
#include "mk_tc.cuh"

namespace mk {
namespace {

constexpr int BD_STAGE = 32 * 1024;
constexpr int BD_NSTAGE = 6;
// Weight stages a GEMM tile streams before its dependencies are met: the
// dependency poll's reads return behind the copies already in flight, so a
// full ring of weights delayed the tile's start; three keep most of the
// prefetch (Llama-3-8B batch 8: 5.185 -> 5.062 ms, Qwen3-8B batch 32 ragged:
// 6.89 -> 6.83 ms; 2 and 4 stages measured slower).
constexpr int BD_PRE_STAGES = 3;
constexpr int BD_THREADS = 320;
constexpr int BD_CBAR = 2;   // named barrier of the compute warps
constexpr int BD_GBAR0 = 3;  // named barriers of the attention's two warp groups (3, 4)
constexpr int BD_NC = 256;   // compute threads (8 warps: two per TMEM lane quarter)
constexpr uint32_t BD_END = 0xffffffffu;
constexpr uint32_t BD_W_BYTES = BD_M * BD_BK * 2;  // weight box(es) of a stage: 16 KB
constexpr int BD_ACC_COLS = 32;                    // TMEM columns per accumulator

struct BdSmem {
  static constexpr int ring = 0;
  static constexpr int scratch = ring + BD_NSTAGE * BD_STAGE;  // [128][BD_NMAX] f32
  static constexpr int qs = scratch + BD_M * BD_NMAX * 4;      // [4][128] f32
  static constexpr int sc = qs + 4 * 128 * 4;                  // [2 groups][4][BD_KEYS] f32
  static constexpr int hs = sc + 2 * 4 * BD_KEYS * 4;          // [2 groups][16]: [4] x {m, l, alpha}; inv norms [64] from 16
  static constexpr int rinv = hs + (16 + 64) * 4;             // [BD_NMAX] 1 / rms per sequence
  static constexpr int bars = rinv + BD_NMAX * 4;
  // full[6] empty[6] ifull[8] iempty[8] accf[2] acce[2]
  static constexpr int n_mbar = 2 * BD_NSTAGE + 2 * NISLOT + 4;
  static constexpr int islot = bars + n_mbar * 8;
  static constexpr int flags = islot + NISLOT * 48;  // [16] u32
  static constexpr int seq = flags + 16 * 4;         // positions, tokens, cache slots [BD_NMAX] each
  static constexpr int total = seq + 3 * BD_NMAX * 4;
};
static_assert(BdSmem::total <= 227 * 1024, "batched decode shared memory budget");
static_assert(BdSmem::scratch % 1024 == 0, "ring stages stay 1024-aligned");

enum BdFlag { BF_GEN = 0, BF_SLOT = 1, BF_ABORT = 2, BF_TMEM = 3, BF_LAST = 4 };

struct BdSh {
  uint8_t* ring;
  float *scratch, *qs, *sc, *hs, *rinv;
  uint64_t *full, *empty, *ifull, *iempty, *accf, *acce;
  uint8_t* islot;
  volatile uint32_t* flags;
  int32_t *pos, *tok, *slot;
};

__device__ __forceinline__ BdSh bd_map(uint8_t* base) {
  BdSh s;
  s.ring = base + BdSmem::ring;
  s.scratch = reinterpret_cast<float*>(base + BdSmem::scratch);
  s.qs = reinterpret_cast<float*>(base + BdSmem::qs);
  s.sc = reinterpret_cast<float*>(base + BdSmem::sc);
  s.hs = reinterpret_cast<float*>(base + BdSmem::hs);
  s.rinv = reinterpret_cast<float*>(base + BdSmem::rinv);
  uint64_t* b = reinterpret_cast<uint64_t*>(base + BdSmem::bars);
  s.full = b;
  s.empty = b + BD_NSTAGE;
  s.ifull = b + 2 * BD_NSTAGE;
  s.iempty = s.ifull + NISLOT;
  s.accf = s.iempty + NISLOT;
  s.acce = s.accf + 2;
  s.islot = base + BdSmem::islot;
  s.flags = reinterpret_cast<volatile uint32_t*>(base + BdSmem::flags);
  s.pos = reinterpret_cast<int32_t*>(base + BdSmem::seq);
  s.tok = s.pos + BD_NMAX;
  s.slot = s.tok + BD_NMAX;
  return s;
}

__device__ void bd_error(const BdParams& P, uint32_t code, uint32_t detail) {
  if (atomicCAS(&P.ctl[CTL_STATUS], 0u, code) == 0u) atomicExch(&P.ctl[CTL_DETAIL], detail);
  atomicExch(&P.ctl[CTL_ABORT], 1u);
}

// Bounded mbarrier wait; after an abort (another wait already gave up) it
// gives up within ~10 us so a broken launch drains.
__device__ __forceinline__ bool bd_wait(const BdParams& P, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t dt = globaltimer() - t0;
    if (dt > P.wait_limit_ns * 4ull) {
      bd_error(P, MK_ERR_TIMEOUT, 0xfffffff2u);
      return false;
    }
    if ((it & 255u) == 0 && dt > 10000ull && ld_volatile(&P.ctl[CTL_ABORT]) != 0u) return false;
  }
}

// Bounded acquire-spin on the counters an instruction waits on: wait_n
// counters, wait_stride apart, each to wait_target releases per step.
__device__ bool bd_wait_deps(const BdParams& P, const Instr& in, uint32_t gen, uint32_t idx) {
  if (P.mode != MODE_MEGA || in.wait_bar == NO_BAR) return true;
  const uint32_t target = (gen + 1u) * in.wait_target;
  const uint64_t t0 = globaltimer();
  for (uint32_t k = 0; k < in.wait_n;) {
    const uint32_t* c = &P.bars[in.wait_bar + k * in.wait_stride];
    if ((int32_t)(ld_acquire_gpu(c) - target) >= 0) {
      ++k;
      continue;
    }
    if (ld_volatile(&P.ctl[CTL_ABORT]) != 0u) return false;
    if (globaltimer() - t0 > P.wait_limit_ns) {
      bd_error(P, MK_ERR_TIMEOUT, idx);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

__device__ __forceinline__ void bd_mark(const BdParams& P, uint32_t i, int word) {
  if (P.trace) P.trace[(size_t)i * TRACE_WORDS + word] = globaltimer();
}

__device__ __forceinline__ const CUtensorMap* tmap(const BdParams& P, int idx) {
  return reinterpret_cast<const CUtensorMap*>(P.tm) + idx;
}
__device__ __forceinline__ int gmap(const BdParams& P, int which) {
  return P.L * BD_TM_PER_LAYER + which;
}

__device__ __forceinline__ bool is_gemm(uint8_t op) {
  return op == BD_QKV || op == BD_O || op == BD_GU || op == BD_DOWN || op == BD_LM;
}
__device__ __forceinline__ bool is_norm(uint8_t op) {
  return op == BD_NORM1 || op == BD_NORM2 || op == BD_NORMF;
}

// GEMM geometry of an instruction (row tile a0, K chunk a1).
struct BdGemm {
  int K;                    // full reduction length
  int k0, nk;               // first column and 64-column steps of this chunk
  int chunks;               // chunks of the row tile
  int a_map, a_row;         // weight map and first row (GU: gate map; up map = a_map + 1)
  bool gu;                  // two 64-row weight boxes (gate, up)
  int x_map;                // activation map (hi rows [0, nb), lo rows [nb, 2 nb))
  uint32_t pslot;           // first split-K partial slot of the row tile
  uint32_t arr;             // its arrival counter
};

__device__ __forceinline__ BdGemm bd_gemm(const BdParams& P, const Instr& in) {
  BdGemm g;
  const int l = in.layer, m = (int)in.a0, c = (int)in.a1;
  const int qd = P.nq * P.d, kd = P.nkv * P.d;
  g.gu = false;
  switch (in.op) {
    case BD_QKV: {
      g.K = P.H;
      g.chunks = (int)P.c_k;
      g.x_map = gmap(P, TMB_HN);
      const int r = m * BD_M;
      if (r < qd) { g.a_map = l * BD_TM_PER_LAYER + TMB_WQ; g.a_row = r; }
      else if (r < qd + kd) { g.a_map = l * BD_TM_PER_LAYER + TMB_WK; g.a_row = r - qd; }
      else { g.a_map = l * BD_TM_PER_LAYER + TMB_WV; g.a_row = r - qd - kd; }
      break;
    }
    case BD_O:
      g.K = qd;
      g.chunks = (int)P.c_q;
      g.x_map = gmap(P, TMB_AO);
      g.a_map = l * BD_TM_PER_LAYER + TMB_WO;
      g.a_row = m * BD_M;
      break;
    case BD_GU:
      g.K = P.H;
      g.chunks = (int)P.c_g;
      g.x_map = gmap(P, TMB_HN);
      g.a_map = l * BD_TM_PER_LAYER + TMB_WG;
      g.a_row = m * (BD_M / 2);
      g.gu = true;
      break;
    case BD_DOWN:
      g.K = P.F;
      g.chunks = (int)P.c_f;
      g.x_map = gmap(P, TMB_ACT);
      g.a_map = l * BD_TM_PER_LAYER + TMB_WD;
      g.a_row = m * BD_M;
      break;
    default:  // BD_LM: one chunk (its 128-row tiles are plentiful)
      g.K = P.H;
      g.chunks = 1;
      g.x_map = gmap(P, TMB_HN);
      g.a_map = gmap(P, TMB_LM);
      g.a_row = m * BD_M;
      break;
  }
  // Partial sums and arrival counters are indexed by the row tile within the
  // operator, in one of two regions: O and down in the first, QKV and gate/up
  // in the second.  A chunk can start while row tiles of the operator before
  // it still sum their chunks (it waits only on the tiles it reads), but not
  // while the operator before that one does, so alternating regions suffice.
  const bool rb = in.op == BD_QKV || in.op == BD_GU;
  g.pslot = (rb ? P.part_b : 0u) + (uint32_t)(m * g.chunks);
  g.arr = (rb ? P.arrive_b : 0u) + (uint32_t)m;
  const int kc = g.K / g.chunks;  // 1024 columns (gate/up 2048, QKV and O 512 where K allows), or all of K
  g.k0 = c * kc;
  g.nk = kc / BD_BK;
  return g;
}

// Attention split extent: keys [lo, hi) of the positions[b] + 1 visible keys.
struct BdAttn {
  int lo, hi;
  bool live;
};
// Splits a sequence of n keys uses: of at least BD_SPLIT_KEYS keys each, at
// most nsplit (the later ones of a short sequence stay empty): a count that
// depends only on the sequence's own length.
__device__ __forceinline__ int attn_splits(const BdParams& P, int n) {
  return min(P.nsplit, max(1, (n + BD_SPLIT_KEYS - 1) / BD_SPLIT_KEYS));
}
__device__ __forceinline__ BdAttn bd_attn(const BdParams& P, const BdSh& S, const Instr& in) {
  BdAttn e;
  const int b = (int)in.a0, s = (int)in.a2;
  e.live = b < P.B;
  e.lo = e.hi = 0;
  if (e.live) {
    const int n = S.pos[b] + 1;
    const int nsp = attn_splits(P, n);
    const int len = (n + nsp - 1) / nsp;
    e.lo = s * len < n ? s * len : n;
    e.hi = e.lo + len < n ? e.lo + len : n;
  }
  return e;
}
__device__ __forceinline__ int attn_blocks(const BdAttn& e) {
  return e.hi > e.lo ? (e.hi - e.lo + BD_KEYS - 1) / BD_KEYS : 0;
}
// Ring stages an instruction occupies (known to every role from the record).
__device__ __forceinline__ int bd_stages(const BdParams& P, const BdSh& S, const Instr& in) {
  if (is_gemm(in.op)) return bd_gemm(P, in).nk;
  if (in.op == BD_ATTN) return 2 * attn_blocks(bd_attn(P, S, in));
  return 0;
}

// First cache row of (layer l, K or V, cache slot, kv head g).
__device__ __forceinline__ size_t cache_row(const BdParams& P, int l, int kv, int slot, int g) {
  return ((((size_t)l * 2 + kv) * P.max_batch + slot) * P.nkv + g) * (size_t)P.max_ctx;
}

// ---------------------------------------------------------------- producer
__device__ void bd_producer(const BdParams& P, const BdSh& S) {
  if ((threadIdx.x & 31) != 0) return;
  const uint64_t pol_w = policy_evict_first();  // weights: streamed once
  const uint64_t pol_a = policy_evict_last();   // activations / KV: re-read by other tiles
  const uint32_t gen = S.flags[BF_GEN];
  uint32_t stage_ctr = 0, islot_ctr = 0;
  uint32_t npop = 0;
  // An instruction is popped only once a ring stage is free, i.e. when this
  // CTA can start streaming it: a CTA whose current tile waits on a
  // dependency does not also claim the next tile ahead of CTAs that are free.
  auto pop = [&]() -> uint32_t {
    const uint32_t k = npop++;
    if (P.mode == MODE_MEGA) {
      if (ld_volatile(&P.ctl[CTL_ABORT])) return BD_END;
      const uint32_t v = atomicAdd(&P.ctl[CTL_HEAD], 1u);
      return v < P.n_instr ? v : BD_END;
    }
    return k == 0 ? P.perop_base + blockIdx.x : BD_END;
  };
  // last counter (and target) seen satisfied: counters only grow within a
  // launch, so repeated waits on it need no new load
  uint32_t ok_bar = NO_BAR, ok_target = 0, ok_n = 0;
  for (;;) {
    const bool room = bd_wait(P, &S.empty[stage_ctr % BD_NSTAGE], ((stage_ctr / BD_NSTAGE) & 1u) ^ 1u);
    const uint32_t i = room ? pop() : BD_END;
    Instr in;
    if (i != BD_END) in = P.queue[i];
    const int si = islot_ctr % NISLOT;
    bool end = i == BD_END;
    if (!bd_wait(P, &S.iempty[si], ((islot_ctr / NISLOT) & 1u) ^ 1u)) end = true;
    if (!end) {
      *reinterpret_cast<Instr*>(S.islot + si * 48 + 16) = in;
      bd_mark(P, i, 4);
    }
    *reinterpret_cast<volatile uint32_t*>(S.islot + si * 48) = end ? BD_END : i;
    mbar_arrive(&S.ifull[si]);
    ++islot_ctr;
    if (end) break;

    if (is_gemm(in.op)) {
      const BdGemm g = bd_gemm(P, in);
      const int npre = g.nk < BD_PRE_STAGES ? g.nk : BD_PRE_STAGES;
      const uint32_t xb = (uint32_t)P.nb * BD_BK * 2;  // one activation plane box
      const uint32_t tx = BD_W_BYTES + 2 * xb;
      const uint32_t s0 = stage_ctr;
      auto load_w = [&](uint8_t* sp, int kb, uint64_t* bar) {
        const int x = g.k0 + kb * BD_BK;
        if (g.gu) {
          tma_load_2d(sp, tmap(P, g.a_map), x, g.a_row, bar, pol_w);
          tma_load_2d(sp + BD_W_BYTES / 2, tmap(P, g.a_map + 1), x, g.a_row, bar, pol_w);
        } else {
          tma_load_2d(sp, tmap(P, g.a_map), x, g.a_row, bar, pol_w);
        }
      };
      auto load_x = [&](uint8_t* sp, int kb, uint64_t* bar) {
        const int x = g.k0 + kb * BD_BK;
        tma_load_2d(sp + BD_W_BYTES, tmap(P, g.x_map), x, 0, bar, pol_a);
        tma_load_2d(sp + BD_W_BYTES + xb, tmap(P, g.x_map), x, P.nb, bar, pol_a);
      };
      // weights first: they depend on nothing
      for (int kb = 0; kb < npre; ++kb) {
        const int st = stage_ctr % BD_NSTAGE;
        bd_wait(P, &S.empty[st], ((stage_ctr / BD_NSTAGE) & 1u) ^ 1u);
        mbar_arrive_expect_tx(&S.full[st], tx);
        load_w(S.ring + st * BD_STAGE, kb, &S.full[st]);
        ++stage_ctr;
      }
      // (after a timeout the loads still run, on stale but valid memory, so
      // that every armed stage completes and the launch can drain)
      const uint32_t target = (gen + 1u) * in.wait_target;
      if (!(in.wait_bar == ok_bar && target == ok_target && in.wait_n == ok_n)) {
        if (bd_wait_deps(P, in, gen, i)) {
          ok_bar = in.wait_bar;
          ok_target = target;
          ok_n = in.wait_n;
        }
        fence_proxy_async_global();
      }
      bd_mark(P, i, 5);
      for (int kb = 0; kb < npre; ++kb) {
        const int st = (s0 + kb) % BD_NSTAGE;
        load_x(S.ring + st * BD_STAGE, kb, &S.full[st]);
      }
      for (int kb = npre; kb < g.nk; ++kb) {
        const int st = stage_ctr % BD_NSTAGE;
        bd_wait(P, &S.empty[st], ((stage_ctr / BD_NSTAGE) & 1u) ^ 1u);
        mbar_arrive_expect_tx(&S.full[st], tx);
        load_w(S.ring + st * BD_STAGE, kb, &S.full[st]);
        load_x(S.ring + st * BD_STAGE, kb, &S.full[st]);
        ++stage_ctr;
      }
      bd_mark(P, i, 6);
    } else if (in.op == BD_ATTN) {
      const BdAttn e = bd_attn(P, S, in);
      const int nblk = attn_blocks(e);
      if (nblk == 0) continue;
      bd_wait_deps(P, in, gen, i);
      fence_proxy_async_global();
      bd_mark(P, i, 5);
      const int l = in.layer, b = (int)in.a0, g = (int)in.a1;
      const int nbox = P.d / 64;
      for (int j = 0; j < nblk; ++j)
        for (int kv = 0; kv < 2; ++kv) {  // the block's K into one stage, its V into the next
          const int st = stage_ctr % BD_NSTAGE;
          bd_wait(P, &S.empty[st], ((stage_ctr / BD_NSTAGE) & 1u) ^ 1u);
          uint8_t* sp = S.ring + st * BD_STAGE;
          mbar_arrive_expect_tx(&S.full[st], (uint32_t)BD_KEYS * P.d * 2);
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(sp + bx * (BD_KEYS * 128), tmap(P, gmap(P, TMB_KV)), bx * 64,
                        (int)(cache_row(P, l, kv, S.slot[b], g) + e.lo + j * BD_KEYS), &S.full[st], pol_a);
          ++stage_ctr;
        }
      bd_mark(P, i, 6);
    }
  }
  // the copies this thread issued have landed before it leaves
  for (uint32_t k = 0; k < BD_NSTAGE && k < stage_ctr; ++k) {
    const uint32_t c = stage_ctr - 1 - k;
    bd_wait(P, &S.full[c % BD_NSTAGE], (c / BD_NSTAGE) & 1u);
  }
}

// ---------------------------------------------------------------- tensor-core issuer
__device__ void bd_mma(const BdParams& P, const BdSh& S, uint32_t tbase) {
  if ((threadIdx.x & 31) != 0) return;
  uint32_t islot_ctr = 0, stage_ctr = 0, use[2] = {0, 0};
  const uint32_t idesc = idesc_bf16_f32(BD_M, P.nb);
  const uint32_t xb = (uint32_t)P.nb * BD_BK * 2;
  for (;;) {
    const int si = islot_ctr % NISLOT;
    bd_wait(P, &S.ifull[si], (islot_ctr / NISLOT) & 1u);
    const uint32_t i = *reinterpret_cast<volatile uint32_t*>(S.islot + si * 48);
    Instr in;
    if (i != BD_END) in = *reinterpret_cast<const Instr*>(S.islot + si * 48 + 16);
    mbar_arrive(&S.iempty[si]);
    ++islot_ctr;
    if (i == BD_END) break;
    if (is_gemm(in.op)) {
      const BdGemm g = bd_gemm(P, in);
      const int ab = (int)((use[0] + use[1]) & 1u);
      bd_wait(P, &S.acce[ab], (use[ab] & 1u) ^ 1u);
      ++use[ab];
      tc_fence_after();
      const uint32_t d = tbase + (uint32_t)ab * BD_ACC_COLS;
      bd_mark(P, i, 7);
      for (int kb = 0; kb < g.nk; ++kb) {
        const int st = stage_ctr % BD_NSTAGE;
        bd_wait(P, &S.full[st], (stage_ctr / BD_NSTAGE) & 1u);
        ++stage_ctr;
        tc_fence_after();
        const uint32_t a0 = smem_u32(S.ring + st * BD_STAGE);
        const uint32_t bh = a0 + BD_W_BYTES, bl = bh + xb;
#pragma unroll
        for (int k = 0; k < BD_BK / 16; ++k) {
          const uint64_t ad = sdesc_sw128(a0 + 32 * k);
          tc_mma(d, ad, sdesc_sw128(bh + 32 * k), idesc, (kb | k) != 0);
          tc_mma(d, ad, sdesc_sw128(bl + 32 * k), idesc, true);
        }
        tc_commit(&S.empty[st]);
      }
      tc_commit(&S.accf[ab]);
      bd_mark(P, i, 8);
    } else if (in.op == BD_ATTN) {
      stage_ctr += (uint32_t)bd_stages(P, S, in);  // consumed by the compute warps
    }
  }
}

// ---------------------------------------------------------------- compute warps
__device__ __forceinline__ void cbar_bd() { named_bar(BD_CBAR, BD_NC); }

__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}
__device__ __forceinline__ float bfw(const uint16_t* p, int i) {
  return __uint_as_float((uint32_t)__ldg(p + i) << 16);
}

// Layer 0's input norm, sequences [BD_RG r, BD_RG r + BD_RG): the embedding
// row times the attention-norm gain into the hi/lo planes of hn, and the row's
// sum of squares into ss1 slot 0 (the QKV epilogue scales by 1 / rms).  One
// warp per sequence, 8 consecutive columns per lane and step.
__device__ void bd_norm(const BdParams& P, const BdSh& S, const Instr& in, int wc, int lane) {
  const int H = P.H;
  const uint16_t* gain = P.layers[0].attn_norm;
  const int b = (int)in.a0 * BD_RG + wc;
  if (wc >= BD_RG || b >= P.B) return;
  int tok = S.tok[b];
  if (tok < 0 || tok >= P.V) {
    if (lane == 0) bd_error(P, MK_ERR_BOUNDS, (uint32_t)b);
    tok = 0;
  }
  const uint16_t* emb = P.embed + (size_t)tok * H;
  float ss = 0.f;
  for (int c = lane * 8; c < H; c += 256) {
    float x[8], gw[8];
    widen8(__ldg(reinterpret_cast<const uint4*>(emb + c)), x);
    widen8(__ldg(reinterpret_cast<const uint4*>(gain + c)), gw);
    uint16_t hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ss = fmaf(x[e], x[e], ss);
      split_bf16(x[e] * gw[e], hi[e], lo[e]);
    }
    uint4 h, o;
    h.x = hi[0] | ((uint32_t)hi[1] << 16); h.y = hi[2] | ((uint32_t)hi[3] << 16);
    h.z = hi[4] | ((uint32_t)hi[5] << 16); h.w = hi[6] | ((uint32_t)hi[7] << 16);
    o.x = lo[0] | ((uint32_t)lo[1] << 16); o.y = lo[2] | ((uint32_t)lo[3] << 16);
    o.z = lo[4] | ((uint32_t)lo[5] << 16); o.w = lo[6] | ((uint32_t)lo[7] << 16);
    *reinterpret_cast<uint4*>(P.hn + (size_t)b * H + c) = h;
    *reinterpret_cast<uint4*>(P.hn + ((size_t)P.nb + b) * H + c) = o;
  }
  ss = warp_sum(ss);
  if (lane == 0) P.ss1[b] = ss;
}

// 1 / rms of every live sequence from the per-tile sums of squares (tile
// order), into S.rinv.  All compute threads call it (it ends with a barrier).
__device__ void bd_rms_inv(const BdParams& P, const BdSh& S, const float* ss, int nslots) {
  const int tc = threadIdx.x - 64;
  if (tc < P.B) {
    float t = 0.f;
    for (int k = 0; k < nslots; ++k) t += __ldcg(ss + (size_t)k * BD_NMAX + tc);
    S.rinv[tc] = 1.0f / sqrtf(t / (float)P.H + P.eps);
  }
  cbar_bd();
}

// The next norm's input for this thread's feature f of row tile m: x * gain
// into the hi/lo planes of hn, and the tile's sum of squares per sequence
// (rows in order) into ss[m].  All compute threads call it.
__device__ void bd_norm_out(const BdParams& P, const BdSh& S, int m, int row, int b0, const float (&x)[16],
                            const uint16_t* gain, float* ss) {
  const int tc = threadIdx.x - 64, H = P.H, f = m * BD_M + row;
  const float gw = bfw(gain, f);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int b = b0 + k;
    if (b < P.B) {
      uint16_t hi, lo;
      split_bf16(x[k] * gw, hi, lo);
      P.hn[(size_t)b * H + f] = hi;
      P.hn[((size_t)P.nb + b) * H + f] = lo;
    }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) S.scratch[row * BD_NMAX + b0 + k] = x[k] * x[k];
  cbar_bd();
  if (tc < P.B) {
    float t = 0.f;
    for (int r = 0; r < BD_M; ++r) t += S.scratch[r * BD_NMAX + tc];
    ss[(size_t)m * BD_NMAX + tc] = t;
  }
  cbar_bd();
}

// Epilogue of a finished GEMM row tile: y[k] is this thread's row (feature
// 128 m + row) for sequence b0 + k.
__device__ void bd_epilogue(const BdParams& P, const BdSh& S, const Instr& in, int row,
                            int b0, const float (&y)[16]) {
  const int l = in.layer, m = (int)in.a0, tc = threadIdx.x - 64;
  const int B = P.B, H = P.H, d = P.d, qd = P.nq * d, kd = P.nkv * d;
  switch (in.op) {
    case BD_O:
    case BD_DOWN: {
      const int f = m * BD_M + row;
      float* dst = in.op == BD_O ? P.xa : P.xb;
      const float* res = in.op == BD_O ? P.xb : P.xa;
      float x[16];
      // every residual input loaded before any is used (sequences past B
      // read sequence 0's word, dropped)
      float r[16];
      if (in.op == BD_O && l == 0) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int b = b0 + k;
          int tok = b < B ? S.tok[b] : 0;
          if (tok < 0 || tok >= P.V) tok = 0;  // reported by the layer-0 norm
          r[k] = bfw(P.embed + (size_t)tok * H, f);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) r[k] = __ldcg(res + (size_t)(b0 + k < B ? b0 + k : 0) * H + f);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int b = b0 + k;
        x[k] = b < B ? r[k] + y[k] : 0.f;
        if (b < B) dst[(size_t)b * H + f] = x[k];
      }
      // the next norm's input: the FFN norm after O, the next layer's
      // attention norm (or the final norm) after down
      const uint16_t* gain = in.op == BD_O ? P.layers[l].ffn_norm
                           : l + 1 < P.L  ? P.layers[l + 1].attn_norm
                                          : P.final_norm;
      bd_norm_out(P, S, m, row, b0, x, gain, in.op == BD_O ? P.ss2 : P.ss1);
      break;
    }
    case BD_LM: {
      bd_rms_inv(P, S, P.ss1, (int)P.n_down_m);
      const int f = m * BD_M + row;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (f < P.V && b0 + k < B) P.logits[(size_t)(b0 + k) * P.V + f] = y[k] * S.rinv[b0 + k];
      break;
    }
    case BD_GU: {
      // rows 0..63 gate, 64..127 up (features 64 m + j), both scaled by the
      // FFN norm's 1 / rms
      bd_rms_inv(P, S, P.ss2, (int)P.n_o_m);
#pragma unroll
      for (int k = 0; k < 16; ++k)
        S.scratch[row * BD_NMAX + b0 + k] = b0 + k < B ? y[k] * S.rinv[b0 + k] : 0.f;
      cbar_bd();
      const int j = tc & 63;
      for (int b = tc >> 6; b < B; b += BD_NC / 64) {
        const float gt = S.scratch[j * BD_NMAX + b], up = S.scratch[(64 + j) * BD_NMAX + b];
        uint16_t hi, lo;
        split_bf16(gt / (1.0f + expf(-gt)) * up, hi, lo);
        const size_t o = (size_t)b * P.F + (size_t)m * (BD_M / 2) + j;
        P.act[o] = hi;
        P.act[o + (size_t)P.nb * P.F] = lo;
      }
      break;
    }
    default: {  // BD_QKV
      // the attention norm's 1 / rms (layer 0: one full-row sum per sequence)
      bd_rms_inv(P, S, P.ss1, l == 0 ? 1 : (int)P.n_down_m);
      const int f0 = m * BD_M;
      if (f0 >= qd + kd) {  // values: straight into the cache
        const int f = f0 + row - qd - kd, g = f / d, dim = f % d;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int b = b0 + k;
          if (b < B)
            P.kv[(cache_row(P, l, 1, S.slot[b], g) + S.pos[b]) * d + dim] =
                __bfloat16_as_ushort(__float2bfloat16_rn(y[k] * S.rinv[b]));
        }
        break;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k)
        S.scratch[row * BD_NMAX + b0 + k] = b0 + k < B ? y[k] * S.rinv[b0 + k] : 0.f;
      cbar_bd();
      const bool is_q = f0 < qd;
      const int hpt = BD_M / d;  // heads in this tile
      float* inv = S.hs + 16;    // [b][hpt] (<= 64)
      if (P.qk_norm) {
        for (int t = tc; t < B * hpt; t += BD_NC) {
          const int b = t / hpt, hh = t % hpt;
          float ss = 0.f;
          for (int i = 0; i < d; ++i) {
            const float v = S.scratch[(hh * d + i) * BD_NMAX + b];
            ss = fmaf(v, v, ss);
          }
          inv[t] = 1.0f / sqrtf(ss / (float)d + P.eps);
        }
        cbar_bd();
      }
      const uint16_t* gn = P.qk_norm ? (is_q ? P.layers[l].q_norm : P.layers[l].k_norm) : nullptr;
      const int half = d / 2;
      // pair i of head hh for sequence b: thread tc takes pair index tc % 64
      const int pi = tc & 63, hh = pi / half, i = pi % half;
      for (int b = tc >> 6; b < B; b += BD_NC / 64) {
        float u1 = S.scratch[(hh * d + i) * BD_NMAX + b];
        float u2 = S.scratch[(hh * d + i + half) * BD_NMAX + b];
        if (gn) {
          const float iv = inv[b * hpt + hh];
          u1 = u1 * iv * bfw(gn, i);
          u2 = u2 * iv * bfw(gn, i + half);
        }
        const float2 cs = __ldg(P.rope + (size_t)S.pos[b] * half + i);
        const float r1 = u1 * cs.x - u2 * cs.y, r2 = u2 * cs.x + u1 * cs.y;
        const int f = f0 + hh * d;  // first feature of the head
        if (is_q) {
          P.q[(size_t)b * qd + f + i] = r1;
          P.q[(size_t)b * qd + f + i + half] = r2;
        } else {
          const int g = (f - qd) / d;
          uint16_t* kr = P.kv + (cache_row(P, l, 0, S.slot[b], g) + S.pos[b]) * d;
          kr[i] = __bfloat16_as_ushort(__float2bfloat16_rn(r1));
          kr[i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
        }
      }
      break;
    }
  }
}

// One attention split of (sequence b, kv head g): online softmax over its key
// blocks (K and V tiles in the ring, 128-byte swizzled rows), then the split's
// (max, sum, unnormalised output) to global memory.  Returns the ring counter.
//  scores  8 lanes per key (lane `sub` holds 8-column groups sub, sub + 8),
//          q in registers, a three-level shuffle per head; warp w takes keys
//          [8 w, 8 w + 8) of the block.
//  P V     warp w the same 8 keys for every head, lane the columns
//          [DPL lane, DPL lane + DPL): each V element is widened once for all
//          heads; the eight warps' partial outputs are added once per split.
template <int D>
__device__ uint32_t bd_attn_split(const BdParams& P, const BdSh& S, const Instr& in, const BdAttn& e,
                                  uint32_t stage_ctr, uint32_t idx) {
  const int tc = threadIdx.x - 64, lane = tc & 31, wc = tc >> 5;
  // Two groups of four warps take the key blocks in turn (group 0 the even
  // blocks, group 1 the odd ones), each with its own online-softmax state, so
  // that one group's score / softmax / P V round trips overlap the other's;
  // the two states are merged at the end in group order.
  const int grp = wc >> 2, wg = wc & 3, tg = tc & 127;
  const int b = (int)in.a0, g = (int)in.a1, s = (int)in.a2, rep = P.rep;
  const int qd = P.nq * D;
  constexpr int DPL = D / 32;  // output columns per lane in P V
  constexpr int KPW = BD_KEYS / 4;  // keys per warp of a group (scores and P V)
  const float scale = 1.0f / sqrtf((float)D);
  float* sc = S.sc + grp * 4 * BD_KEYS;  // this group's [rep][BD_KEYS]
  float* hs = S.hs + grp * 16;           // this group's [rep] x {m, l, alpha}
  auto gbar = [&]() { named_bar(BD_GBAR0 + grp, BD_NC / 2); };
  // Scores on the tensor cores, 8 keys per m16n8k16 product: A rows r < rep
  // hold q of head r rounded to bf16, rows rep .. 2 rep - 1 the bf16 of its
  // remainder (hi + lo keeps q's float32 precision against the exact bf16
  // keys), the other rows zero.  The reduction index is permuted so that lane
  // t's four values of k-step 2 s + u are dimensions 32 s + 8 t + 4 u .. + 3:
  // one 16-byte load per key row gives two k-steps of B.
  constexpr int KSTEPS = D / 16;
  const int gq = lane >> 2, tq = lane & 3;
  const int hq = gq < rep ? gq : gq - rep;
  uint32_t af[KSTEPS][2];
#pragma unroll
  for (int ks = 0; ks < KSTEPS; ++ks) {
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gq < 2 * rep)
      u = __ldcg(reinterpret_cast<const float4*>(P.q + (size_t)b * qd + (size_t)(g * rep + hq) * D +
                                                 32 * (ks >> 1) + 8 * tq + 4 * (ks & 1)));
    const float f[4] = {u.x, u.y, u.z, u.w};
    uint32_t hv[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(f[x]);
      const __nv_bfloat16 v = gq < rep ? hi : __float2bfloat16_rn(f[x] - __bfloat162float(hi));
      hv[x] = (uint32_t)__bfloat16_as_ushort(v);
    }
    af[ks][0] = hv[0] | (hv[1] << 16);
    af[ks][1] = hv[2] | (hv[3] << 16);
  }
  if (tg < rep) {
    hs[tg * 3 + 0] = -INFINITY;
    hs[tg * 3 + 1] = 0.f;
    hs[tg * 3 + 2] = 0.f;
  }
  float acc[4][DPL];
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[h][k] = 0.f;
  cbar_bd();
  const int nblk = attn_blocks(e);
  for (int j = grp; j < nblk; j += 2) {
    const uint32_t cj = stage_ctr + 2u * (uint32_t)j;  // this block's K stage; V in the next
    const int st = cj % BD_NSTAGE;
    const int st_v = (cj + 1) % BD_NSTAGE;
    bd_wait(P, &S.full[st], (cj / BD_NSTAGE) & 1u);
    if (j == 0 && tc == 0) bd_mark(P, idx, 9);
    const uint8_t* kt = S.ring + st * BD_STAGE;
    const uint8_t* vt = S.ring + st_v * BD_STAGE;
    const int base = e.lo + j * BD_KEYS;
#pragma unroll 2
    for (int nn = 0; nn < KPW / 8; ++nn) {
      // keys KPW wg + 8 nn .. + 7: row gq of this product; the K block is
      // [D / 64 halves][BD_KEYS][64] with 16-byte chunk c of key k at c ^ (k & 7)
      const int kr = wg * KPW + nn * 8 + gq;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s2 = 0; s2 < KSTEPS / 2; ++s2) {
        const int chunk = 4 * (s2 & 1) + tq;
        const uint4 kk = *reinterpret_cast<const uint4*>(kt + (s2 >> 1) * (BD_KEYS * 128) + kr * 128 +
                                                         ((chunk ^ (kr & 7)) << 4));
        mma_bf16_16816(c, af[2 * s2][0], 0u, af[2 * s2][1], 0u, kk.x, kk.y);
        mma_bf16_16816(c, af[2 * s2 + 1][0], 0u, af[2 * s2 + 1][1], 0u, kk.z, kk.w);
      }
      // row gq (hi) + row gq + rep (lo): lanes 4 rep apart
      const float s0 = c[0] + __shfl_xor_sync(0xffffffffu, c[0], 4 * rep);
      const float s1 = c[1] + __shfl_xor_sync(0xffffffffu, c[1], 4 * rep);
      const int k = wg * KPW + nn * 8 + 2 * tq;
      if (gq < rep) {
        sc[gq * BD_KEYS + k] = base + k < e.hi ? s0 * scale : -INFINITY;
        sc[gq * BD_KEYS + k + 1] = base + k + 1 < e.hi ? s1 * scale : -INFINITY;
      }
    }
    gbar();
    // online softmax: warp h of the group owns head h
    if (wg < rep) {
      float sv[BD_KEYS / 32];
#pragma unroll
      for (int u = 0; u < BD_KEYS / 32; ++u) sv[u] = sc[wg * BD_KEYS + lane + 32 * u];
      float mx = sv[0];
#pragma unroll
      for (int u = 1; u < BD_KEYS / 32; ++u) mx = fmaxf(mx, sv[u]);
      mx = warp_max(mx);
      const float m_old = hs[wg * 3 + 0];
      const float m_new = fmaxf(m_old, mx);
      const float alpha = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
      float psum = 0.f;
#pragma unroll
      for (int u = 0; u < BD_KEYS / 32; ++u) {
        const float pv = sv[u] == -INFINITY ? 0.f : expf(sv[u] - m_new);
        sc[wg * BD_KEYS + lane + 32 * u] = pv;
        psum += pv;
      }
      const float ps = warp_sum(psum);
      __syncwarp();
      if (lane == 0) {
        hs[wg * 3 + 0] = m_new;
        hs[wg * 3 + 1] = hs[wg * 3 + 1] * alpha + ps;
        hs[wg * 3 + 2] = alpha;
      }
    }
    gbar();
    // P V over this warp's KPW keys (keys past the split are skipped, not
    // weighted by zero: the cache rows there may hold anything)
    {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float alpha = h < rep ? hs[h * 3 + 2] : 0.f;
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[h][k] *= alpha;
      }
      const int col = lane * DPL, bx = col >> 6, cin = col & 63;
      const int k0 = wg * KPW;
      const int k1 = e.hi - base < k0 + KPW ? e.hi - base : k0 + KPW;
      // the block's values are in the next stage
      bd_wait(P, &S.full[st_v], ((cj + 1) / BD_NSTAGE) & 1u);
#pragma unroll 4
      for (int k = k0; k < k1; ++k) {
        const uint8_t* vr = vt + bx * (BD_KEYS * 128) + k * 128 + ((((cin >> 3) ^ (k & 7))) << 4) + (cin & 7) * 2;
        float vx[DPL];
        if constexpr (DPL == 4) {
          const uint2 u = *reinterpret_cast<const uint2*>(vr);
          vx[0] = bf_lo(u.x); vx[1] = bf_hi(u.x); vx[2] = bf_lo(u.y); vx[3] = bf_hi(u.y);
        } else {
          const uint32_t u = *reinterpret_cast<const uint32_t*>(vr);
          vx[0] = bf_lo(u); vx[1] = bf_hi(u);
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          if (h < rep) {
            const float p = sc[h * BD_KEYS + k];
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[h][t] = fmaf(p, vx[t], acc[h][t]);
          }
        }
      }
    }
    gbar();  // the group is done with its stages and its probabilities
    if (tg == 0) {
      mbar_arrive(&S.empty[st]);
      mbar_arrive(&S.empty[st_v]);
    }
  }
  stage_ctr += 2u * (uint32_t)nblk;
  if (tc == 0) bd_mark(P, idx, 10);
  cbar_bd();
  // merge: each group's output scaled to the split's maximum, then the eight
  // warps' partial outputs added in warp order; the split's partial is
  // o (unnormalised), max, sum per head
  float* red = S.scratch;  // [8 warps][4 heads][D]
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float f = 0.f;
    if (h < rep) {
      const float m0 = S.hs[h * 3 + 0], m1 = S.hs[16 + h * 3 + 0];
      const float M = fmaxf(m0, m1);
      const float mg = grp == 0 ? m0 : m1;
      f = mg == -INFINITY ? 0.f : expf(mg - M);
    }
#pragma unroll
    for (int k = 0; k < DPL; ++k) red[(wc * 4 + h) * D + lane * DPL + k] = acc[h][k] * f;
  }
  cbar_bd();
  float* part = P.apart + (((size_t)b * P.nkv + g) * P.nsplit + s) * rep * (D + 2);
  for (int t = tc; t < rep * D; t += BD_NC) {
    const int h = t / D, c = t % D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) o += red[(w * 4 + h) * D + c];
    part[h * (D + 2) + c] = o;
  }
  if (tc < rep) {
    const float m0 = S.hs[tc * 3 + 0], m1 = S.hs[16 + tc * 3 + 0];
    const float l0 = S.hs[tc * 3 + 1], l1 = S.hs[16 + tc * 3 + 1];
    const float M = fmaxf(m0, m1);
    const float f0 = m0 == -INFINITY ? 0.f : expf(m0 - M);
    const float f1 = m1 == -INFINITY ? 0.f : expf(m1 - M);
    part[tc * (D + 2) + D] = M;
    part[tc * (D + 2) + D + 1] = l0 * f0 + l1 * f1;
  }
  return stage_ctr;
}

// Combine the splits of (b, g) in split order into the hi/lo planes of ao.
template <int D>
__device__ void bd_attn_combine(const BdParams& P, int b, int g, int nsp) {
  const int tc = threadIdx.x - 64, rep = P.rep, qd = P.nq * D;
  const float* gp = P.apart + ((size_t)b * P.nkv + g) * P.nsplit * rep * (D + 2);
  for (int t = tc; t < rep * D; t += BD_NC) {
    const int h = t / D, c = t % D;
    // the first W splits' (max, sum, o) words loaded together before any is
    // used (split indices clamped to a valid split, whose values are
    // dropped): one round trip instead of one per split; splits from W on
    // follow in a loop
    constexpr int W = 4;
    float mv[W], lv[W], ov[W];
#pragma unroll
    for (int s = 0; s < W; ++s) {
      const int sc = s < nsp ? s : nsp - 1;
      const float* ps = gp + ((size_t)sc * rep + h) * (D + 2);
      mv[s] = __ldcg(ps + D);
      lv[s] = __ldcg(ps + D + 1);
      ov[s] = __ldcg(ps + c);
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < W; ++s)
      if (s < nsp) M = fmaxf(M, mv[s]);
    for (int s = W; s < nsp; ++s) M = fmaxf(M, __ldcg(gp + ((size_t)s * rep + h) * (D + 2) + D));
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int s = 0; s < W; ++s) {
      if (s < nsp) {
        const float f = mv[s] == -INFINITY ? 0.f : expf(mv[s] - M);
        Lsum = fmaf(lv[s], f, Lsum);
        O = fmaf(ov[s], f, O);
      }
    }
    for (int s = W; s < nsp; ++s) {
      const float* ps = gp + ((size_t)s * rep + h) * (D + 2);
      const float ms = __ldcg(ps + D);
      const float f = ms == -INFINITY ? 0.f : expf(ms - M);
      Lsum = fmaf(__ldcg(ps + D + 1), f, Lsum);
      O = fmaf(__ldcg(ps + c), f, O);
    }
    uint16_t hi, lo;
    split_bf16(O / Lsum, hi, lo);
    const size_t o = (size_t)b * qd + (size_t)(g * rep + h) * D + c;
    P.ao[o] = hi;
    P.ao[o + (size_t)P.nb * qd] = lo;
  }
}

__device__ void bd_compute(const BdParams& P, const BdSh& S, uint32_t tbase) {
  const int wc = (threadIdx.x >> 5) - 2;  // compute warp 0..7
  const int lane = threadIdx.x & 31;
  const int tc = threadIdx.x - 64;
  const int q = (threadIdx.x >> 5) & 3;   // TMEM lane quarter this warp may access
  const int row = 32 * q + lane;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const uint32_t gen = S.flags[BF_GEN];
  uint32_t islot_ctr = 0, use[2] = {0, 0}, stage_ctr = 0;
  for (;;) {
    const int si = islot_ctr % NISLOT;
    if (tc == 0) {
      uint32_t v = BD_END;
      if (bd_wait(P, &S.ifull[si], (islot_ctr / NISLOT) & 1u))
        v = *reinterpret_cast<volatile uint32_t*>(S.islot + si * 48);
      S.flags[BF_SLOT] = v;
    }
    cbar_bd();
    const uint32_t i = S.flags[BF_SLOT];
    Instr in;
    if (i != BD_END) in = *reinterpret_cast<const Instr*>(S.islot + si * 48 + 16);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.iempty[si]);
    ++islot_ctr;
    if (i == BD_END) break;
    if (tc == 0) {
      bd_mark(P, i, 1);
      if (P.trace)
        P.trace[(size_t)i * TRACE_WORDS] =
            (unsigned long long)smid() | ((unsigned long long)(in.op | (in.layer << 8)) << 32);
    }
    bool release = true;
    if (is_gemm(in.op)) {
      const BdGemm gm = bd_gemm(P, in);
      const int ab = (int)((use[0] + use[1]) & 1u);
      bd_wait(P, &S.accf[ab], use[ab] & 1u);
      ++use[ab];
      stage_ctr += (uint32_t)gm.nk;
      tc_fence_after();
      if (tc == 0) bd_mark(P, i, 2);
      // batch columns [b0, b0 + 16) of this thread's row (feature)
      const int b0 = 16 * (wc >> 2);
      float y[16];
      tmem_ld16(tbase + (uint32_t)ab * BD_ACC_COLS + lane_base + (uint32_t)b0, y);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acce[ab]);
      if (gm.chunks > 1) {
        // split-K: publish this chunk's partial; the last chunk to arrive adds
        // all chunks in chunk order and runs the epilogue
        float* mine = P.part + ((size_t)gm.pslot + in.a1) * BD_NMAX * BD_M;
#pragma unroll
        for (int k = 0; k < 16; ++k) mine[(b0 + k) * BD_M + row] = y[k];
        cbar_bd();
        if (tc == 0) {
          uint32_t* arr = P.arrive + gm.arr;
          const uint32_t old = atom_add_acq_rel_gpu(arr, 1u);
          const bool last = old == (uint32_t)(gm.chunks - 1);
          if (last) *arr = 0u;
          S.flags[BF_LAST] = last ? 1u : 0u;
        }
        cbar_bd();
        release = S.flags[BF_LAST] != 0u;
        if (release) {
          const float* base = P.part + (size_t)gm.pslot * BD_NMAX * BD_M;
#pragma unroll
          for (int k = 0; k < 16; ++k) y[k] = 0.f;
          // the chunks' partials CG chunks at a time, every load of a group
          // issued before any is added (chunk indices past the last clamped
          // to it, their values dropped): one round trip per group instead
          // of one per chunk; the adds stay in chunk order
          constexpr int CG = 4;
          for (int c0 = 0; c0 < gm.chunks; c0 += CG) {
            float v[CG][16];
#pragma unroll
            for (int u = 0; u < CG; ++u) {
              const int c = c0 + u < gm.chunks ? c0 + u : gm.chunks - 1;
#pragma unroll
              for (int k = 0; k < 16; ++k) v[u][k] = __ldcg(base + ((size_t)c * BD_NMAX + b0 + k) * BD_M + row);
            }
#pragma unroll
            for (int u = 0; u < CG; ++u)
              if (c0 + u < gm.chunks)
#pragma unroll
                for (int k = 0; k < 16; ++k) y[k] += v[u][k];
          }
        }
      }
      if (release) bd_epilogue(P, S, in, row, b0, y);
    } else if (in.op == BD_ATTN) {
      const BdAttn e = bd_attn(P, S, in);
      if (!e.live) {
        release = in.a2 == 0;  // one release per dead (b, g) group
      } else {
        // Splits s >= nsp (past the keys of a sequence whose length uses
        // fewer splits) hold nothing and do nothing: no wait, no arrival.
        // The arrival counter of (b, g) is shared by the layers, so only the
        // splits that waited for this layer's queries may count on it (their
        // wait orders them after the previous layer's combine).
        const int nsp = attn_splits(P, S.pos[in.a0] + 1);
        release = false;
        if ((int)in.a2 < nsp) {
          if (tc == 0) {
            S.flags[BF_ABORT] = bd_wait_deps(P, in, gen, i) ? 0u : 1u;
            bd_mark(P, i, 2);
          }
          cbar_bd();
          if (P.d == 128) stage_ctr = bd_attn_split<128>(P, S, in, e, stage_ctr, i);
          else stage_ctr = bd_attn_split<64>(P, S, in, e, stage_ctr, i);
          cbar_bd();
          if (tc == 0) {
            uint32_t* arr = P.arrive + P.n_arrive_gemm + (size_t)in.a0 * P.nkv + in.a1;
            const uint32_t old = atom_add_acq_rel_gpu(arr, 1u);
            const bool last = old == (uint32_t)(nsp - 1);
            if (last) *arr = 0u;
            S.flags[BF_LAST] = last ? 1u : 0u;
          }
          cbar_bd();
          release = S.flags[BF_LAST] != 0u;
          if (release) {
            if (P.d == 128) bd_attn_combine<128>(P, (int)in.a0, (int)in.a1, nsp);
            else bd_attn_combine<64>(P, (int)in.a0, (int)in.a1, nsp);
          }
        }
      }
    } else if (is_norm(in.op)) {
      if (tc == 0) {
        S.flags[BF_ABORT] = bd_wait_deps(P, in, gen, i) ? 0u : 1u;
        bd_mark(P, i, 2);
      }
      cbar_bd();
      if (!S.flags[BF_ABORT]) bd_norm(P, S, in, wc, lane);
    }
    fence_proxy_async_global();  // outputs are read by other CTAs' TMA loads
    cbar_bd();
    if (tc == 0 && release && P.mode == MODE_MEGA && in.rel_bar != NO_BAR)
      red_release_gpu_add(&P.bars[in.rel_bar], 1u);
    if (tc == 0) bd_mark(P, i, 3);
  }
}

__global__ void __launch_bounds__(BD_THREADS, 1) mk_bdecode_kernel(const __grid_constant__ BdParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const BdSh S = bd_map(smem);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < BD_NSTAGE; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < NISLOT; ++s) {
      mbar_init(&S.ifull[s], 1);
      mbar_init(&S.iempty[s], 9);  // issuer + 8 compute warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.accf[b], 1);
      mbar_init(&S.acce[b], 8);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    S.flags[BF_GEN] = P.mode == MODE_MEGA ? ld_volatile(&P.ctl[CTL_GEN]) : 0u;
  }
  if (threadIdx.x < BD_NMAX) {
    const bool live = (int)threadIdx.x < P.B;
    int pos = live ? P.positions[threadIdx.x] : 0;
    if (pos < 0 || pos >= P.max_ctx) {
      // the new key would land outside its cache slot: report it and run the
      // sequence at position 0 (in bounds; its result is not meaningful)
      if (blockIdx.x == 0) bd_error(P, MK_ERR_BOUNDS, threadIdx.x);
      pos = 0;
    }
    // the column's cache slot: its own index, or the caller's map (several
    // columns of one slot at consecutive positions: a prompt chunk)
    int slot = !live ? 0 : P.slots ? P.slots[threadIdx.x] : (int)threadIdx.x;
    if (slot < 0 || slot >= P.max_batch) {
      if (blockIdx.x == 0) bd_error(P, MK_ERR_BOUNDS, threadIdx.x);
      slot = 0;
    }
    S.pos[threadIdx.x] = pos;
    S.tok[threadIdx.x] = live ? P.tokens[threadIdx.x] : 0;
    S.slot[threadIdx.x] = slot;
  }
  if (warp == 1) tmem_alloc(reinterpret_cast<uint32_t*>(const_cast<uint32_t*>(&S.flags[BF_TMEM])), 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.flags[BF_TMEM];
  if (warp == 0) bd_producer(P, S);
  else if (warp == 1) bd_mma(P, S, tbase);
  else bd_compute(P, S, tbase);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 64);
  }
  if (threadIdx.x == 0 && P.mode == MODE_MEGA) {
    __threadfence();
    const uint32_t old = atomicAdd(&P.ctl[CTL_EXIT], 1u);
    if (old == gridDim.x - 1) {
      P.ctl[CTL_HEAD] = 0u;
      P.ctl[CTL_EXIT] = 0u;
      P.ctl[CTL_GEN] = S.flags[BF_GEN] + 1u;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t bd_setup() {
  return cudaFuncSetAttribute(mk_bdecode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              BdSmem::total);
}
cudaError_t bd_launch_mega(const BdParams& p, int ctas, cudaStream_t st) {
  BdParams pp = p;
  void* args[] = {(void*)&pp};
  return cudaLaunchCooperativeKernel((const void*)mk_bdecode_kernel, dim3(ctas), dim3(BD_THREADS), args,
                                     (size_t)BdSmem::total, st);
}
cudaError_t bd_launch_perop(const BdParams& p, uint32_t first, uint32_t count, cudaStream_t st) {
  BdParams pp = p;
  pp.mode = MODE_PEROP;
  pp.perop_base = first;
  mk_bdecode_kernel<<<count, BD_THREADS, BdSmem::total, st>>>(pp);
  return cudaGetLastError();
}

}  // namespace mk
