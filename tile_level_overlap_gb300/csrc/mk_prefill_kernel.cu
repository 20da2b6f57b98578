// Prefill interpreter (sm_103a): tensor-core tiles with tile-level
// dependencies, one persistent CTA per SM.
//
//  warp 0      producer: pops instructions (one atomic each), streams weight
//              k-blocks ahead of the instruction's dependencies and activation
//              k-blocks once they are satisfied (acquire + async-proxy fence),
//              all with 2D TMA loads into a 3 x 64 KB ring.
//  warp 1      tensor-core issuer: owns 512 TMEM columns (two 128 x 256 f32
//              accumulators), issues tcgen05.mma and commits to mbarriers.
//  warps 2-5   compute: GEMM epilogues (RoPE + K/V cache write, residual adds,
//              SwiGLU), RMSNorm blocks, and the softmax half of causal
//              attention (S = Q K^T and O = P V run on the tensor cores, Q and
//              P are written into TMEM as the A operand).
//
// Precision: every activation operand of a tensor-core product is split into
// two bf16 values, hi = bf16(x) and lo = bf16(x - hi), and multiplied as two
// MMAs into the same float32 accumulator.  The weights are bf16 already and
// the keys and values are the bf16 cache entries, so every product carries
// float32-level precision; one bf16 rounding per operand would not (its error
// grows to a few percent of the logits' RMS after two layers).
//
// "MegaOps" (Abstract): a consumer waits only on the tiles it reads (here:
// attention of block m on the QKV tiles of blocks <= m, the next layer's norm
// of block m on the down tiles of block m) and weights are prefetched while
// the preceding operator is still running.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mk.h"
#include "mk_device.cuh"
#include "mk_internal.h"
#include "mk_plan.h"
#include "mk_prefill.h"
#include "mk_tc.cuh"

namespace mk {
namespace {

// GEMM stage: A hi 16 KB | A lo 16 KB | B 32 KB.  Attention stage: K_j | V_j.
constexpr int PF_STAGE = 64 * 1024;
constexpr int PF_NSTAGE = 3;
constexpr uint32_t PF_A_BYTES = PF_BM * PF_BK * 2;
constexpr int PF_THREADS = 192;
constexpr int PF_CBAR = 2;             // named barrier of the compute warps
constexpr int PF_NC = 128;             // compute threads
constexpr uint32_t PF_END = 0xffffffffu;

struct PfSmem {
  static constexpr int ring = 0;
  static constexpr int bars = ring + PF_NSTAGE * PF_STAGE;
  // full[3] empty[3] ifull[8] iempty[8] accf[2] acce[2] qfull sfull pfull ofull
  static constexpr int n_mbar = 2 * PF_NSTAGE + 2 * NISLOT + 4 + 4;
  static constexpr int islot = bars + n_mbar * 8;
  static constexpr int flags = islot + NISLOT * 48;          // [16] u32
  static constexpr int scratch = flags + 16 * 4;             // [128] f32
  static constexpr int total = scratch + 128 * 4;
};
static_assert(PfSmem::total <= 227 * 1024, "prefill shared memory budget");

enum PfFlag { PFF_GEN = 0, PFF_SLOT = 1, PFF_ABORT = 2, PFF_TMEM = 3 };

struct PfSh {
  uint8_t* ring;
  uint64_t *full, *empty, *ifull, *iempty, *accf, *acce, *qfull, *sfull, *pfull, *ofull;
  uint8_t* islot;
  volatile uint32_t* flags;
  float* scratch;
};

__device__ __forceinline__ PfSh pf_map(uint8_t* base) {
  PfSh s;
  s.ring = base + PfSmem::ring;
  uint64_t* b = reinterpret_cast<uint64_t*>(base + PfSmem::bars);
  s.full = b;
  s.empty = b + PF_NSTAGE;
  s.ifull = b + 2 * PF_NSTAGE;
  s.iempty = s.ifull + NISLOT;
  s.accf = s.iempty + NISLOT;
  s.acce = s.accf + 2;
  s.qfull = s.acce + 2;
  s.sfull = s.qfull + 1;
  s.pfull = s.sfull + 1;
  s.ofull = s.pfull + 1;
  s.islot = base + PfSmem::islot;
  s.flags = reinterpret_cast<volatile uint32_t*>(base + PfSmem::flags);
  s.scratch = reinterpret_cast<float*>(base + PfSmem::scratch);
  return s;
}

__device__ void pf_error(const PfParams& P, uint32_t code, uint32_t detail) {
  if (atomicCAS(&P.ctl[CTL_STATUS], 0u, code) == 0u) atomicExch(&P.ctl[CTL_DETAIL], detail);
  atomicExch(&P.ctl[CTL_ABORT], 1u);
}

// Bounded mbarrier wait.  After an abort (another wait already gave up) it
// gives up within ~10 us, so a broken launch drains quickly.
__device__ __forceinline__ bool pf_wait(const PfParams& P, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t dt = globaltimer() - t0;
    if (dt > P.wait_limit_ns * 4ull) {
      pf_error(P, MK_ERR_TIMEOUT, 0xfffffff1u);
      return false;
    }
    if ((it & 255u) == 0 && dt > 10000ull && ld_volatile(&P.ctl[CTL_ABORT]) != 0u) return false;
  }
}

__device__ __forceinline__ const CUtensorMap* tmap(const PfParams& P, int idx) {
  return reinterpret_cast<const CUtensorMap*>(P.tm) + idx;
}
__device__ __forceinline__ int am(const PfParams& P, int which) { return P.L * TM_PER_LAYER + which; }

__device__ __forceinline__ bool pf_live(const PfParams& P, const Instr& in) {
  return x_eval(P.xw + PXS_BLOCK_LIVE * X_MAX_WORDS, in, 1, P.S, nullptr, 0) > 0;
}

// Bounded acquire-spin on every barrier an instruction waits on.  Returns
// false (abort) on timeout or when another CTA aborted.
__device__ bool pf_wait_deps(const PfParams& P, const Instr& in, uint32_t gen, uint32_t idx) {
  if (P.mode != MODE_MEGA || in.wait_bar == NO_BAR) return true;
  const uint32_t target = (in.flags & IF_ABS_TARGET) ? in.wait_target : (gen + 1u) * in.wait_target;
  const uint64_t t0 = globaltimer();
  for (uint32_t k = 0; k < in.wait_n;) {
    const uint32_t* c = &P.bars[in.wait_bar + k * in.wait_stride];
    if ((int32_t)(ld_acquire_gpu(c) - target) >= 0) {
      ++k;
      continue;
    }
    if (ld_volatile(&P.ctl[CTL_ABORT]) != 0u) return false;
    if (globaltimer() - t0 > P.wait_limit_ns) {
      pf_error(P, MK_ERR_TIMEOUT, idx);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

__device__ __forceinline__ bool is_gemm(uint8_t op) {
  return op == PF_QKV || op == PF_O || op == PF_GU || op == PF_DOWN || op == PF_LM;
}

// GEMM geometry of an instruction.
struct PfGemm {
  int K;          // reduction length
  int a_map;      // activation tensor map
  int bn;         // tcgen05 N (output columns of the tile)
  int b_map0, b_row0, b_rows0;  // first weight box: map, first row, rows
  int b_map1, b_row1;           // second weight box (gate/up), rows = b_rows0
};

__device__ __forceinline__ PfGemm pf_gemm(const PfParams& P, const Instr& in) {
  PfGemm g;
  const int l = in.layer, n = (int)in.a1;
  const int qd = P.nq * P.d, kd = P.nkv * P.d;
  g.b_map1 = -1;
  g.b_row1 = 0;
  switch (in.op) {
    case PF_QKV: {
      g.K = P.H;
      g.a_map = am(P, AM_HN1);
      g.bn = P.bn_qkv;
      const int r = n * P.bn_qkv;
      g.b_rows0 = P.bn_qkv;
      if (r < qd) {
        g.b_map0 = l * TM_PER_LAYER + TM_WQ;
        g.b_row0 = r;
      } else if (r < qd + kd) {
        g.b_map0 = l * TM_PER_LAYER + TM_WK;
        g.b_row0 = r - qd;
      } else {
        g.b_map0 = l * TM_PER_LAYER + TM_WV;
        g.b_row0 = r - qd - kd;
      }
      break;
    }
    case PF_LM:
      g.K = P.H;
      g.a_map = am(P, AM_HN1);
      g.bn = PF_BN;
      g.b_map0 = am(P, AM_LMW);
      g.b_row0 = n * PF_BN;
      g.b_rows0 = PF_BN;
      break;
    case PF_O:
      g.K = qd;
      g.a_map = am(P, AM_AO);
      g.bn = PF_BN;
      g.b_map0 = l * TM_PER_LAYER + TM_WO;
      g.b_row0 = n * PF_BN;
      g.b_rows0 = PF_BN;
      break;
    case PF_GU:
      g.K = P.H;
      g.a_map = am(P, AM_HN2);
      g.bn = 2 * PF_BN_GU;
      g.b_map0 = l * TM_PER_LAYER + TM_WG;
      g.b_row0 = n * PF_BN_GU;
      g.b_rows0 = PF_BN_GU;
      g.b_map1 = l * TM_PER_LAYER + TM_WU;
      g.b_row1 = n * PF_BN_GU;
      break;
    default:  // PF_DOWN
      g.K = P.F;
      g.a_map = am(P, AM_ACT);
      g.bn = PF_BN;
      g.b_map0 = l * TM_PER_LAYER + TM_WD;
      g.b_row0 = n * PF_BN;
      g.b_rows0 = PF_BN;
      break;
  }
  return g;
}

__device__ __forceinline__ int kv_row(const PfParams& P, int l, int kv, int g, int slot) {
  return (((l * 2 + kv) * P.max_batch + slot) * P.nkv + g) * P.max_ctx;
}

// The chunk that block m of the launch belongs to: its cache slot, its first
// block in the launch, the cache position of its first token, its length and
// its first token's index in `tokens`.  One prompt (no table): slot `slot`,
// position 0, length S.
struct PfBlk {
  int slot, first, pos0, len, tok;
};
__device__ __forceinline__ PfBlk pf_blk(const PfParams& P, int m) {
  if (!P.blk) return PfBlk{P.slot, 0, 0, P.S, 0};
  const int4 b = P.blk[m];
  return PfBlk{b.x & 0xffff, b.x >> 16, b.y, b.z, b.w};
}
// Where plane row p of the launch belongs: its chunk's cache slot, its cache
// position, the end of its chunk's keys, its index in `tokens`, and whether it
// holds a token (rows past a chunk's end pad its last block).
struct PfRow {
  int slot, pos, kend, tok;
  bool live;
};
__device__ __forceinline__ PfRow pf_row(const PfParams& P, int p) {
  const PfBlk b = pf_blk(P, p / PF_BM);
  const int r = p - b.first * PF_BM;  // row within the chunk
  PfRow w;
  w.slot = b.slot;
  w.pos = b.pos0 + r;
  w.kend = b.pos0 + b.len;
  w.tok = b.tok + r;
  w.live = r < b.len;
  return w;
}
// Key blocks (128 cache positions each, from position 0) that block m's rows
// attend to: up to its last live row's position (causal; keys before the
// chunk come from the cache, the chunk's own from its QKV tiles).
__device__ __forceinline__ int pf_key_blocks(const PfParams& P, int m) {
  const PfBlk b = pf_blk(P, m);
  const int r0 = (m - b.first) * PF_BM;
  const int last = (b.len < r0 + PF_BM ? b.len : r0 + PF_BM) - 1;
  return (b.pos0 + last) / PF_BM + 1;
}

// ---------------------------------------------------------------- producer
__device__ void pf_producer(const PfParams& P, const PfSh& S) {
  if ((threadIdx.x & 31) != 0) return;
  const uint64_t pol_w = policy_evict_first();  // weights: streamed
  const uint64_t pol_a = policy_evict_last();   // activations / KV: re-read by other tiles
  const uint32_t gen = S.flags[PFF_GEN];
  uint32_t stage_ctr = 0, islot_ctr = 0;
  bool first = true;
  for (;;) {
    uint32_t i;
    if (P.mode == MODE_MEGA) {
      i = ld_volatile(&P.ctl[CTL_ABORT]) ? PF_END : atomicAdd(&P.ctl[CTL_HEAD], 1u);
      if (i >= P.n_instr) i = PF_END;
    } else {
      i = first ? P.perop_base + blockIdx.x : PF_END;
      first = false;
    }
    const int si = islot_ctr % NISLOT;
    bool end = i == PF_END;
    if (!pf_wait(P, &S.iempty[si], ((islot_ctr / NISLOT) & 1u) ^ 1u)) end = true;
    Instr in;
    if (!end) {
      in = P.queue[i];
      *reinterpret_cast<Instr*>(S.islot + si * 48 + 16) = in;
    }
    *reinterpret_cast<volatile uint32_t*>(S.islot + si * 48) = end ? PF_END : i;
    mbar_arrive(&S.ifull[si]);
    ++islot_ctr;
    if (end) break;
    if (!pf_live(P, in)) continue;

    if (is_gemm(in.op)) {
      const PfGemm g = pf_gemm(P, in);
      const int nk = g.K / PF_BK;
      const int npre = nk < PF_NSTAGE ? nk : PF_NSTAGE;
      const uint32_t b_bytes = (uint32_t)g.bn * PF_BK * 2;
      const uint32_t tx = 2 * PF_A_BYTES + b_bytes;
      const uint32_t s0 = stage_ctr;
      // weights first: they depend on nothing
      for (int kb = 0; kb < npre; ++kb) {
        const int st = stage_ctr % PF_NSTAGE;
        pf_wait(P, &S.empty[st], ((stage_ctr / PF_NSTAGE) & 1u) ^ 1u);
        uint8_t* sp = S.ring + st * PF_STAGE + 2 * PF_A_BYTES;
        mbar_arrive_expect_tx(&S.full[st], tx);
        tma_load_2d(sp, tmap(P, g.b_map0), kb * PF_BK, g.b_row0, &S.full[st], pol_w);
        if (g.b_map1 >= 0)
          tma_load_2d(sp + g.b_rows0 * 128, tmap(P, g.b_map1), kb * PF_BK, g.b_row1, &S.full[st], pol_w);
        ++stage_ctr;
      }
      // (after a timeout the loads still run -- on stale but valid memory -- so
      // that every armed stage completes and the launch can drain)
      pf_wait_deps(P, in, gen, i);
      fence_proxy_async_global();
      const int arow = (int)in.a0 * PF_BM, lrow = arow + P.plane_rows;
      for (int kb = 0; kb < npre; ++kb) {
        uint8_t* sp = S.ring + ((s0 + kb) % PF_NSTAGE) * PF_STAGE;
        uint64_t* fb = &S.full[(s0 + kb) % PF_NSTAGE];
        tma_load_2d(sp, tmap(P, g.a_map), kb * PF_BK, arow, fb, pol_a);
        tma_load_2d(sp + PF_A_BYTES, tmap(P, g.a_map), kb * PF_BK, lrow, fb, pol_a);
      }
      for (int kb = npre; kb < nk; ++kb) {
        const int st = stage_ctr % PF_NSTAGE;
        pf_wait(P, &S.empty[st], ((stage_ctr / PF_NSTAGE) & 1u) ^ 1u);
        uint8_t* sp = S.ring + st * PF_STAGE;
        mbar_arrive_expect_tx(&S.full[st], tx);
        tma_load_2d(sp + 2 * PF_A_BYTES, tmap(P, g.b_map0), kb * PF_BK, g.b_row0, &S.full[st], pol_w);
        if (g.b_map1 >= 0)
          tma_load_2d(sp + 2 * PF_A_BYTES + g.b_rows0 * 128, tmap(P, g.b_map1), kb * PF_BK, g.b_row1,
                      &S.full[st], pol_w);
        tma_load_2d(sp, tmap(P, g.a_map), kb * PF_BK, arow, &S.full[st], pol_a);
        tma_load_2d(sp + PF_A_BYTES, tmap(P, g.a_map), kb * PF_BK, lrow, &S.full[st], pol_a);
        ++stage_ctr;
      }
    } else if (in.op == PF_ATTN) {
      pf_wait_deps(P, in, gen, i);
      fence_proxy_async_global();
      // one stage per key block: K_j at +0, V_j at +tile (Q goes to TMEM
      // through the compute warps)
      const int m = (int)in.a0, gq = (int)in.a1, l = in.layer;
      const int nkb = pf_key_blocks(P, m), slot = pf_blk(P, m).slot;
      const uint32_t tile = PF_BM * P.d * 2;  // one 128-row tile of d columns
      const int nbox = P.d / 64;
      for (int h = 0; h < P.rep; ++h)
        for (int j = 0; j < nkb; ++j) {
          const int st = stage_ctr % PF_NSTAGE;
          pf_wait(P, &S.empty[st], ((stage_ctr / PF_NSTAGE) & 1u) ^ 1u);
          uint8_t* sp = S.ring + st * PF_STAGE;
          mbar_arrive_expect_tx(&S.full[st], 2 * tile);
          for (int kvsel = 0; kvsel < 2; ++kvsel)
            for (int bx = 0; bx < nbox; ++bx)
              tma_load_2d(sp + kvsel * tile + bx * 16384, tmap(P, am(P, AM_KV)), bx * 64,
                          kv_row(P, l, kvsel, gq, slot) + j * PF_BM, &S.full[st], pol_a);
          ++stage_ctr;
        }
    }
  }
  // Before leaving, make sure the copies this thread issued have landed
  // (normally already consumed; after an abort some may still be in flight).
  for (uint32_t k = 0; k < PF_NSTAGE && k < stage_ctr; ++k) {
    const uint32_t c = stage_ctr - 1 - k;
    pf_wait(P, &S.full[c % PF_NSTAGE], (c / PF_NSTAGE) & 1u);
  }
}

// ---------------------------------------------------------------- tensor-core issuer
__device__ void pf_mma(const PfParams& P, const PfSh& S, uint32_t tbase) {
  if ((threadIdx.x & 31) != 0) return;
  uint32_t islot_ctr = 0, stage_ctr = 0, use[2] = {0, 0}, qctr = 0, sctr = 0;
  for (;;) {
    const int si = islot_ctr % NISLOT;
    pf_wait(P, &S.ifull[si], (islot_ctr / NISLOT) & 1u);
    const uint32_t i = *reinterpret_cast<volatile uint32_t*>(S.islot + si * 48);
    Instr in;
    if (i != PF_END) in = *reinterpret_cast<const Instr*>(S.islot + si * 48 + 16);
    mbar_arrive(&S.iempty[si]);
    ++islot_ctr;
    if (i == PF_END) break;
    if (!pf_live(P, in)) continue;
    if (is_gemm(in.op)) {
      const PfGemm g = pf_gemm(P, in);
      const int nk = g.K / PF_BK;
      const int ab = (int)((use[0] + use[1]) & 1u);
      pf_wait(P, &S.acce[ab], (use[ab] & 1u) ^ 1u);
      ++use[ab];
      tc_fence_after();
      const uint32_t d = tbase + (uint32_t)ab * 256;
      const uint32_t idesc = idesc_bf16_f32(PF_BM, g.bn);
      for (int kb = 0; kb < nk; ++kb) {
        const int st = stage_ctr % PF_NSTAGE;
        pf_wait(P, &S.full[st], (stage_ctr / PF_NSTAGE) & 1u);
        ++stage_ctr;
        tc_fence_after();
        const uint32_t a0 = smem_u32(S.ring + st * PF_STAGE);
        const uint32_t a1 = a0 + PF_A_BYTES, b0 = a0 + 2 * PF_A_BYTES;
#pragma unroll
        for (int k = 0; k < PF_BK / 16; ++k) {
          const uint64_t bd = sdesc_sw128(b0 + 32 * k);
          tc_mma(d, sdesc_sw128(a0 + 32 * k), bd, idesc, (kb | k) != 0);
          tc_mma(d, sdesc_sw128(a1 + 32 * k), bd, idesc, true);
        }
        tc_commit(&S.empty[st]);
      }
      tc_commit(&S.accf[ab]);
    } else if (in.op == PF_ATTN) {
      // attention takes both accumulators: S at +0, O at +128, P hi/lo at
      // +256/+320, Q hi/lo at +384/+448 (bf16 pairs, 16 elements per 8 columns)
      for (int b = 0; b < 2; ++b) {
        pf_wait(P, &S.acce[b], (use[b] & 1u) ^ 1u);
        ++use[b];
      }
      tc_fence_after();
      const int nkb = pf_key_blocks(P, (int)in.a0);
      const uint32_t s_t = tbase, o_t = tbase + 128, p_t = tbase + 256, pl_t = tbase + 320;
      const uint32_t q_t = tbase + 384, ql_t = tbase + 448;
      const uint32_t id_s = idesc_bf16_f32(PF_BM, PF_BM);
      const uint32_t id_o = idesc_bf16_f32(PF_BM, P.d, true);
      const uint32_t tile = PF_BM * P.d * 2;
      for (int h = 0; h < P.rep; ++h) {
        pf_wait(P, S.qfull, qctr & 1u);
        ++qctr;
        tc_fence_after();
        for (int j = 0; j < nkb; ++j) {
          // S = Q K_j^T (K = head_dim, in 64-column atoms 16 KB apart)
          const int st = stage_ctr % PF_NSTAGE;
          pf_wait(P, &S.full[st], (stage_ctr / PF_NSTAGE) & 1u);
          ++stage_ctr;
          tc_fence_after();
          const uint32_t kb0 = smem_u32(S.ring + st * PF_STAGE);
          for (int kk = 0; kk < P.d / 16; ++kk) {
            const uint64_t kd = sdesc_sw128(kb0 + (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u);
            tc_mma_ta(s_t, q_t + (uint32_t)kk * 8, kd, id_s, kk != 0);
            tc_mma_ta(s_t, ql_t + (uint32_t)kk * 8, kd, id_s, true);
          }
          tc_commit(S.sfull);
          // O_j = P_j V_j (P from TMEM, V as an MN-major operand)
          pf_wait(P, S.pfull, sctr & 1u);
          ++sctr;
          tc_fence_after();
          const uint32_t vb0 = kb0 + tile;
#pragma unroll
          for (int kk = 0; kk < PF_BM / 16; ++kk) {
            const uint64_t vd = sdesc_sw128_mn(vb0 + (uint32_t)kk * 2048u, 16384u);
            tc_mma_ta(o_t, p_t + (uint32_t)kk * 8, vd, id_o, kk != 0);
            tc_mma_ta(o_t, pl_t + (uint32_t)kk * 8, vd, id_o, true);
          }
          tc_commit(&S.empty[st]);
          tc_commit(S.ofull);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- compute warps
__device__ __forceinline__ void cbar_pf() { named_bar(PF_CBAR, PF_NC); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}
__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const float (&v)[16]) {
  uint4 a, b;
  a.x = pack_bf16(v[0], v[1]);   a.y = pack_bf16(v[2], v[3]);
  a.z = pack_bf16(v[4], v[5]);   a.w = pack_bf16(v[6], v[7]);
  b.x = pack_bf16(v[8], v[9]);   b.y = pack_bf16(v[10], v[11]);
  b.z = pack_bf16(v[12], v[13]); b.w = pack_bf16(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = a;
  reinterpret_cast<uint4*>(dst)[1] = b;
}
// (hi, lo) bf16 pairs of two values: hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_pack(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
  hi = (uint32_t)__bfloat16_as_ushort(ha) | ((uint32_t)__bfloat16_as_ushort(hb) << 16);
  lo = pack_bf16(a - __bfloat162float(ha), b - __bfloat162float(hb));
}
__device__ __forceinline__ void store_split8(uint16_t* hi, uint16_t* lo, const float* v) {
  uint4 h, l;
  split_pack(v[0], v[1], h.x, l.x);
  split_pack(v[2], v[3], h.y, l.y);
  split_pack(v[4], v[5], h.z, l.z);
  split_pack(v[6], v[7], h.w, l.w);
  *reinterpret_cast<uint4*>(hi) = h;
  *reinterpret_cast<uint4*>(lo) = l;
}
__device__ __forceinline__ void store_split16(uint16_t* hi, uint16_t* lo, const float (&v)[16]) {
  store_split8(hi, lo, v);
  store_split8(hi + 8, lo + 8, v + 8);
}
__device__ __forceinline__ float bf(const uint16_t* p, int i) {
  return __uint_as_float((uint32_t)__ldg(p + i) << 16);
}

// QKV epilogue of one head: columns [c0, c0 + d) of the tile accumulator.
// The TMEM loads run on every thread of the warp; only live rows store.
__device__ void pf_qkv_head(const PfParams& P, uint32_t tacc, int c0, int col, int p, int l,
                            const PfRow& pr) {
  const bool live = pr.live;
  const int d = P.d, qd = P.nq * d, kd = P.nkv * d;
  const LayerW& W = P.layers[l];
  const bool is_v = col >= qd + kd;
  const int half = d / 2;
  if (is_v) {
    const int g = (col - qd - kd) / d;
    uint16_t* dst = P.kv + ((size_t)kv_row(P, l, 1, g, pr.slot) + pr.pos) * d;
    for (int c = 0; c < d; c += 16) {
      float v[16];
      tmem_ld16(tacc + (uint32_t)(c0 + c), v);
      if (live) store_bf16x16(dst + c, v);
    }
    return;
  }
  const bool is_q = col < qd;
  float inv = 1.f;
  const uint16_t* gn = nullptr;
  if (P.qk_norm) {
    gn = is_q ? W.q_norm : W.k_norm;
    float ss = 0.f;
    for (int c = 0; c < d; c += 16) {
      float v[16];
      tmem_ld16(tacc + (uint32_t)(c0 + c), v);
#pragma unroll
      for (int e = 0; e < 16; ++e) ss = fmaf(v[e], v[e], ss);
    }
    inv = 1.0f / sqrtf(ss / (float)d + P.eps);
  }
  // queries: hi/lo planes (tensor-core operand); keys: the bf16 cache entry
  uint16_t* dst = is_q ? P.qb + (size_t)p * qd + col
                       : P.kv + ((size_t)kv_row(P, l, 0, (col - qd) / d, pr.slot) + pr.pos) * d;
  uint16_t* dst_lo = is_q ? dst + (size_t)P.plane_rows * qd : nullptr;
  const float2* rt = P.rope + (size_t)(pr.live ? pr.pos : 0) * half;
  for (int c = 0; c < half; c += 16) {
    float u1[16], u2[16];
    tmem_ld16(tacc + (uint32_t)(c0 + c), u1);
    tmem_ld16(tacc + (uint32_t)(c0 + c + half), u2);
    if (gn) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        u1[e] = u1[e] * inv * bf(gn, c + e);
        u2[e] = u2[e] * inv * bf(gn, c + half + e);
      }
    }
    float r1[16], r2[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float2 cs = __ldg(rt + c + e);
      r1[e] = u1[e] * cs.x - u2[e] * cs.y;
      r2[e] = u2[e] * cs.x + u1[e] * cs.y;
    }
    if (live) {
      if (is_q) {
        store_split16(dst + c, dst_lo + c, r1);
        store_split16(dst + c + half, dst_lo + c + half, r2);
      } else {
        store_bf16x16(dst + c, r1);
        store_bf16x16(dst + c + half, r2);
      }
    }
  }
}

// Every thread of a warp executes the TMEM loads (they are warp-collective);
// rows past the prompt are computed on a clamped row and not stored.
__device__ void pf_gemm_epilogue(const PfParams& P, const Instr& in, uint32_t tacc, int p_row) {
  const int l = in.layer, n = (int)in.a1;
  const PfRow pr = pf_row(P, p_row);
  const bool live = pr.live;
  const int p = live ? p_row : 0;  // dead rows read row 0's inputs and store nothing
  switch (in.op) {
    case PF_QKV: {
      const int base = n * P.bn_qkv;
      for (int c0 = 0; c0 < P.bn_qkv; c0 += P.d) pf_qkv_head(P, tacc, c0, base + c0, p, l, pr);
      break;
    }
    case PF_O:
    case PF_DOWN: {
      const int col0 = n * PF_BN;
      float* dst = (in.op == PF_O ? P.xa : P.xb) + (size_t)p * P.H + col0;
      const float* res = in.op == PF_O ? P.xb : P.xa;
      const uint16_t* emb = nullptr;
      if (in.op == PF_O && l == 0) {
        int tok = P.tokens[live ? pr.tok : 0];
        if (tok < 0 || tok >= P.V) tok = 0;
        emb = P.embed + (size_t)tok * P.H + col0;
      }
      for (int c = 0; c < PF_BN; c += 16) {
        float v[16];
        tmem_ld16(tacc + (uint32_t)c, v);
        float r[16];
        if (emb) {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = bf(emb, c + e);
        } else {
          const float4* rp = reinterpret_cast<const float4*>(res + (size_t)p * P.H + col0 + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 x = __ldcg(rp + q);
            r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
          }
        }
        float4* dp = reinterpret_cast<float4*>(dst + c);
        if (live) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dp[q] = make_float4(r[4 * q] + v[4 * q], r[4 * q + 1] + v[4 * q + 1],
                                r[4 * q + 2] + v[4 * q + 2], r[4 * q + 3] + v[4 * q + 3]);
        }
      }
      break;
    }
    case PF_LM: {  // logits of token p, vocabulary rows [256 n, 256 n + 256) (< V)
      const int col0 = n * PF_BN;
      float* dst = P.logits + (size_t)p * P.V + col0;
      for (int c = 0; c < PF_BN; c += 16) {
        float v[16];
        tmem_ld16(tacc + (uint32_t)c, v);
        if (live) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (col0 + c + e < P.V) dst[c + e] = v[e];
        }
      }
      break;
    }
    default: {  // PF_GU: columns [0,128) gate, [128,256) up
      uint16_t* dst = P.act + (size_t)p * P.F + n * PF_BN_GU;
      uint16_t* dst_lo = dst + (size_t)P.plane_rows * P.F;
      for (int c = 0; c < PF_BN_GU; c += 16) {
        float gt[16], up[16], a[16];
        tmem_ld16(tacc + (uint32_t)c, gt);
        tmem_ld16(tacc + (uint32_t)(PF_BN_GU + c), up);
#pragma unroll
        for (int e = 0; e < 16; ++e) a[e] = gt[e] / (1.0f + expf(-gt[e])) * up[e];
        if (live) store_split16(dst + c, dst_lo + c, a);
      }
      break;
    }
  }
}

// RMSNorm of one 128-token block: warp w handles rows w, w + 4, ...
__device__ void pf_norm(const PfParams& P, const Instr& in, int wc, int lane) {
  const int l = in.layer, m = (int)in.a0, H = P.H;
  // NORM1 (and the final norm, PF_NORMF) read the residual after the FFN and
  // write the hn1 planes; NORM2 reads the residual after attention
  const bool first = in.op == PF_NORM1;
  const bool fin = in.op == PF_NORMF;
  const float* src = (first || fin) ? P.xb : P.xa;
  const uint16_t* gain = fin ? P.final_norm : first ? P.layers[l].attn_norm : P.layers[l].ffn_norm;
  uint16_t* dst = (first || fin) ? P.hn1 : P.hn2;
  for (int r = wc; r < PF_BM; r += 4) {
    const int p = m * PF_BM + r;
    const PfRow pr = pf_row(P, p);
    if (!pr.live) break;
    const uint16_t* emb = nullptr;
    if (first && l == 0) {
      int tok = P.tokens[pr.tok];
      if (tok < 0 || tok >= P.V) {
        if (lane == 0) pf_error(P, MK_ERR_BOUNDS, (uint32_t)p);
        tok = 0;
      }
      emb = P.embed + (size_t)tok * H;
    }
    float ss = 0.f;
    for (int c = lane * 8; c < H; c += 256) {
      float x[8];
      if (emb) {
        widen8(__ldg(reinterpret_cast<const uint4*>(emb + c)), x);
      } else {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src + (size_t)p * H + c));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src + (size_t)p * H + c + 4));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
    }
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)H + P.eps);
    for (int c = lane * 8; c < H; c += 256) {
      float x[8], gw[8];
      if (emb) {
        widen8(__ldg(reinterpret_cast<const uint4*>(emb + c)), x);
      } else {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src + (size_t)p * H + c));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src + (size_t)p * H + c + 4));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      }
      widen8(__ldg(reinterpret_cast<const uint4*>(gain + c)), gw);
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = x[e] * inv * gw[e];
      store_split8(dst + (size_t)p * H + c, dst + ((size_t)P.plane_rows + p) * H + c, y);
    }
  }
}

// Softmax side of one (block, kv group).  Per head: this row's query (hi and
// lo planes) goes into TMEM as the A operand of S = Q K^T, then an online
// softmax runs over key blocks 0..m; P_j goes back into TMEM as (hi, lo) bf16
// pairs for O_j = P_j V_j, and O accumulates in registers (this thread's row).
template <int D>
__device__ void pf_attn(const PfParams& P, const PfSh& S, const Instr& in, uint32_t tbase, int row,
                        uint32_t lane_base, uint32_t& sctr) {
  const int m = (int)in.a0, gq = (int)in.a1, lane = threadIdx.x & 31;
  const int qi = m * PF_BM + row;  // < plane_rows: rows past the prompt are never stored
  // cache positions: this row's, and the end of its chunk's keys; key block j
  // holds positions 128 j .. 128 j + 127
  const PfRow pr = pf_row(P, qi);
  const int nkb = pf_key_blocks(P, m);
  const int qpos = pr.pos, klen = pr.kend;
  const int qd = P.nq * D;
  const float c = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(d)
  const uint32_t s_t = tbase + lane_base, o_t = tbase + 128 + lane_base;
  const uint32_t p_t = tbase + 256 + lane_base, pl_t = tbase + 320 + lane_base;
  const uint32_t q_t = tbase + 384 + lane_base, ql_t = tbase + 448 + lane_base;
  for (int h = 0; h < P.rep; ++h) {
    // The previous head's (or instruction's) S products completed before its
    // last S block was handed to these warps, so the Q columns are free.
    const uint16_t* qh = P.qb + (size_t)qi * qd + (size_t)(gq * P.rep + h) * D;
    const uint16_t* ql = qh + (size_t)P.plane_rows * qd;
#pragma unroll
    for (int c8 = 0; c8 < D / 2; c8 += 8) {
      const uint4 a = __ldcg(reinterpret_cast<const uint4*>(qh + 2 * c8));
      const uint4 b = __ldcg(reinterpret_cast<const uint4*>(qh + 2 * c8 + 8));
      const uint4 e = __ldcg(reinterpret_cast<const uint4*>(ql + 2 * c8));
      const uint4 f = __ldcg(reinterpret_cast<const uint4*>(ql + 2 * c8 + 8));
      const uint32_t wh[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const uint32_t wl[8] = {e.x, e.y, e.z, e.w, f.x, f.y, f.z, f.w};
      tmem_st8(q_t + (uint32_t)c8, wh);
      tmem_st8(ql_t + (uint32_t)c8, wl);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(S.qfull);

    float o[D];
#pragma unroll
    for (int e = 0; e < D; ++e) o[e] = 0.f;
    float mrun = -INFINITY, lrun = 0.f, alpha_prev = 0.f;
    for (int j = 0; j < nkb; ++j) {
      pf_wait(P, S.sfull, sctr & 1u);
      tc_fence_after();
      // the blocks that can hold keys past this row (the causal diagonal of a
      // chunk not aligned to 128 positions may cross two of them)
      const bool diag = (j + 1) * PF_BM > qpos || (j + 1) * PF_BM > klen;
      // pass 1: row max of the scaled scores
      float mx = -INFINITY;
      for (int c0 = 0; c0 < PF_BM; c0 += 16) {
        float s[16];
        tmem_ld16(s_t + (uint32_t)c0, s);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int kj = j * PF_BM + c0 + e;
          const bool masked = diag && (kj > qpos || kj >= klen);
          if (!masked) mx = fmaxf(mx, s[e] * c);
        }
      }
      const float mnew = fmaxf(mrun, mx);
      const float alpha = mrun == -INFINITY ? 0.f : exp2f(mrun - mnew);
      if (j > 0) {
        // O_{j-1} = P_{j-1} V_{j-1} was issued before S_j, so it is complete
        // (and P's columns are free); fold it in at the scale of block j-1
        pf_wait(P, S.ofull, (sctr - 1) & 1u);
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float v[16];
          tmem_ld16(o_t + (uint32_t)c0, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[c0 + e] = o[c0 + e] * alpha_prev + v[e];
        }
      }
      // pass 2: probabilities, row sum, (hi, lo) bf16 P into TMEM
      float sum = 0.f;
      for (int c0 = 0; c0 < PF_BM; c0 += 16) {
        float s[16];
        tmem_ld16(s_t + (uint32_t)c0, s);
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const int kj = j * PF_BM + c0 + e;
          const bool m0 = diag && (kj > qpos || kj >= klen);
          const bool m1 = diag && (kj + 1 > qpos || kj + 1 >= klen);
          const float p0 = m0 ? 0.f : exp2f(s[e] * c - mnew);
          const float p1 = m1 ? 0.f : exp2f(s[e + 1] * c - mnew);
          sum += p0 + p1;
          split_pack(p0, p1, hi[e / 2], lo[e / 2]);
        }
        tmem_st8(p_t + (uint32_t)(c0 / 2), hi);
        tmem_st8(pl_t + (uint32_t)(c0 / 2), lo);
      }
      lrun = lrun * alpha + sum;
      mrun = mnew;
      alpha_prev = alpha;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(S.pfull);
      ++sctr;
    }
    pf_wait(P, S.ofull, (sctr - 1) & 1u);
    tc_fence_after();
    const float linv = 1.0f / lrun;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      float v[16];
      tmem_ld16(o_t + (uint32_t)c0, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) o[c0 + e] = (o[c0 + e] * alpha_prev + v[e]) * linv;
    }
    if (pr.live) {
      uint16_t* dst = P.ao + (size_t)qi * qd + (size_t)(gq * P.rep + h) * D;
      uint16_t* dst_lo = dst + (size_t)P.plane_rows * qd;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = o[c0 + e];
        store_split16(dst + c0, dst_lo + c0, v);
      }
    }
  }
}

__device__ void pf_compute(const PfParams& P, const PfSh& S, uint32_t tbase) {
  const int wc = (threadIdx.x >> 5) - 2;  // 0..3
  const int lane = threadIdx.x & 31;
  const int tc = threadIdx.x - 64;
  const int q = (threadIdx.x >> 5) & 3;   // TMEM lane quarter this warp may access
  const int row = 32 * q + lane;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const uint32_t gen = S.flags[PFF_GEN];
  // use[]: hand-outs of each accumulator (GEMM tiles and attention), which pace
  // the "accumulator free" barrier; gemm_use[]: GEMM tiles only, which pace the
  // "accumulator full" barrier (attention commits none)
  uint32_t islot_ctr = 0, use[2] = {0, 0}, gemm_use[2] = {0, 0}, sctr = 0;
  for (;;) {
    const int si = islot_ctr % NISLOT;
    if (tc == 0) {
      uint32_t v = PF_END;
      if (pf_wait(P, &S.ifull[si], (islot_ctr / NISLOT) & 1u))
        v = *reinterpret_cast<volatile uint32_t*>(S.islot + si * 48);
      S.flags[PFF_SLOT] = v;
    }
    cbar_pf();
    const uint32_t i = S.flags[PFF_SLOT];
    Instr in;
    if (i != PF_END) in = *reinterpret_cast<const Instr*>(S.islot + si * 48 + 16);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.iempty[si]);
    ++islot_ctr;
    if (i == PF_END) break;
    const bool live = pf_live(P, in);
    if (live) {
      if (is_gemm(in.op)) {
        const int ab = (int)((use[0] + use[1]) & 1u);
        pf_wait(P, &S.accf[ab], gemm_use[ab] & 1u);
        ++use[ab];
        ++gemm_use[ab];
        tc_fence_after();
        pf_gemm_epilogue(P, in, tbase + (uint32_t)ab * 256 + lane_base, (int)in.a0 * PF_BM + row);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.acce[ab]);
      } else if (in.op == PF_ATTN) {
        // the queries are read here with plain loads: wait for their QKV tiles
        // (after a timeout the launch drains on stale data, as the producer does)
        if (tc == 0) pf_wait_deps(P, in, gen, i);
        cbar_pf();
        use[0]++;
        use[1]++;
        if (P.d == 128) pf_attn<128>(P, S, in, tbase, row, lane_base, sctr);
        else pf_attn<64>(P, S, in, tbase, row, lane_base, sctr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.acce[0]);
          mbar_arrive(&S.acce[1]);
        }
      } else {
        if (tc == 0) S.flags[PFF_ABORT] = pf_wait_deps(P, in, gen, i) ? 0u : 1u;
        cbar_pf();
        if (!S.flags[PFF_ABORT]) pf_norm(P, in, wc, lane);
      }
    }
    fence_proxy_async_global();  // outputs are read by other CTAs' TMA loads
    cbar_pf();
    if (tc == 0 && P.mode == MODE_MEGA && in.rel_bar != NO_BAR)
      red_release_gpu_add(&P.bars[in.rel_bar], 1u);
  }
}

__global__ void __launch_bounds__(PF_THREADS, 1) mk_prefill_kernel(const __grid_constant__ PfParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const PfSh S = pf_map(smem);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PF_NSTAGE; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < NISLOT; ++s) {
      mbar_init(&S.ifull[s], 1);
      mbar_init(&S.iempty[s], 5);  // issuer + 4 compute warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.accf[b], 1);
      mbar_init(&S.acce[b], 4);
    }
    mbar_init(S.qfull, 4);  // the compute warps, once the head's queries are in TMEM
    mbar_init(S.sfull, 1);
    mbar_init(S.pfull, 4);
    mbar_init(S.ofull, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    S.flags[PFF_GEN] = P.mode == MODE_MEGA ? ld_volatile(&P.ctl[CTL_GEN]) : 0u;
  }
  if (warp == 1) tmem_alloc(reinterpret_cast<uint32_t*>(const_cast<uint32_t*>(&S.flags[PFF_TMEM])), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.flags[PFF_TMEM];
  if (warp == 0) pf_producer(P, S);
  else if (warp == 1) pf_mma(P, S, tbase);
  else pf_compute(P, S, tbase);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && P.mode == MODE_MEGA) {
    __threadfence();
    const uint32_t old = atomicAdd(&P.ctl[CTL_EXIT], 1u);
    if (old == gridDim.x - 1) {
      P.ctl[CTL_HEAD] = 0u;
      P.ctl[CTL_EXIT] = 0u;
      P.ctl[CTL_GEN] = S.flags[PFF_GEN] + 1u;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t pf_setup() {
  return cudaFuncSetAttribute(mk_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PfSmem::total);
}
cudaError_t pf_launch_mega(const PfParams& p, int ctas, cudaStream_t st) {
  PfParams pp = p;
  void* args[] = {(void*)&pp};
  return cudaLaunchCooperativeKernel((const void*)mk_prefill_kernel, dim3(ctas), dim3(PF_THREADS), args,
                                     (size_t)PfSmem::total, st);
}
cudaError_t pf_launch_perop(const PfParams& p, uint32_t first, uint32_t count, cudaStream_t st) {
  PfParams pp = p;
  pp.mode = MODE_PEROP;
  pp.perop_base = first;
  mk_prefill_kernel<<<count, PF_THREADS, PfSmem::total, st>>>(pp);
  return cudaGetLastError();
}

}  // namespace mk
