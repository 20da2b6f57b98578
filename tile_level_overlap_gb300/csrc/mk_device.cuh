// Inline-PTX helpers for sm_103a: mbarriers, bulk async copies (TMA engine),
// gpu-scope acquire/release on barrier counters, timers, named barriers.
#pragma once
#include <stdint.h>

#include "mk_internal.h"

namespace mk {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive when `pred` holds (predicated inside the asm: no branch, so the
// caller's straight-line code stays one scheduling block).
__device__ __forceinline__ void mbar_arrive_if(uint64_t* bar, bool pred) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %1, 0;\n @p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(
          smem_u32(bar)),
      "r"((uint32_t)pred)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(tx)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- timers
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t smid() {
  uint32_t s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}

// ---------------------------------------------------------------- bulk copies
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Global -> shared bulk copy completing on `bar` (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- gpu-scope sync
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// ---------------------------------------------------------------- tagged words
// An element of an intermediate tensor of the decode step is one 64-bit word:
// the float in the low half, the tag of the launch step that wrote it in the
// high half.  An aligned 64-bit access is single-copy atomic, so a reader that
// sees the tag it expects also sees the value stored with it: each word is its
// own barrier (a barrier tensor partitioned down to single elements), and the
// writer needs no fence and no counter release after its stores.  (u64 is
// declared in mk_internal.h.)

__device__ __forceinline__ u64 tag_word(float v, uint32_t tag) {
  return ((u64)tag << 32) | (u64)__float_as_uint(v);
}
__device__ __forceinline__ float tag_val(u64 w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ uint32_t tag_of(u64 w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ void st_tagged(u64* p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(tag_word(v, tag)) : "memory");
}
__device__ __forceinline__ u64 ld_tagged(const u64* p) {
  u64 w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
// Two consecutive words (16-byte aligned); each is read atomically.
__device__ __forceinline__ void ld_tagged2(const u64* p, u64& a, u64& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Warpgroup register re-allocation (every warp of the warpgroup executes the
// same instruction): give registers back to the CTA's pool, or take them.
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

// Named barrier among `n` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void widen8(const uint4 w, float (&x)[8]) {
  x[0] = bf_lo(w.x); x[1] = bf_hi(w.x);
  x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
  x[4] = bf_lo(w.z); x[5] = bf_hi(w.z);
  x[6] = bf_lo(w.w); x[7] = bf_hi(w.w);
}

// a + sum_i w[i] * x[i] over 8 bf16 weights, in index order.
__device__ __forceinline__ float dot8(const uint4 w, const float* x, float a) {
  a = fmaf(bf_lo(w.x), x[0], a);
  a = fmaf(bf_hi(w.x), x[1], a);
  a = fmaf(bf_lo(w.y), x[2], a);
  a = fmaf(bf_hi(w.y), x[3], a);
  a = fmaf(bf_lo(w.z), x[4], a);
  a = fmaf(bf_hi(w.z), x[5], a);
  a = fmaf(bf_lo(w.w), x[6], a);
  a = fmaf(bf_hi(w.w), x[7], a);
  return a;
}

// Packed f32 pairs (sm_100 fma.rn.f32x2: two independent fp32 FMAs, each
// rounded once, in one instruction).  A pair is a u64: element 0 in the low
// word.
__device__ __forceinline__ u64 pack_f32x2(float lo, float hi) {
  return ((u64)__float_as_uint(hi) << 32) | (u64)__float_as_uint(lo);
}
__device__ __forceinline__ u64 fma_f32x2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// acc + (w's 8 bf16, as (even, odd) pairs) * x pairs: four packed FMAs, the
// even columns accumulating in the low lane, the odd ones in the high lane.
__device__ __forceinline__ u64 dot8_x2(const uint4 w, const u64 (&x)[4], u64 acc) {
  acc = fma_f32x2(((u64)(w.x & 0xffff0000u) << 32) | (u64)(w.x << 16), x[0], acc);
  acc = fma_f32x2(((u64)(w.y & 0xffff0000u) << 32) | (u64)(w.y << 16), x[1], acc);
  acc = fma_f32x2(((u64)(w.z & 0xffff0000u) << 32) | (u64)(w.z << 16), x[2], acc);
  acc = fma_f32x2(((u64)(w.w & 0xffff0000u) << 32) | (u64)(w.w << 16), x[3], acc);
  return acc;
}
__device__ __forceinline__ float pair_sum(u64 p) {
  return __uint_as_float((uint32_t)p) + __uint_as_float((uint32_t)(p >> 32));
}

// Warp-level tensor-core product c += A (16 x 16, rows g and g + 8 held as
// a0..a3) x B (16 x 8, b0..b1), bf16 operands, f32 accumulators; the standard
// m16n8k16 fragment layout (lane = 4 g + t).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Sums of four values over the 8 lanes of an aligned lane group (xor 4, 2, 1),
// as a multi-value butterfly: 4 shuffles instead of 12.  Afterwards the lane
// holds the total of value ((lane & 7) >> 1), in both lanes of each pair.
__device__ __forceinline__ float sum8_multi4(float (&a)[4], int lane) {
  const bool u4 = (lane & 4) != 0, u2 = (lane & 2) != 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = u4 ? a[k] : a[k + 2];
    const float keep = u4 ? a[k + 2] : a[k];
    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float send = u2 ? a[0] : a[1];
  float r = (u2 ? a[1] : a[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Reduce N (power of two, <= 32) per-lane values across the warp with a
// halving butterfly.  Returns the total of value index `warp_multi_index(lane)`
// (every lane pair {2k, 2k+1} holds the same index).
template <int N>
__device__ __forceinline__ float warp_reduce_multi(float (&v)[N], int lane) {
  int off = 16;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      float send = upper ? v[k] : v[k + n / 2];
      float keep = upper ? v[k + n / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
  for (; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}
template <int N>
__device__ __forceinline__ int warp_multi_index(int lane) {
  int idx = 0, off = 16;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, off >>= 1) idx = idx * 2 + ((lane & off) ? 1 : 0);
  return idx;
}

}  // namespace mk
