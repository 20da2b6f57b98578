// Tensor-core GEMM tile (tcgen05 + TMEM + TMA), the building block of the
// batched-decode and prefill projections, exposed on its own for testing:
//   C[M][N] (f32) = A[M][K] (bf16) * B[N][K]^T (bf16)
// One CTA per 128 x BN output tile.  Warp 0 streams A/B k-blocks (64 columns)
// into a 4-stage ring with 2D TMA loads; warp 1 allocates TMEM and issues
// tcgen05.mma (M = 128, N = BN, K = 16 per instruction), releasing each stage
// with tcgen05.commit; warps 2-5 read the f32 accumulator out of TMEM.
#include <cuda_runtime.h>

#include "../../include/mk.h"
#include "mk_device.cuh"
#include "mk_tc.cuh"
#include "mk_tmap.h"

namespace mk {
namespace {

constexpr int G_STAGES = 4;
constexpr int G_BM = 128;
constexpr int G_BK = 64;
constexpr int G_THREADS = 192;

template <int BN>
struct GemmSmem {
  static constexpr int a_bytes = G_BM * G_BK * 2;  // 16 KB
  static constexpr int b_bytes = BN * G_BK * 2;
  static constexpr int stage = a_bytes + b_bytes;
  static constexpr int bars = G_STAGES * stage;
  static constexpr int total = bars + (2 * G_STAGES + 1) * 8 + 16;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 2000000000ull) {
      atomicExch(err, (uint32_t)MK_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// BT: B stored [K][N] (N contiguous, the MN-major operand form), loaded as
// BN/64 boxes of 64 N-columns x 64 K-rows placed 8 KB apart.
template <int BN, bool BT>
__global__ void __launch_bounds__(G_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                   float* __restrict__ C, int M, int N, int K, uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using L = GemmSmem<BN>;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty = full + G_STAGES;
  uint64_t* done = empty + G_STAGES;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * G_BM, n0 = blockIdx.x * BN;
  const int nk = K / G_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0 && lane == 0) {
    const uint64_t pol = policy_evict_last();
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % G_STAGES;
      wait_bounded(&empty[s], ((kb / G_STAGES) & 1) ^ 1, err);
      uint8_t* st = smem + s * L::stage;
      mbar_arrive_expect_tx(&full[s], L::stage);
      tma_load_2d(st, &ta, kb * G_BK, m0, &full[s], pol);
      if constexpr (BT) {
#pragma unroll
        for (int i = 0; i < BN / 64; ++i)
          tma_load_2d(st + L::a_bytes + i * 8192, &tb, n0 + 64 * i, kb * G_BK, &full[s], pol);
      } else {
        tma_load_2d(st + L::a_bytes, &tb, kb * G_BK, n0, &full[s], pol);
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(G_BM, BN, BT);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % G_STAGES;
      wait_bounded(&full[s], (kb / G_STAGES) & 1, err);
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + s * L::stage);
      const uint32_t b0 = a0 + L::a_bytes;
#pragma unroll
      for (int k = 0; k < G_BK / 16; ++k) {
        const uint64_t bd = BT ? sdesc_sw128_mn(b0 + 2048 * k, 8192) : sdesc_sw128(b0 + 32 * k);
        tc_mma(tbase, sdesc_sw128(a0 + 32 * k), bd, idesc, (kb | k) != 0);
      }
      tc_commit(&empty[s]);
    }
    tc_commit(done);
  } else if (warp >= 2) {
    wait_bounded(done, 0, err);
    tc_fence_after();
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row = m0 + 32 * q + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      float v[16];
      tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
      if (row < M) {
        float4* dst = reinterpret_cast<float4*>(C + (size_t)row * N + n0 + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, BN);
  }
}

template <int BN, bool BT>
int run_gemm(const void* A, const void* B, float* C, int M, int N, int K, cudaStream_t st) {
  CUtensorMap ta, tb;
  const bool okb = BT ? make_tmap_bf16(&tb, B, (uint64_t)K, (uint64_t)N, 64)
                      : make_tmap_bf16(&tb, B, (uint64_t)N, (uint64_t)K, BN);
  if (!make_tmap_bf16(&ta, A, (uint64_t)M, (uint64_t)K, G_BM) || !okb) return MK_ERR_CUDA;
  static uint32_t* err = nullptr;
  if (!err) {
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return MK_ERR_CUDA;
  }
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), st) != cudaSuccess) return MK_ERR_CUDA;
  using L = GemmSmem<BN>;
  if (cudaFuncSetAttribute(tc_gemm_kernel<BN, BT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::total) != cudaSuccess)
    return MK_ERR_CUDA;
  dim3 grid(N / BN, (M + G_BM - 1) / G_BM);
  tc_gemm_kernel<BN, BT><<<grid, G_THREADS, L::total, st>>>(ta, tb, C, M, N, K, err);
  if (cudaGetLastError() != cudaSuccess) return MK_ERR_CUDA;
  uint32_t e = 0;
  if (cudaMemcpyAsync(&e, err, sizeof(e), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return MK_ERR_CUDA;
  return (int)e;
}

}  // namespace
}  // namespace mk

extern "C" int mk_debug_gemm_bf16(const void* A, const void* B, float* C, int M, int N, int K,
                                  int b_layout, void* stream) {
  if (!A || !B || !C || M < 1 || N < 128 || K < 64 || N % 128 || K % 64) return MK_ERR_INVALID_ARG;
  if (((uintptr_t)A | (uintptr_t)B | (uintptr_t)C) & 15u) return MK_ERR_INVALID_ARG;
  if (b_layout != 0 && b_layout != 1) return MK_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (b_layout == 1)
    return N % 256 == 0 ? mk::run_gemm<256, true>(A, B, C, M, N, K, st)
                        : mk::run_gemm<128, true>(A, B, C, M, N, K, st);
  return N % 256 == 0 ? mk::run_gemm<256, false>(A, B, C, M, N, K, st)
                      : mk::run_gemm<128, false>(A, B, C, M, N, K, st);
}
