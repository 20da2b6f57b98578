// Compiled specialisations of the interpreter kernel.  Each is one
// translation unit (compiled in parallel); the host picks the one that matches
// the model shape, else the generic one.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {

struct KernelVariant {
  int mh, mf, ad, arep;  // register-path K multiples (0: generic), head_dim, q heads per kv head
  cudaError_t (*setup)();
  cudaError_t (*occupancy)(int* per_sm);
  cudaError_t (*mega)(const KParams& p, int ctas, cudaStream_t st);
  cudaError_t (*mega_steps)(const KParams& p, int ctas, cudaStream_t st);  // mk_decode_steps
  cudaError_t (*perop)(const KParams& p, uint32_t first, uint32_t count, int ctas, cudaStream_t st);
};

// Shapes with a batch-1 register-path specialisation (K = M * 2048).
struct VariantShape {
  int mh, mf, ad, arep;
};
constexpr VariantShape kFastShapes[] = {{1, 4, 64, 4}, {2, 7, 128, 4}, {2, 6, 128, 4}};

inline bool has_fast_variant(int hidden, int ffn, int q_heads, int kv_heads, int head_dim) {
  if (q_heads * head_dim != hidden || kv_heads < 1 || q_heads % kv_heads) return false;
  for (const VariantShape& v : kFastShapes)
    if (v.mh * 2048 == hidden && v.mf * 2048 == ffn && v.ad == head_dim &&
        v.arep == q_heads / kv_heads)
      return true;
  return false;
}

KernelVariant variant_generic();      // any supported shape
KernelVariant variant_h1_f4_d64_r4();  // hidden 2048, ffn 8192, head_dim 64, 4 q heads per kv head
KernelVariant variant_h2_f7_d128_r4(); // hidden 4096, ffn 14336, head_dim 128, 4 q / kv
KernelVariant variant_h2_f6_d128_r4(); // hidden 4096, ffn 12288, head_dim 128, 4 q / kv

}  // namespace mk
