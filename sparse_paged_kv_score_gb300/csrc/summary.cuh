// Pooled-key sub-block sums: the one summation order shared by the summary build, the append
// and the fused decode append, so that every route gives bitwise the same sums.
#pragma once
#include "common.cuh"

namespace spkv {

// Sum of the valid rows of sub-block j of one page-head for dims 2i, 2i+1 (fixed token order).
__device__ __forceinline__ float2 subblock_sum(const uint32_t* page_words, int j, int cnt, int i) {
  float s0 = 0.f, s1 = 0.f;
  const int hi = min(kSubblock * (j + 1), cnt);
  for (int t = kSubblock * j; t < hi; ++t) {
    const uint32_t w = page_words[t * (kHeadDim / 2) + i];
    s0 += bf16lo_to_f32(w);
    s1 += bf16hi_to_f32(w);
  }
  return make_float2(s0, s1);
}

// Stores the sums of dims 2i, 2i+1 at element pair `pair` of the summary array (fp32 or bf16).
template <bool BF16>
__device__ __forceinline__ void store_pair(void* ksum, int64_t pair, float2 v) {
  if (BF16) reinterpret_cast<uint32_t*>(ksum)[pair] = pack_bf16x2(v.x, v.y);
  else reinterpret_cast<float2*>(ksum)[pair] = v;
}

}  // namespace spkv
