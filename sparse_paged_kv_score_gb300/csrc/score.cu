// Block scores from the pooled-key summaries (second pooling stage + query dot).
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1": block-wise
// implementation (mean pooling inside sub-blocks, then max pooling to the block) feeding the
// query-aware selection Gamma_q.  For unit (b, h) and a complete page p before the local page:
//   s = max_j (sum_g q_g) . ksum[h][phys(p)][j] / (16 sqrt(128))
// The group's sub-block scores are summed before the max; by linearity the kernel forms the
// summed query once.  This pass is bound by HBM: it reads 2 KiB of fp32 summary per page-head.
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace spkv {
namespace {

constexpr int kPagesPerBlock = 64;
constexpr int kWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kWarps * 32)
    score_kernel(const uint32_t* __restrict__ q, const float* __restrict__ ksum, const int32_t* __restrict__ page_table,
                 const int32_t* __restrict__ seq_len, float* __restrict__ scores, int Hq, int Hk, int G, int np_max,
                 int64_t n_phys, float scale, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.y, b = u / Hk, h = u % Hk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p_begin = blockIdx.x * kPagesPerBlock;
  const int p_end = min(np_max, p_begin + kPagesPerBlock);
  // Each warp owns 8 consecutive pages: one load round for their physical ids (lanes 0..7,
  // issued before the query sum so both latencies overlap), then two rounds of 4 pages x 4
  // sub-blocks = 16 independent 16-byte loads per lane.
  const int pw0 = p_begin + warp * 8;
  int ph = 0;
  if (lane < 8 && pw0 + lane < p_end) ph = page_table[int64_t(b) * np_max + pw0 + lane];
  const int L = seq_len[b];
  __shared__ float qs[kHeadDim];
  if (tid < kHeadDim / 2) {
    float s0 = 0.f, s1 = 0.f;
    for (int g = 0; g < G; ++g) {
      const uint32_t w = q[(int64_t(b) * Hq + h * G + g) * (kHeadDim / 2) + tid];
      s0 += bf16lo_to_f32(w);
      s1 += bf16hi_to_f32(w);
    }
    qs[2 * tid] = s0;
    qs[2 * tid + 1] = s1;
  }
  __syncthreads();
  const float4 qv = reinterpret_cast<const float4*>(qs)[lane];
  const int local = L >= 1 ? (L - 1) / kPageTokens : 0;
  if (L < 1 && tid == 0 && blockIdx.x == 0) flag_error(err, SPKV_DEVERR_PAGE_ID);
  const float* plane = ksum + int64_t(h) * n_phys * (kNSub * kHeadDim);
  float* srow = scores + int64_t(u) * np_max;
  bool okp = false;
  if (lane < 8 && pw0 + lane < p_end && pw0 + lane < local) {
    okp = ph >= 0 && ph < n_phys;
    if (!okp) flag_error(err, SPKV_DEVERR_PHYS);
  }
  if (!okp) ph = 0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float4 v[4][kNSub];
    bool live[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int src = half * 4 + k;
      const int phk = __shfl_sync(0xffffffffu, ph, src);
      live[k] = __shfl_sync(0xffffffffu, okp ? 1 : 0, src) != 0;
      const float4* base = reinterpret_cast<const float4*>(plane + int64_t(phk) * (kNSub * kHeadDim));
#pragma unroll
      for (int j = 0; j < kNSub; ++j)
        v[k][j] = live[k] ? __ldcs(base + j * (kHeadDim / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pg = pw0 + half * 4 + k;
      float best = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < kNSub; ++j) {
        const float d = warp_sum(v[k][j].x * qv.x + v[k][j].y * qv.y + v[k][j].z * qv.z + v[k][j].w * qv.w);
        best = fmaxf(best, d);
      }
      if (lane == 0 && pg < p_end) srow[pg] = live[k] ? best * scale : -CUDART_INF_F;
    }
  }
}

}  // namespace

cudaError_t launch_score(const spkv_cache* c, const void* q, int B, int Hq, const int32_t* page_table, int np_max,
                         const int32_t* seq_len, float* scores, cudaStream_t st) {
  const int Hk = c->d.n_kv_heads;
  const int G = Hq / Hk;
  dim3 grid((np_max + kPagesPerBlock - 1) / kPagesPerBlock, B * Hk);
  const float scale = static_cast<float>(1.0 / (16.0 * 11.313708498984760390));  // 1 / (16 sqrt(128))
  return launch_pdl(score_kernel, grid, dim3(kWarps * 32), 0, st, static_cast<const uint32_t*>(q),
                    static_cast<const float*>(c->d.ksum), page_table, seq_len, scores, Hq, Hk, G, np_max,
                    static_cast<int64_t>(c->d.n_phys_pages), scale, c->dev_err);
}

}  // namespace spkv
