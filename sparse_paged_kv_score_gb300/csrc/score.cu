// Block scores from the pooled-key summaries (second pooling stage + query dot).
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1": block-wise
// implementation (mean pooling inside sub-blocks, then max pooling to the block) feeding the
// query-aware selection Gamma_q.  For unit (b, h) and a complete page p before the local page:
//   s = max_j (sum_g q_g) . ksum[h][phys(p)][j] / (16 sqrt(128))
// The group's sub-block scores are summed before the max; by linearity the kernel forms the
// summed query once.  This pass is bound by HBM: it reads 2 KiB of fp32 summary per page-head
// (1 KiB with bf16 summaries: [Spin] 2C, cheaper scoring at long context).
//
// The fused decode form adds one block column that appends each request's new token (position
// seq_len - 1, in the request's local page) and refreshes that sub-block's sum.  The scores never
// read the local page, so doing both in one launch gives exactly append-then-score.
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "summary.cuh"

namespace spkv {
namespace {

constexpr int kWarps = 8;
constexpr int kPagesPerWarp = 16;                         // load rounds of four (fp32) or eight (bf16) pages
constexpr int kPagesPerBlock = kWarps * kPagesPerWarp;    // 128: a 512-page context is 4 CTAs per unit

// Lane l's four summary values of sub-block row `row` (dims 4 l .. 4 l + 3), as fp32.
template <bool BF16>
__device__ __forceinline__ float4 load4(const void* ksum, int64_t row, int lane) {
  if (BF16) {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(ksum) + row * (kHeadDim / 4) + lane);
    return make_float4(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x), bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
  }
  return __ldcs(reinterpret_cast<const float4*>(ksum) + row * (kHeadDim / 4) + lane);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The new K/V row of unit (b, h) into the request's local page, then that sub-block's sum again
// (threads 0..63: thread i owns dims 2i, 2i+1).  Each request's local page is its own, so the
// page count read here is the old one or already raised by head 0: the count used is the same.
template <bool BF16>
__device__ void append_local_row(const AppendRows& a, const int32_t* page_table, const PageDir& pd,
                                 const int32_t* seq_len, void* ksum, int np_max, int64_t n_phys, int b, int h, int Hk,
                                 uint32_t* err) {
  const int i = threadIdx.x;
  if (i >= kHeadDim / 2) return;
  const int L = seq_len[b];
  if (L < 1) return;                                  // flagged by the scoring blocks
  const int pg = (L - 1) / kPageTokens, t = (L - 1) % kPageTokens;
  if (pg >= np_max) {
    if (i == 0) flag_error(err, SPKV_DEVERR_PAGE_ID);
    return;
  }
  const int p = page_lookup(page_table, np_max, pd, b, pg);
  if (p < 0 || p >= n_phys) {
    if (i == 0) flag_error(err, SPKV_DEVERR_PHYS);
    return;
  }
  const int64_t ph = int64_t(h) * n_phys + p;
  const int64_t src = (int64_t(b) * Hk + h) * (kHeadDim / 2) + i;
  uint32_t* pw = a.kpool + ph * (kPageTokens * kHeadDim / 2);
  pw[t * (kHeadDim / 2) + i] = a.k_new[src];
  a.vpool[ph * (kPageTokens * kHeadDim / 2) + t * (kHeadDim / 2) + i] = a.v_new[src];
  int cnt = a.page_cnt[p];
  if (h == 0 && i == 0) atomicMax(&a.page_cnt[p], t + 1);
  cnt = max(0, min(kPageTokens, max(cnt, t + 1)));
  const int j = t / kSubblock;                        // this thread reads back its own word of row t
  store_pair<BF16>(ksum, (ph * kNSub + j) * (kHeadDim / 2) + i, subblock_sum(pw, j, cnt, i));
}

template <bool BF16, bool APPEND>
__global__ void __launch_bounds__(kWarps * 32)
    score_kernel(const uint32_t* __restrict__ q, const void* __restrict__ ksum, const int32_t* __restrict__ page_table,
                 const int32_t* __restrict__ seq_len, float* __restrict__ scores, int Hq, int Hk, int G, int np_max,
                 int64_t n_phys, float scale, uint32_t* err, AppendRows app, PageDir pd) {
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.y, b = u / Hk, h = u % Hk;
  if (APPEND && blockIdx.x == gridDim.x - 1) {
    append_local_row<BF16>(app, page_table, pd, seq_len, const_cast<void*>(ksum), np_max, n_phys, b, h, Hk, err);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p_begin = blockIdx.x * kPagesPerBlock;
  const int p_end = min(np_max, p_begin + kPagesPerBlock);
  // Each warp owns 16 consecutive pages: one load round for their physical ids (lanes 0..15,
  // issued before the query sum so both latencies overlap), then rounds of R pages x 4
  // sub-blocks = 4 R independent loads per lane (R = 4 fp32 pages, 16 bytes each, or 8 bf16
  // pages, 8 bytes each: 8 KiB in flight per warp either way).
  constexpr int R = BF16 ? 8 : 4;
  const int pw0 = p_begin + warp * kPagesPerWarp;
  int ph = 0;
  if (lane < kPagesPerWarp && pw0 + lane < p_end) ph = page_lookup(page_table, np_max, pd, b, pw0 + lane);
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
  const int64_t plane_rows = int64_t(h) * n_phys * kNSub;   // first sub-block row of this head
  float* srow = scores + int64_t(u) * np_max;
  bool okp = false;
  if (lane < kPagesPerWarp && pw0 + lane < p_end && pw0 + lane < local) {
    okp = ph >= 0 && ph < n_phys;
    if (!okp) flag_error(err, SPKV_DEVERR_PHYS);
  }
  if (!okp) ph = 0;
#pragma unroll
  for (int half = 0; half < kPagesPerWarp / R; ++half) {
    float4 v[R][kNSub];
    bool live[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int src = half * R + k;
      const int phk = __shfl_sync(0xffffffffu, ph, src);
      live[k] = __shfl_sync(0xffffffffu, okp ? 1 : 0, src) != 0;
      const int64_t row0 = plane_rows + int64_t(phk) * kNSub;
#pragma unroll
      for (int j = 0; j < kNSub; ++j)
        v[k][j] = live[k] ? load4<BF16>(ksum, row0 + j, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int pg = pw0 + half * R + k;
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
                         const int32_t* seq_len, float* scores, cudaStream_t st, const void* k_new,
                         const void* v_new, const PageDir* pd) {
  const int Hk = c->d.n_kv_heads;
  const int G = Hq / Hk;
  const bool append = k_new != nullptr;
  dim3 grid((np_max + kPagesPerBlock - 1) / kPagesPerBlock + (append ? 1 : 0), B * Hk);
  const float scale = static_cast<float>(1.0 / (16.0 * 11.313708498984760390));  // 1 / (16 sqrt(128))
  AppendRows app{static_cast<uint32_t*>(c->d.k_pool), static_cast<uint32_t*>(c->d.v_pool), c->d.page_cnt,
                 static_cast<const uint32_t*>(k_new), static_cast<const uint32_t*>(v_new)};
  auto kern = c->d.ksum_bf16 ? (append ? score_kernel<true, true> : score_kernel<true, false>)
                             : (append ? score_kernel<false, true> : score_kernel<false, false>);
  return launch_pdl(kern, grid, dim3(kWarps * 32), 0, st, static_cast<const uint32_t*>(q),
                    static_cast<const void*>(c->d.ksum), page_table, seq_len, scores, Hq, Hk, G, np_max,
                    static_cast<int64_t>(c->d.n_phys_pages), scale, c->dev_err, app, pd ? *pd : PageDir{});
}

}  // namespace spkv
