// Block scores from the pooled-key summaries (second pooling stage + query dot).
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1": block-wise
// implementation (mean pooling inside sub-blocks, then max pooling to the block) feeding the
// query-aware selection Gamma_q.  For unit (b, h) and a complete page p before the local page:
//   s = max_j (sum_g q_g) . ksum[h][phys(p)][j] / (16 sqrt(128))
// The group's sub-block scores are summed before the max; by linearity the kernel forms the
// summed query once.  This pass is bound by HBM: it reads 2 KiB of fp32 summary per page-head.
// Requires q 8-byte aligned (each lane reads 4 bf16 of a query row).
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace spkv {
namespace {

constexpr int kWarps = 8;
constexpr int kItemPages = 8;      // pages per warp item

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Persistent: every warp takes items of 8 consecutive pages of one unit, striding over all
// units' items, so the whole grid stays busy to the end (no partial last wave).  Per item: one
// load round for the 8 physical ids and the group's query rows -- issued one item ahead, so it
// overlaps the previous item -- then two rounds of 4 pages x 4 sub-blocks = 16 independent
// 16-byte loads per lane.
template <int GMAX>
struct ItemIn {
  int ph;          // lane < 8: physical page of page pw0 + lane
  uint2 qw[GMAX];  // this lane's 4 dims of each query row of the group (G <= GMAX)
  int L;
};

template <int GMAX>
__device__ __forceinline__ void load_item(ItemIn<GMAX>& in, int64_t it, int items_per_unit, const uint32_t* q,
                                          const int32_t* page_table, const int32_t* seq_len, int Hq, int Hk, int G,
                                          int np_max, int lane) {
  const int u = static_cast<int>(it / items_per_unit);
  const int pw0 = static_cast<int>(it % items_per_unit) * kItemPages;
  const int b = u / Hk, h = u % Hk;
  in.L = seq_len[b];
  in.ph = (lane < kItemPages && pw0 + lane < np_max) ? page_table[int64_t(b) * np_max + pw0 + lane] : 0;
#pragma unroll
  for (int g = 0; g < GMAX; ++g)
    in.qw[g] = g < G ? reinterpret_cast<const uint2*>(q + (int64_t(b) * Hq + h * G + g) * (kHeadDim / 2))[lane]
                     : make_uint2(0u, 0u);
}

template <int GMAX>
__global__ void __launch_bounds__(kWarps * 32)
    score_kernel(const uint32_t* __restrict__ q, const float* __restrict__ ksum, const int32_t* __restrict__ page_table,
                 const int32_t* __restrict__ seq_len, float* __restrict__ scores, int Hq, int Hk, int G, int np_max,
                 int64_t n_phys, float scale, uint32_t* err, int U) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int items_per_unit = (np_max + kItemPages - 1) / kItemPages;
  const int64_t n_items = int64_t(U) * items_per_unit;
  const int64_t wstride = int64_t(gridDim.x) * kWarps;
  int64_t it = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (it >= n_items) return;
  ItemIn<GMAX> cur;
  load_item(cur, it, items_per_unit, q, page_table, seq_len, Hq, Hk, G, np_max, lane);
  for (; it < n_items; it += wstride) {
    ItemIn<GMAX> nxt;
    if (it + wstride < n_items)
      load_item(nxt, it + wstride, items_per_unit, q, page_table, seq_len, Hq, Hk, G, np_max, lane);
    const int u = static_cast<int>(it / items_per_unit);
    const int pw0 = static_cast<int>(it % items_per_unit) * kItemPages;
    const int h = u % Hk;
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
      qv.x += bf16lo_to_f32(cur.qw[g].x);
      qv.y += bf16hi_to_f32(cur.qw[g].x);
      qv.z += bf16lo_to_f32(cur.qw[g].y);
      qv.w += bf16hi_to_f32(cur.qw[g].y);
    }
    const int L = cur.L;
    const int local = L >= 1 ? (L - 1) / kPageTokens : 0;
    if (L < 1 && lane == 0 && pw0 == 0) flag_error(err, SPKV_DEVERR_PAGE_ID);
    int ph = cur.ph;
    bool okp = false;
    if (lane < kItemPages && pw0 + lane < np_max && pw0 + lane < local) {
      okp = ph >= 0 && ph < n_phys;
      if (!okp) flag_error(err, SPKV_DEVERR_PHYS);
    }
    if (!okp) ph = 0;
    const float* plane = ksum + int64_t(h) * n_phys * (kNSub * kHeadDim);
    float* srow = scores + int64_t(u) * np_max;
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
        if (lane == 0 && pg < np_max) srow[pg] = live[k] ? best * scale : -CUDART_INF_F;
      }
    }
    cur = nxt;
  }
}

template <int GMAX>
cudaError_t launch_score_g(const spkv_cache* c, const void* q, int B, int Hq, const int32_t* page_table, int np_max,
                           const int32_t* seq_len, float* scores, cudaStream_t st) {
  static int per_sm[64] = {};   // resident CTAs per SM, looked up once per device
  const int dev = c->device < 64 ? c->device : 0;
  if (per_sm[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_kernel<GMAX>, kWarps * 32, 0) != cudaSuccess || n < 1)
      n = 1;
    per_sm[dev] = n;
  }
  const int Hk = c->d.n_kv_heads;
  const int G = Hq / Hk;
  const int U = B * Hk;
  const int64_t items = int64_t(U) * ((np_max + kItemPages - 1) / kItemPages);
  int64_t grid = int64_t(c->sm_count) * per_sm[dev];
  const int64_t need = (items + kWarps - 1) / kWarps;
  if (need < grid) grid = need;
  const float scale = static_cast<float>(1.0 / (16.0 * 11.313708498984760390));  // 1 / (16 sqrt(128))
  return launch_pdl(score_kernel<GMAX>, dim3(static_cast<unsigned>(grid)), dim3(kWarps * 32), 0, st,
                    static_cast<const uint32_t*>(q), static_cast<const float*>(c->d.ksum), page_table, seq_len,
                    scores, Hq, Hk, G, np_max, static_cast<int64_t>(c->d.n_phys_pages), scale, c->dev_err, U);
}

}  // namespace

cudaError_t launch_score(const spkv_cache* c, const void* q, int B, int Hq, const int32_t* page_table, int np_max,
                         const int32_t* seq_len, float* scores, cudaStream_t st) {
  const int G = Hq / c->d.n_kv_heads;
  if (G <= 4) return launch_score_g<4>(c, q, B, Hq, page_table, np_max, seq_len, scores, st);
  if (G <= 8) return launch_score_g<8>(c, q, B, Hq, page_table, np_max, seq_len, scores, st);
  return launch_score_g<16>(c, q, B, Hq, page_table, np_max, seq_len, scores, st);
}

}  // namespace spkv
