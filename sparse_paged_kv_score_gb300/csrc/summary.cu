// Pooled-key summaries (first pooling stage) and token append.
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1", block-wise
// implementation: the selection score pools keys by their mean inside 16-token sub-blocks.
// [NOSA] section "Method 2: NOSI", kernel fusion: pooling is produced where K is written.
// We keep the fp32 *sum* of each sub-block's valid keys (mean = sum / count), written in a fixed
// token order so that a create and any sequence of appends give bitwise the same sums; a handle
// with bf16 summaries stores that fp32 sum rounded once to bf16 (round to nearest even).
#include "common.cuh"
#include "internal.h"
#include "summary.cuh"

namespace spkv {
namespace {

// One group of 64 threads per page-head; thread i owns dims 2i, 2i+1.
template <bool BF16>
__global__ void __launch_bounds__(256) summary_build_kernel(const uint32_t* __restrict__ kpool, void* __restrict__ ksum,
                                                            const int32_t* __restrict__ page_cnt, int64_t n_ph,
                                                            int64_t n_phys) {
  pdl_wait();
  pdl_trigger();
  const int64_t ph = int64_t(blockIdx.x) * 4 + threadIdx.x / 64;
  if (ph >= n_ph) return;
  const int i = threadIdx.x % 64;
  const int cnt = max(0, min(kPageTokens, page_cnt[ph % n_phys]));
  const uint32_t* pw = kpool + ph * (kPageTokens * kHeadDim / 2);
#pragma unroll
  for (int j = 0; j < kNSub; ++j)
    store_pair<BF16>(ksum, (ph * kNSub + j) * (kHeadDim / 2) + i, subblock_sum(pw, j, cnt, i));
}

// Writes row r of every head into the pool and raises page_cnt.  One 64-thread group per
// (row, head).
__global__ void __launch_bounds__(256) append_write_kernel(uint32_t* __restrict__ kpool, uint32_t* __restrict__ vpool,
                                                           int32_t* __restrict__ page_cnt, const int32_t* __restrict__ phys,
                                                           const int32_t* __restrict__ tok, const uint32_t* __restrict__ k_new,
                                                           const uint32_t* __restrict__ v_new, int n_rows, int Hk,
                                                           int64_t n_phys, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int64_t item = int64_t(blockIdx.x) * 4 + threadIdx.x / 64;
  if (item >= int64_t(n_rows) * Hk) return;
  const int row = static_cast<int>(item / Hk), h = static_cast<int>(item % Hk);
  const int i = threadIdx.x % 64;
  const int p = phys[row], t = tok[row];
  if (p < 0 || p >= n_phys || t < 0 || t >= kPageTokens) {
    if (i == 0 && h == 0) flag_error(err, (p < 0 || p >= n_phys) ? SPKV_DEVERR_PHYS : SPKV_DEVERR_PAGE_ID);
    return;
  }
  const int64_t dst = ((int64_t(h) * n_phys + p) * kPageTokens + t) * (kHeadDim / 2) + i;
  const int64_t src = (int64_t(row) * Hk + h) * (kHeadDim / 2) + i;
  kpool[dst] = k_new[src];
  vpool[dst] = v_new[src];
  if (i == 0 && h == 0) atomicMax(&page_cnt[p], t + 1);
}

// Recomputes the sub-block sum that row r touched, for every head.
template <bool BF16>
__global__ void __launch_bounds__(256) append_sum_kernel(const uint32_t* __restrict__ kpool, void* __restrict__ ksum,
                                                         const int32_t* __restrict__ page_cnt,
                                                         const int32_t* __restrict__ phys, const int32_t* __restrict__ tok,
                                                         int n_rows, int Hk, int64_t n_phys) {
  pdl_wait();
  pdl_trigger();
  const int64_t item = int64_t(blockIdx.x) * 4 + threadIdx.x / 64;
  if (item >= int64_t(n_rows) * Hk) return;
  const int row = static_cast<int>(item / Hk), h = static_cast<int>(item % Hk);
  const int i = threadIdx.x % 64;
  const int p = phys[row], t = tok[row];
  if (p < 0 || p >= n_phys || t < 0 || t >= kPageTokens) return;
  const int j = t / kSubblock;
  const int cnt = max(0, min(kPageTokens, page_cnt[p]));
  const int64_t ph = int64_t(h) * n_phys + p;
  const uint32_t* pw = kpool + ph * (kPageTokens * kHeadDim / 2);
  store_pair<BF16>(ksum, (ph * kNSub + j) * (kHeadDim / 2) + i, subblock_sum(pw, j, cnt, i));
}

}  // namespace

cudaError_t launch_summary_build(const spkv_cache* c, cudaStream_t st) {
  const int64_t n_ph = int64_t(c->d.n_kv_heads) * c->d.n_phys_pages;
  if (n_ph == 0) return cudaSuccess;
  const int64_t blocks = (n_ph + 3) / 4;
  return launch_pdl(c->d.ksum_bf16 ? summary_build_kernel<true> : summary_build_kernel<false>,
                    dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, static_cast<const uint32_t*>(c->d.k_pool),
                    c->d.ksum, static_cast<const int32_t*>(c->d.page_cnt), n_ph, static_cast<int64_t>(c->d.n_phys_pages));
}

cudaError_t launch_append(const spkv_cache* c, const int32_t* phys, const int32_t* tok, const void* k_new,
                          const void* v_new, int n_rows, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const int Hk = c->d.n_kv_heads;
  const int64_t blocks = (int64_t(n_rows) * Hk + 3) / 4;
  cudaError_t e = launch_pdl(append_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                             static_cast<uint32_t*>(c->d.k_pool), static_cast<uint32_t*>(c->d.v_pool),
                             c->d.page_cnt, phys, tok, static_cast<const uint32_t*>(k_new),
                             static_cast<const uint32_t*>(v_new), n_rows, Hk, static_cast<int64_t>(c->d.n_phys_pages),
                             c->dev_err);
  if (e != cudaSuccess) return e;
  return launch_pdl(c->d.ksum_bf16 ? append_sum_kernel<true> : append_sum_kernel<false>,
                    dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, static_cast<const uint32_t*>(c->d.k_pool),
                    c->d.ksum, static_cast<const int32_t*>(c->d.page_cnt), phys, tok, n_rows, Hk,
                    static_cast<int64_t>(c->d.n_phys_pages));
}

}  // namespace spkv
