// Residency bookkeeping around the sparse decode step.
//
// resident_setdiff: [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 2:
//   NOSI", optimised memory layout -- a custom kernel computes the set difference between the
//   selected blocks and the GPU-resident blocks to decide what to swap in.
// lru_bucket_update: [Spin] "Unifying Sparse Attention with Hierarchical Memory for Scalable
//   Long-Context LLM Serving", section 2B, bucketed LRU -- resident pages are grouped into 64
//   recency buckets by timestamp so victims are chosen in parallel without a global sort.
//
// Both run one CTA per unit; everything is integer arithmetic and bitwise deterministic.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace spkv {
namespace {

constexpr int kSdThreads = 256;
constexpr int kLruThreads = 512;

__device__ int block_excl_scan_i(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < nw; ++w) {
    const int t = warp_tot[w];
    if (w < warp) base += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

__global__ void __launch_bounds__(kSdThreads)
    setdiff_kernel(const int32_t* __restrict__ resident, int n_slots, const int32_t* __restrict__ sel,
                   const int32_t* __restrict__ n_sel, int stride, int32_t* __restrict__ missing,
                   int32_t* __restrict__ n_missing, int32_t* __restrict__ slot, uint32_t* err) {
  extern __shared__ int32_t sd[];
  pdl_wait();
  pdl_trigger();
  int32_t* ssel = sd;
  int32_t* sslot = sd + stride;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int n = max(0, min(stride, n_sel[u]));
  const int32_t* srow = sel + int64_t(u) * stride;
  for (int i = tid; i < stride; i += blockDim.x) {
    ssel[i] = i < n ? srow[i] : INT_MAX;
    sslot[i] = -1;
  }
  __syncthreads();
  for (int i = tid; i + 1 < n; i += blockDim.x)
    if (ssel[i] >= ssel[i + 1]) flag_error(err, SPKV_DEVERR_ORDER);
  const int32_t* rrow = resident + int64_t(u) * n_slots;
  for (int s = tid; s < n_slots; s += blockDim.x) {
    const int id = rrow[s];
    if (id < 0) continue;
    int lo = 0, hi = n;  // binary search in the ascending selected list
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (ssel[mid] < id) lo = mid + 1;
      else hi = mid;
    }
    if (lo < n && ssel[lo] == id) {
      if (atomicCAS(&sslot[lo], -1, s) != -1) flag_error(err, SPKV_DEVERR_ORDER);
    }
  }
  __syncthreads();
  int32_t* mrow = missing + int64_t(u) * stride;
  int32_t* orow = slot + int64_t(u) * stride;
  for (int i = tid; i < stride; i += blockDim.x) orow[i] = sslot[i];
  if (tid < 32) {
    int base = 0;
    for (int i0 = 0; i0 < stride; i0 += 32) {
      const int i = i0 + tid;
      const bool miss = i < n && sslot[i] < 0;
      const unsigned bal = __ballot_sync(0xffffffffu, miss);
      if (miss) mrow[base + __popc(bal & ((1u << tid) - 1u))] = ssel[i];
      base += __popc(bal);
    }
    for (int i = base + tid; i < stride; i += 32) mrow[i] = -1;
    if (tid == 0) n_missing[u] = base;
  }
}

__global__ void __launch_bounds__(kLruThreads)
    lru_kernel(int32_t* __restrict__ resident, int32_t* __restrict__ ts, int n_slots, const int32_t* __restrict__ slot,
               const int32_t* __restrict__ n_sel, const int32_t* __restrict__ missing,
               const int32_t* __restrict__ n_missing, int stride, int32_t t_now, int W, int32_t* __restrict__ victims,
               int32_t* __restrict__ hist_out, uint32_t* err) {
  extern __shared__ uint8_t lm[];
  uint8_t* bucket = lm;
  uint8_t* touched = lm + n_slots;
  int32_t* vic = reinterpret_cast<int32_t*>(lm + ((2 * n_slots + 15) & ~15));
  __shared__ int hist[64], hist_u[64], warp_tot[kLruThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.x, tid = threadIdx.x;
  const int n = max(0, min(stride, n_sel[u]));
  int nm = max(0, min(stride, n_missing[u]));
  int32_t* rrow = resident + int64_t(u) * n_slots;
  int32_t* trow = ts + int64_t(u) * n_slots;
  const int32_t* srow = slot + int64_t(u) * stride;
  for (int s = tid; s < n_slots; s += blockDim.x) touched[s] = 0;
  if (tid < 64) hist[tid] = hist_u[tid] = 0;
  __syncthreads();
  // 1. touch the hits
  for (int i = tid; i < n; i += blockDim.x) {
    const int s = srow[i];
    if (s < 0) continue;
    if (s >= n_slots) {
      flag_error(err, SPKV_DEVERR_SLOT);
      continue;
    }
    trow[s] = t_now;
    touched[s] = 1;
  }
  __syncthreads();
  // 2. buckets and histograms
  for (int s0 = 0; s0 < n_slots; s0 += blockDim.x) {   // whole warps iterate together
    const int s = s0 + tid;
    int bk = 63;
    const bool in = s < n_slots;
    if (in && rrow[s] >= 0) {
      const int64_t age = int64_t(t_now) - trow[s];
      bk = age <= 0 ? 0 : static_cast<int>(age / W < 63 ? age / W : 63);
    }
    if (in) bucket[s] = static_cast<uint8_t>(bk);
    warp_hist_add(hist, bk, in);
    warp_hist_add(hist_u, bk, in && !touched[s]);
  }
  __syncthreads();
  int avail = 0;
  for (int k = 0; k < 64; ++k) avail += hist_u[k];
  if (nm > avail) {
    if (tid == 0) flag_error(err, SPKV_DEVERR_CAPACITY);
    nm = avail;
  }
  // 3. victims: untouched slots, oldest bucket first, ascending slot inside a bucket
  const int chunk = (n_slots + blockDim.x - 1) / blockDim.x;
  const int lo = min(n_slots, tid * chunk), hi = min(n_slots, lo + chunk);
  int filled = 0;
  for (int bk = 63; bk >= 0 && filled < nm; --bk) {
    if (hist_u[bk] == 0) continue;
    int mine = 0;
    for (int s = lo; s < hi; ++s) mine += (bucket[s] == bk && !touched[s]) ? 1 : 0;
    int total;
    int pos = filled + block_excl_scan_i(mine, warp_tot, &total);
    for (int s = lo; s < hi && pos < nm; ++s)
      if (bucket[s] == bk && !touched[s]) vic[pos++] = s;
    filled += min(total, nm - filled);
  }
  __syncthreads();
  // 4. install the missing pages
  const int32_t* mrow = missing + int64_t(u) * stride;
  int32_t* vrow = victims + int64_t(u) * stride;
  for (int i = tid; i < stride; i += blockDim.x) {
    if (i < nm) {
      const int s = vic[i];
      rrow[s] = mrow[i];
      trow[s] = t_now;
      vrow[i] = s;
    } else {
      vrow[i] = -1;
    }
  }
  if (tid < 64) hist_out[int64_t(u) * 64 + tid] = hist[tid];
}

}  // namespace

cudaError_t resid_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(setdiff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 4096 * 2 * 4);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lru_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * 16384 + 4096 * 4);
}

cudaError_t launch_setdiff(uint32_t* err, const int32_t* resident, int n_slots, const int32_t* sel,
                           const int32_t* n_sel, int sel_stride, int n_units, int32_t* missing, int32_t* n_missing,
                           int32_t* slot, cudaStream_t st) {
  if (n_units == 0) return cudaSuccess;
  const size_t smem = size_t(sel_stride) * 2 * sizeof(int32_t);
  return launch_pdl(setdiff_kernel, dim3(n_units), dim3(kSdThreads), smem, st, resident, n_slots, sel, n_sel,
                    sel_stride, missing, n_missing, slot, err);
}

cudaError_t launch_lru(uint32_t* err, int32_t* resident, int32_t* ts, int n_slots, const int32_t* slot,
                       const int32_t* n_sel, const int32_t* missing, const int32_t* n_missing, int sel_stride,
                       int n_units, int32_t t_now, int bucket_width, int32_t* victims, int32_t* hist,
                       cudaStream_t st) {
  if (n_units == 0) return cudaSuccess;
  const size_t smem = size_t((2 * n_slots + 15) & ~15) + size_t(sel_stride) * sizeof(int32_t);
  return launch_pdl(lru_kernel, dim3(n_units), dim3(kLruThreads), smem, st, resident, ts, n_slots, slot, n_sel,
                    missing, n_missing, sel_stride, t_now, bucket_width, victims, hist, err);
}

}  // namespace spkv
