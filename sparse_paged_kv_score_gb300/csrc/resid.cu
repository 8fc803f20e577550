// Residency bookkeeping around the sparse decode step: the stand-alone set-difference and
// bucketed-LRU kernels (their per-unit cores, with citations, are in resid.cuh).
//
// Both run one CTA per unit; everything is integer arithmetic and bitwise deterministic.
#include "common.cuh"
#include "internal.h"
#include "resid.cuh"

namespace spkv {
namespace {

constexpr int kSdThreads = 256;
constexpr int kLruThreads = 512;

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
  setdiff_core(resident + int64_t(u) * n_slots, n_slots, ssel, n, stride, sslot, missing + int64_t(u) * stride,
               n_missing + u, slot + int64_t(u) * stride, err);
}

__global__ void __launch_bounds__(kLruThreads)
    lru_kernel(int32_t* __restrict__ resident, int32_t* __restrict__ ts, int n_slots, const int32_t* __restrict__ slot,
               const int32_t* __restrict__ n_sel, const int32_t* __restrict__ missing,
               const int32_t* __restrict__ n_missing, int stride, int32_t t_now, int W, int32_t* __restrict__ victims,
               int32_t* __restrict__ hist_out, uint32_t* err) {
  extern __shared__ uint8_t lm[];
  __shared__ int hist[64], hist_u[64], warp_tot[kLruThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.x;
  const int n = max(0, min(stride, n_sel[u]));
  const int nm = max(0, min(stride, n_missing[u]));
  LruSmem sm;
  sm.bucket = lm;
  sm.touched = lm + n_slots;
  sm.vic = reinterpret_cast<int32_t*>(lm + ((2 * n_slots + 15) & ~15));
  sm.hist = hist;
  sm.hist_u = hist_u;
  sm.warp_tot = warp_tot;
  lru_core(resident + int64_t(u) * n_slots, ts + int64_t(u) * n_slots, n_slots, slot + int64_t(u) * stride, n,
           missing + int64_t(u) * stride, nm, stride, t_now, W, victims + int64_t(u) * stride,
           hist_out + int64_t(u) * 64, sm, err);
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
