// select_resident_update: the selection and residency bookkeeping of one decode step in one
// kernel -- dual top-k selection ([NOSA] "Method 1"), set difference against the resident pages
// ([NOSA] "Method 2: NOSI") and the bucketed LRU update ([Spin] 2B) -- with results identical
// to select_topk, resident_setdiff and lru_bucket_update called in turn.  The pages describe the
// three operations separately; running them as one kernel (one launch, each unit's tables read
// once, the selected list handed over in shared memory) is this library's choice.
//
// One CTA of 256 threads per unit.  Up to 2048 slots, every thread first loads its eight slots'
// resident ids and timestamps into registers (slot tid + 256 k), so the loads overlap the
// selection and neither core reads the rows again; more slots, the other warps prefetch the rows
// into L2 instead.  Warp 0 selects (warp form, scores in registers) while the other warps clear
// the slot list; then all threads run the set-difference and LRU cores of resid.cuh on the list
// in shared memory.
#include "common.cuh"
#include "internal.h"
#include "resid.cuh"
#include "select_warp.cuh"

namespace spkv {
namespace {

constexpr int kFuseThreads = 256;   // several CTAs per SM fit beside the selection warp's registers
constexpr int kRegSlots = 8;        // slots per thread kept in registers (n_slots <= 2048)

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <int R>
__global__ void __launch_bounds__(kFuseThreads, R >= 32 ? 1 : 2)
    select_resident_kernel(const float* __restrict__ qs, const float* __restrict__ es, uint32_t* __restrict__ alive,
                           const int32_t* __restrict__ seq_len, int Hk, int np_max, int k_q, int k_e,
                           int32_t* __restrict__ sel, int32_t* __restrict__ n_sel, int32_t* __restrict__ resident,
                           int32_t* __restrict__ ts, int n_slots, int32_t t_now, int W, int32_t* __restrict__ missing,
                           int32_t* __restrict__ n_missing, int32_t* __restrict__ slot, int32_t* __restrict__ victims,
                           int32_t* __restrict__ hist_out, uint32_t* err) {
  extern __shared__ __align__(16) uint8_t fm[];
  __shared__ int hist[64], hist_u[64], warp_tot[kFuseThreads / 32];
  __shared__ int n_sh, nm_sh;
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.x, tid = threadIdx.x;
  const int stride = k_q + k_e + 1;
  int32_t* ssel = reinterpret_cast<int32_t*>(fm);
  int32_t* sslot = ssel + stride;
  LruSmem sm;
  sm.vic = sslot + stride;
  sm.bucket = reinterpret_cast<uint8_t*>(sm.vic + stride);
  sm.touched = sm.bucket + n_slots;
  sm.hist = hist;
  sm.hist_u = hist_u;
  sm.warp_tot = warp_tot;
  int32_t* rrow = resident + int64_t(u) * n_slots;
  int32_t* trow = ts + int64_t(u) * n_slots;
  const bool in_regs = n_slots <= kRegSlots * kFuseThreads;
  int rid[kRegSlots], tsv[kRegSlots];
  if (in_regs && tid >= 32) {   // warp 0 loads its share after the selection's loads
#pragma unroll
    for (int k = 0; k < kRegSlots; ++k) {
      const int s = tid + k * kFuseThreads;
      rid[k] = s < n_slots ? rrow[s] : -1;
      tsv[k] = s < n_slots ? trow[s] : 0;
    }
  }

  if (tid < 32) {
    const int n = warp_select_unit<R>(qs, es, alive, seq_len, u, Hk, np_max, k_q, k_e, sel, n_sel, ssel, err);
    if (tid == 0) n_sh = n;
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < kRegSlots; ++k) {
        const int s = tid + k * kFuseThreads;
        rid[k] = s < n_slots ? rrow[s] : -1;
        tsv[k] = s < n_slots ? trow[s] : 0;
      }
    }
  } else {
    for (int i = tid - 32; i < stride; i += kFuseThreads - 32) sslot[i] = -1;
    if (!in_regs) {
      const int lines = (n_slots * 4 + 127) / 128;   // 128-byte lines of each row
      for (int l = tid - 32; l < 2 * lines; l += kFuseThreads - 32)
        prefetch_l2(l < lines ? static_cast<const void*>(rrow + 32 * l) : static_cast<const void*>(trow + 32 * (l - lines)));
    }
  }
  __syncthreads();
  const int n = n_sh;
  int32_t* mrow = missing + int64_t(u) * stride;
  if (in_regs) {
    setdiff_core_regs(rid, ssel, n, stride, sslot, mrow, n_missing + u, slot + int64_t(u) * stride, &nm_sh, err);
    __syncthreads();   // the missing list and its length are visible now
    lru_core_regs(rid, tsv, rrow, trow, n_slots, sslot, n, mrow, nm_sh, stride, t_now, W,
                  victims + int64_t(u) * stride, hist_out + int64_t(u) * 64, sm, err);
  } else {
    setdiff_core(rrow, n_slots, ssel, n, stride, sslot, mrow, n_missing + u, slot + int64_t(u) * stride, err);
    __syncthreads();   // the missing list and its length (global, this CTA's writes) are visible now
    const int nm = n_missing[u];
    lru_core(rrow, trow, n_slots, sslot, n, mrow, nm, stride, t_now, W, victims + int64_t(u) * stride,
             hist_out + int64_t(u) * 64, sm, err);
  }
}

size_t fused_smem(int stride, int n_slots) { return size_t(3) * stride * 4 + size_t(2) * n_slots; }

}  // namespace

cudaError_t fused_init_attributes() {
  const int bytes = static_cast<int>(fused_smem(4096, 16384));
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(select_resident_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(select_resident_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(select_resident_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
      cudaSuccess)
    return e;
  return cudaFuncSetAttribute(select_resident_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

bool fused_supported(int np_max) { return np_max <= 32 * 32; }

cudaError_t launch_select_resident(const spkv_cache* c, const float* qs, const float* es, uint32_t* alive, int B,
                                   int np_max, const int32_t* seq_len, int k_q, int k_e, int32_t* sel,
                                   int32_t* n_sel, int32_t* resident, int32_t* ts, int n_slots, int32_t t_now,
                                   int W, int32_t* missing, int32_t* n_missing, int32_t* slot, int32_t* victims,
                                   int32_t* hist, cudaStream_t st) {
  const int Hk = c->d.n_kv_heads;
  const dim3 grid(B * Hk), block(kFuseThreads);
  const size_t smem = fused_smem(k_q + k_e + 1, n_slots);
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, grid, block, smem, st, qs, es, alive, seq_len, Hk, np_max, k_q, k_e, sel, n_sel,
                      resident, ts, n_slots, t_now, W, missing, n_missing, slot, victims, hist, c->dev_err);
  };
  if (np_max <= 32 * 4) return go(select_resident_kernel<4>);
  if (np_max <= 32 * 8) return go(select_resident_kernel<8>);
  if (np_max <= 32 * 16) return go(select_resident_kernel<16>);
  return go(select_resident_kernel<32>);
}

}  // namespace spkv
