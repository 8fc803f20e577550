// Per-unit cores of the residency bookkeeping, shared by the stand-alone kernels (resid.cu) and
// the fused selection + residency kernel (fused.cu).  Every function is called by all threads of
// the CTA (they contain __syncthreads) and works on one unit.
//
// resident_setdiff: [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 2:
//   NOSI", optimised memory layout -- the set difference between the selected blocks and the
//   GPU-resident blocks decides what to swap in.
// lru_bucket_update: [Spin] "Unifying Sparse Attention with Hierarchical Memory for Scalable
//   Long-Context LLM Serving", section 2B, bucketed LRU -- resident pages are grouped into 64
//   recency buckets by timestamp so victims are chosen in parallel without a global sort.
#pragma once

#include <climits>

#include "common.cuh"

namespace spkv {

// Exclusive scan of v over the CTA; the total goes to *total.
__device__ __forceinline__ int block_excl_scan_i(int v, int* warp_tot, int* total) {
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

// Binary search of resident id `id` (slot s) in the ascending selected list; a hit records s.
__device__ __forceinline__ void setdiff_probe(int id, int s, const int32_t* ssel, int n, int32_t* sslot,
                                              uint32_t* err) {
  if (id < 0) return;
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ssel[mid] < id) lo = mid + 1;
    else hi = mid;
  }
  if (lo < n && ssel[lo] == id && atomicCAS(&sslot[lo], -1, s) != -1) flag_error(err, SPKV_DEVERR_ORDER);
}

// Second half of the set difference (after the probes and a barrier): the slot list, the missing
// list in ascending order (-1 padded) and its length, also to *nm_sh when it is not null.
__device__ __forceinline__ void setdiff_finish(const int32_t* ssel, int n, int stride, const int32_t* sslot,
                                               int32_t* __restrict__ mrow, int32_t* __restrict__ n_missing_u,
                                               int32_t* __restrict__ orow, int* nm_sh) {
  const int tid = threadIdx.x;
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
    if (tid == 0) {
      *n_missing_u = base;
      if (nm_sh) *nm_sh = base;
    }
  }
}

// Set difference of one unit.  On entry (after a barrier): ssel[0..n) is the selected list in
// ascending order and sslot[0..stride) == -1.  On return sslot[i] is the resident slot of
// ssel[i] (or -1), and missing (ascending, -1 padded), *n_missing and slot are written.
__device__ __forceinline__ void setdiff_core(const int32_t* __restrict__ rrow, int n_slots,
                                             const int32_t* ssel, int n, int stride, int32_t* sslot,
                                             int32_t* __restrict__ mrow, int32_t* __restrict__ n_missing_u,
                                             int32_t* __restrict__ orow, uint32_t* err) {
  const int tid = threadIdx.x;
  constexpr int kBatch = 4;   // resident ids loaded per thread before any is searched
  for (int s0 = tid; s0 < n_slots; s0 += kBatch * blockDim.x) {
    int id[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = s0 + k * blockDim.x;
      id[k] = s < n_slots ? rrow[s] : -1;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) setdiff_probe(id[k], s0 + k * static_cast<int>(blockDim.x), ssel, n, sslot, err);
  }
  __syncthreads();
  setdiff_finish(ssel, n, stride, sslot, mrow, n_missing_u, orow, nullptr);
}

// The same with the unit's resident ids already in registers: rid[k] is slot tid + k blockDim
// (-1 past n_slots).  Also leaves the missing count in *nm_sh (visible after a barrier).
template <int P>
__device__ __forceinline__ void setdiff_core_regs(const int (&rid)[P], const int32_t* ssel, int n, int stride,
                                                  int32_t* sslot, int32_t* __restrict__ mrow,
                                                  int32_t* __restrict__ n_missing_u, int32_t* __restrict__ orow,
                                                  int* nm_sh, uint32_t* err) {
#pragma unroll
  for (int k = 0; k < P; ++k)
    setdiff_probe(rid[k], static_cast<int>(threadIdx.x + k * blockDim.x), ssel, n, sslot, err);
  __syncthreads();
  setdiff_finish(ssel, n, stride, sslot, mrow, n_missing_u, orow, nm_sh);
}

// Shared-memory work space of lru_core.
struct LruSmem {
  uint8_t* bucket;    // [n_slots]
  uint8_t* touched;   // [n_slots]
  int32_t* vic;       // [stride]
  int* hist;          // [64]
  int* hist_u;        // [64] untouched slots per bucket
  int* warp_tot;      // [blockDim / 32]
};

// LRU steps 0-1: clear the work space, then touch the hits (timestamp t_now).  Ends on a barrier.
__device__ __forceinline__ void lru_touch(int32_t* __restrict__ trow, int n_slots, const int32_t* srow, int n,
                                          int32_t t_now, const LruSmem& sm, uint32_t* err) {
  const int tid = threadIdx.x;
  for (int s = tid; s < n_slots; s += blockDim.x) sm.touched[s] = 0;
  if (tid < 64) sm.hist[tid] = sm.hist_u[tid] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const int s = srow[i];
    if (s < 0) continue;
    if (s >= n_slots) {
      flag_error(err, SPKV_DEVERR_SLOT);
      continue;
    }
    trow[s] = t_now;
    sm.touched[s] = 1;
  }
  __syncthreads();
}

// LRU step 2 for one slot: its bucket and the two histograms (whole warps call it together).
__device__ __forceinline__ void lru_bucket_one(int s, bool in, int rv, int tv, int32_t t_now, int W,
                                               const LruSmem& sm) {
  int bk = 63;
  if (in && rv >= 0) {
    const int64_t age = int64_t(t_now) - tv;
    bk = age <= 0 ? 0 : static_cast<int>(age / W < 63 ? age / W : 63);
  }
  if (in) sm.bucket[s] = static_cast<uint8_t>(bk);
  warp_hist_add(sm.hist, bk, in);
  warp_hist_add(sm.hist_u, bk, in && !sm.touched[s]);
}

// LRU steps 3-4 (after the buckets and a barrier): victims are untouched slots, oldest bucket
// first, ascending slot inside a bucket; the missing pages are installed in them.
__device__ __forceinline__ void lru_pick_install(int32_t* __restrict__ rrow, int32_t* __restrict__ trow,
                                                 int n_slots, const int32_t* mrow, int nm, int stride,
                                                 int32_t t_now, int32_t* __restrict__ vrow,
                                                 int32_t* __restrict__ hist_row, const LruSmem& sm, uint32_t* err) {
  const int tid = threadIdx.x;
  int avail = 0;
  for (int k = 0; k < 64; ++k) avail += sm.hist_u[k];
  if (nm > avail) {
    if (tid == 0) flag_error(err, SPKV_DEVERR_CAPACITY);
    nm = avail;
  }
  const int chunk = (n_slots + blockDim.x - 1) / blockDim.x;
  const int lo = min(n_slots, tid * chunk), hi = min(n_slots, lo + chunk);
  int filled = 0;
  for (int bk = 63; bk >= 0 && filled < nm; --bk) {
    if (sm.hist_u[bk] == 0) continue;
    int mine = 0;
    for (int s = lo; s < hi; ++s) mine += (sm.bucket[s] == bk && !sm.touched[s]) ? 1 : 0;
    int total;
    int pos = filled + block_excl_scan_i(mine, sm.warp_tot, &total);
    for (int s = lo; s < hi && pos < nm; ++s)
      if (sm.bucket[s] == bk && !sm.touched[s]) sm.vic[pos++] = s;
    filled += min(total, nm - filled);
  }
  __syncthreads();
  for (int i = tid; i < stride; i += blockDim.x) {
    if (i < nm) {
      const int s = sm.vic[i];
      rrow[s] = mrow[i];
      trow[s] = t_now;
      vrow[i] = s;
    } else {
      vrow[i] = -1;
    }
  }
  if (tid < 64) hist_row[tid] = sm.hist[tid];
}

// Bucketed LRU update of one unit at time t_now; srow[0..n) is the slot list (slot of each
// selected page or -1), mrow[0..nm) the missing pages.  Needs no barrier before it.
__device__ __forceinline__ void lru_core(int32_t* __restrict__ rrow, int32_t* __restrict__ trow, int n_slots,
                                         const int32_t* srow, int n, const int32_t* mrow, int nm, int stride,
                                         int32_t t_now, int W, int32_t* __restrict__ vrow,
                                         int32_t* __restrict__ hist_row, const LruSmem& sm, uint32_t* err) {
  const int tid = threadIdx.x;
  lru_touch(trow, n_slots, srow, n, t_now, sm, err);
  constexpr int kBatch = 4;   // a batch of slots is loaded before any is bucketed
  for (int s0 = 0; s0 < n_slots; s0 += kBatch * blockDim.x) {
    int rv[kBatch], tv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = s0 + k * blockDim.x + tid;
      const bool in = s < n_slots;
      rv[k] = in ? rrow[s] : -1;
      tv[k] = in ? trow[s] : 0;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = s0 + k * blockDim.x + tid;
      lru_bucket_one(s, s < n_slots, rv[k], tv[k], t_now, W, sm);
    }
  }
  __syncthreads();
  lru_pick_install(rrow, trow, n_slots, mrow, nm, stride, t_now, vrow, hist_row, sm, err);
}

// The same with the unit's rows in registers as read before the update: rid[k], tsv[k] are the
// resident id and timestamp of slot tid + k blockDim.  A touched slot's timestamp is t_now, as
// lru_touch has just written it.
template <int P>
__device__ __forceinline__ void lru_core_regs(const int (&rid)[P], const int (&tsv)[P], int32_t* __restrict__ rrow,
                                              int32_t* __restrict__ trow, int n_slots, const int32_t* srow, int n,
                                              const int32_t* mrow, int nm, int stride, int32_t t_now, int W,
                                              int32_t* __restrict__ vrow, int32_t* __restrict__ hist_row,
                                              const LruSmem& sm, uint32_t* err) {
  lru_touch(trow, n_slots, srow, n, t_now, sm, err);
#pragma unroll
  for (int k = 0; k < P; ++k) {
    const int s = static_cast<int>(threadIdx.x + k * blockDim.x);
    const bool in = s < n_slots;
    lru_bucket_one(s, in, rid[k], in && sm.touched[s] ? t_now : tsv[k], t_now, W, sm);
  }
  __syncthreads();
  lru_pick_install(rrow, trow, n_slots, mrow, nm, stride, t_now, vrow, hist_row, sm, err);
}

}  // namespace spkv
