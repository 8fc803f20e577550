// retrieve_pages: brings the selected pages that are not GPU-resident in from host memory.
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 2: the NOSI system":
//   the full KV cache is kept in host memory and a UVA host-to-device transfer kernel moves the
//   swapped-in blocks straight into their GPU buffer slots (no staging copy).
// [Spin] "Unifying Sparse Attention with Hierarchical Memory for Scalable Long-Context LLM
//   Serving", section 2A, the Retrieve operation (selected blocks fetched from the slower tier).
//
// The kernel reads the pinned host pool through its device-mapped address (on GB300 the loads
// cross NVLink-C2C) and writes each page into the victim slot the LRU update chose for it.  One
// CTA copies one page-head (16 KiB of K and 16 KiB of V) with all of its 16-byte loads in flight
// before the first store; the grid strides over the missing pages of all units, numbered through
// a per-unit prefix table that each CTA builds in shared memory.  It also completes
// the per-page slot list in place, so attention can read every selected page from its slot.
#include "common.cuh"
#include "internal.h"

namespace spkv {
namespace {

constexpr int kRtThreads = 256;
constexpr int kVecPerPage = 16384 / 16;                 // uint4 per K (or V) page-head
constexpr int kVecPerThread = kVecPerPage / kRtThreads;   // 4
constexpr int kMaxUnits = 4096;                           // largest max_units of a handle

__global__ void __launch_bounds__(kRtThreads)
    retrieve_kernel(const uint4* __restrict__ k_host, const uint4* __restrict__ v_host, int64_t n_host, int Hk,
                    const int32_t* __restrict__ page_table, int np_max, const int32_t* __restrict__ missing,
                    const int32_t* __restrict__ n_missing, const int32_t* __restrict__ victims,
                    int32_t* __restrict__ slot, const int32_t* __restrict__ n_sel, int stride, int n_units,
                    uint4* __restrict__ k_slots, uint4* __restrict__ v_slots, int64_t n_slot_pages, int n_slots,
                    uint32_t* err, PageDir pd) {
  __shared__ int prefix[kMaxUnits + 1];
  __shared__ int warp_tot[kRtThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 0. prefix[u] = first copy item of unit u (every CTA builds the table; n_units <= 4096)
  {
    const int c0 = static_cast<int>(int64_t(tid) * n_units / kRtThreads);
    const int c1 = static_cast<int>(int64_t(tid + 1) * n_units / kRtThreads);
    int sum = 0;
    for (int u = c0; u < c1; ++u) sum += max(0, min(stride, n_missing[u]));
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int acc = x - sum;
    for (int w = 0; w < warp; ++w) acc += warp_tot[w];
    for (int u = c0; u < c1; ++u) {
      prefix[u] = acc;
      acc += max(0, min(stride, n_missing[u]));
    }
    if (c1 == n_units) prefix[n_units] = acc;
    __syncthreads();
  }
  const int n_items = prefix[n_units];

  // 1. copies: item w = (unit u, missing index j)
  for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
    int lo = 0, hi = n_units;   // last u with prefix[u] <= w
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= w) lo = mid;
      else hi = mid;
    }
    const int u = lo, j = w - prefix[lo];
    const int b = u / Hk, h = u % Hk;
    const int lp = missing[int64_t(u) * stride + j];
    const int vs = victims[int64_t(u) * stride + j];
    uint32_t bad = 0;
    int64_t hp = -1;
    if (lp < 0 || lp >= np_max) bad |= SPKV_DEVERR_PAGE_ID;
    else {
      hp = page_lookup(page_table, np_max, pd, b, lp);
      if (hp < 0 || hp >= n_host) bad |= SPKV_DEVERR_PHYS;
    }
    if (vs < 0 || vs >= n_slots) bad |= SPKV_DEVERR_SLOT;
    if (bad) {
      if (tid == 0) flag_error(err, bad);
      continue;
    }
    const int64_t src = (int64_t(h) * n_host + hp) * kVecPerPage;
    const int64_t dst = (int64_t(h) * n_slot_pages + int64_t(b) * n_slots + vs) * kVecPerPage;
    uint4 kr[kVecPerThread], vr[kVecPerThread];
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) {
      kr[r] = __ldcs(k_host + src + r * kRtThreads + tid);
      vr[r] = __ldcs(v_host + src + r * kRtThreads + tid);
    }
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) {
      k_slots[dst + r * kRtThreads + tid] = kr[r];
      v_slots[dst + r * kRtThreads + tid] = vr[r];
    }
  }

  // 2. slot list: the r-th page of unit u without a slot (slot == -1, in list order, the order
  //    in which the set difference listed the missing pages) gets victims[r].
  const int warps = kRtThreads / 32;
  for (int u = blockIdx.x * warps + warp; u < n_units; u += gridDim.x * warps) {
    const int n = max(0, min(stride, n_sel[u]));
    const int nm = max(0, min(stride, n_missing[u]));
    int32_t* srow = slot + int64_t(u) * stride;
    const int32_t* vrow = victims + int64_t(u) * stride;
    int base = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      const int s = i < n ? srow[i] : 0;
      const bool need = i < n && s < 0;
      const unsigned bal = __ballot_sync(0xffffffffu, need);
      if (need) {
        const int r = base + __popc(bal & ((1u << lane) - 1u));
        const int v = r < nm ? vrow[r] : -1;
        if (v < 0 || v >= n_slots) flag_error(err, SPKV_DEVERR_SLOT);
        else srow[i] = v;
      }
      base += __popc(bal);
    }
    if (lane == 0 && base != nm) flag_error(err, SPKV_DEVERR_SLOT);
  }
}

}  // namespace

cudaError_t launch_retrieve(const spkv_cache* c, const void* k_host, const void* v_host, int64_t n_host_pages,
                            const int32_t* page_table, int np_max, int B, const int32_t* missing,
                            const int32_t* n_missing, const int32_t* victims, int32_t* slot, const int32_t* n_sel,
                            int sel_stride, int n_slots, cudaStream_t st, const PageDir* pd) {
  const int Hk = c->d.n_kv_heads;
  const int n_units = B * Hk;
  const int64_t items = int64_t(n_units) * sel_stride;
  const int64_t cap = int64_t(c->sm_count) * 4;   // 4 resident CTAs per SM (48 registers x 256 threads)
  const int grid = static_cast<int>(items < cap ? items : cap);
  return launch_pdl(retrieve_kernel, dim3(grid), dim3(kRtThreads), 0, st, static_cast<const uint4*>(k_host),
                    static_cast<const uint4*>(v_host), n_host_pages, Hk, page_table, np_max, missing, n_missing,
                    victims, slot, n_sel, sel_stride, n_units, static_cast<uint4*>(c->d.k_pool),
                    static_cast<uint4*>(c->d.v_pool), c->d.n_phys_pages, n_slots, c->dev_err, pd ? *pd : PageDir{});
}

}  // namespace spkv
