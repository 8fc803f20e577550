// Dual top-k page selection per (request, kv head) unit.
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1": dual selection
// (query-aware Gamma_q with budget k_q, query-agnostic eviction head Gamma_e with budget k_e),
// eviction policy (a block not chosen by Gamma_e can never be chosen by it again), locality
// guarantee, and ED-DMA (blocks ranked on pre-exp eviction scores; exp is never applied).
//
// Up to 1024 pages per unit: one warp per unit, scores in registers (warp form, below).
// Longer contexts: one CTA per unit.  Each top-k is an exact radix select over 32-bit order-preserving keys of
// the fp32 scores (4 passes of 8 bits, shared-memory histograms), followed by a page-ordered
// pick among keys equal to the threshold, which realises the total order
// (score descending, page ascending).  The union is emitted in ascending page order by a
// block-wide scan, then the local page.
#include "common.cuh"
#include "internal.h"
#include "select_warp.cuh"

namespace spkv {
namespace {

constexpr int kSelThreads = 512;
constexpr uint8_t kInE = 1, kInQ = 2;

struct SelShared {
  int hist[256];
  int warp_tot[kSelThreads / 32];
  int prefix;
  int remaining;
  int count;
};

// Exclusive scan of v over the block; returns the prefix and stores the total in *total.
__device__ int block_excl_scan(int v, int* warp_tot, int* total) {
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

__device__ int block_sum(int v, int* warp_tot) {
  int tot;
  block_excl_scan(v, warp_tot, &tot);
  return tot;
}

// Marks (flags |= bit) the k best candidates of keys[0..n) (cand[i] != 0), best = larger key,
// ties broken by smaller index.
__device__ void block_topk(const uint32_t* keys, const uint8_t* cand, uint8_t* flags, int n, int k, uint8_t bit,
                           SelShared& sh) {
  const int tid = threadIdx.x;
  int nc = 0;
  for (int i = tid; i < n; i += blockDim.x) nc += cand[i] ? 1 : 0;
  nc = block_sum(nc, sh.warp_tot);
  if (k <= 0) return;
  if (nc <= k) {
    for (int i = tid; i < n; i += blockDim.x)
      if (cand[i]) flags[i] |= bit;
    __syncthreads();
    return;
  }
  if (tid == 0) {
    sh.prefix = 0;
    sh.remaining = k;
  }
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int i = tid; i < 256; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t pre = static_cast<uint32_t>(sh.prefix);
    for (int i0 = 0; i0 < n; i0 += blockDim.x) {   // whole warps iterate together
      const int i = i0 + tid;
      const bool take = i < n && cand[i] && (keys[i] & hmask) == (pre & hmask);
      warp_hist_add(sh.hist, take ? static_cast<int>((keys[i] >> shift) & 255u) : 0, take);
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns bins 8*(31-L) .. 8*(31-L)+7, so lane 0 holds the largest bins
      const int lane = tid;
      int cnt[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cnt[q] = sh.hist[8 * (31 - lane) + 7 - q];  // q = 0 is the largest bin of the lane
        tot += cnt[q];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int above = incl - tot;  // keys in bins larger than this lane's block
      const int rem = sh.remaining;
      if (above < rem && rem <= incl) {
        int acc = above;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (acc + cnt[q] >= rem) {
            const int bin = 8 * (31 - lane) + 7 - q;
            sh.prefix = static_cast<int>(pre | (static_cast<uint32_t>(bin) << shift));
            sh.remaining = rem - acc;
            break;
          }
          acc += cnt[q];
        }
      }
    }
    __syncthreads();
  }
  const uint32_t thr = static_cast<uint32_t>(sh.prefix);
  const int need_eq = sh.remaining;
  // strictly better than the threshold: all taken; equal: the first need_eq in page order
  const int chunk = (n + blockDim.x - 1) / blockDim.x;
  const int lo = min(n, tid * chunk), hi = min(n, lo + chunk);
  int eq = 0;
  for (int i = lo; i < hi; ++i) {
    if (!cand[i]) continue;
    if (keys[i] > thr) flags[i] |= bit;
    else if (keys[i] == thr) ++eq;
  }
  int tot;
  int rank = block_excl_scan(eq, sh.warp_tot, &tot);
  for (int i = lo; i < hi && rank < need_eq; ++i) {
    if (cand[i] && keys[i] == thr) {
      flags[i] |= bit;
      ++rank;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const float* __restrict__ qs, const float* __restrict__ es, uint32_t* __restrict__ alive,
                  const int32_t* __restrict__ seq_len, int Hk, int np_max, int k_q, int k_e, int32_t* __restrict__ sel,
                  int32_t* __restrict__ n_sel, uint32_t* err) {
  extern __shared__ uint8_t sm[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(sm);
  uint8_t* cand = sm + sizeof(uint32_t) * np_max;
  uint8_t* flags = cand + np_max;
  __shared__ SelShared sh;
  pdl_wait();
  pdl_trigger();

  const int u = blockIdx.x, b = u / Hk, tid = threadIdx.x;
  const int L = seq_len[b];
  int local = L >= 1 ? (L - 1) / kPageTokens : 0;
  if (tid == 0 && (L < 1 || local >= np_max)) flag_error(err, SPKV_DEVERR_PAGE_ID);
  const int nc = min(local, np_max);
  const int words = (np_max + 31) / 32;
  const int64_t row = int64_t(u) * np_max;
  uint32_t* aw = alive + int64_t(u) * words;

  // query-score keys of this thread's first pages, loaded now so the load overlaps Gamma_e
  constexpr int kPre = 4;
  uint32_t qkey[kPre];
#pragma unroll
  for (int r = 0; r < kPre; ++r) {
    const int i = tid + r * blockDim.x;
    qkey[r] = i < np_max ? float_order_key(qs[row + i]) : 0u;
  }
  // ---- Gamma_e: top-k_e of the alive candidates by eviction score
  for (int i = tid; i < np_max; i += blockDim.x) {
    const bool a = (aw[i >> 5] >> (i & 31)) & 1u;
    cand[i] = (i < nc && a) ? 1 : 0;
    keys[i] = float_order_key(es[row + i]);
    flags[i] = 0;
  }
  __syncthreads();
  block_topk(keys, cand, flags, np_max, k_e, kInE, sh);
  // alive candidates outside E die
  for (int w = tid; w < words; w += blockDim.x) {
    uint32_t word = aw[w], clear = 0;
    for (int bit = 0; bit < 32; ++bit) {
      const int i = 32 * w + bit;
      if (i < nc && ((word >> bit) & 1u) && !(flags[i] & kInE)) clear |= 1u << bit;
    }
    if (clear) aw[w] = word & ~clear;
  }
  // ---- Gamma_q: top-k_q of the candidates outside E by query score
#pragma unroll
  for (int r = 0; r < kPre; ++r) {
    const int i = tid + r * blockDim.x;
    if (i < np_max) {
      cand[i] = (i < nc && !(flags[i] & kInE)) ? 1 : 0;
      keys[i] = qkey[r];
    }
  }
  for (int i = tid + kPre * blockDim.x; i < np_max; i += blockDim.x) {
    cand[i] = (i < nc && !(flags[i] & kInE)) ? 1 : 0;
    keys[i] = float_order_key(qs[row + i]);
  }
  __syncthreads();
  block_topk(keys, cand, flags, np_max, k_q, kInQ, sh);

  // ---- ascending union, then the local page
  const int stride = k_e + k_q + 1;
  const int chunk = (nc + blockDim.x - 1) / blockDim.x;
  const int lo = min(nc, tid * chunk), hi = min(nc, lo + chunk);
  int mine = 0;
  for (int i = lo; i < hi; ++i) mine += flags[i] ? 1 : 0;
  int total;
  int pos = block_excl_scan(mine, sh.warp_tot, &total);
  int32_t* out = sel + int64_t(u) * stride;
  for (int i = lo; i < hi; ++i)
    if (flags[i]) out[pos++] = i;
  for (int i = total + 1 + tid; i < stride; i += blockDim.x) out[i] = -1;
  if (tid == 0) {
    out[total] = local;
    n_sel[u] = total + 1;
  }
}

// ---------------------------------------------------------------- warp form (np_max <= 32 R)
// One warp per unit (warp_select_unit in select_warp.cuh), two units per 64-thread CTA.
template <int R>
__global__ void __launch_bounds__(64)
    select_warp_kernel(const float* __restrict__ qs, const float* __restrict__ es, uint32_t* __restrict__ alive,
                       const int32_t* __restrict__ seq_len, int Hk, int n_units, int np_max, int k_q, int k_e,
                       int32_t* __restrict__ sel, int32_t* __restrict__ n_sel, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (u >= n_units) return;
  warp_select_unit<R>(qs, es, alive, seq_len, u, Hk, np_max, k_q, k_e, sel, n_sel, nullptr, err);
}

}  // namespace

cudaError_t select_init_attributes() {
  return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32768 * 6);
}

cudaError_t launch_select(const spkv_cache* c, const float* qs, const float* es, uint32_t* alive, int B, int np_max,
                          const int32_t* seq_len, int k_q, int k_e, int32_t* sel, int32_t* n_sel, cudaStream_t st) {
  const int Hk = c->d.n_kv_heads;
  const int U = B * Hk;
  if (np_max <= 32 * 32) {
    // warp form: two units per 64-thread CTA, all scores in registers
    const dim3 grid((U + 1) / 2), block(64);
    if (np_max <= 32 * 4)
      return launch_pdl(select_warp_kernel<4>, grid, block, 0, st, qs, es, alive, seq_len, Hk, U, np_max, k_q, k_e,
                        sel, n_sel, c->dev_err);
    if (np_max <= 32 * 8)
      return launch_pdl(select_warp_kernel<8>, grid, block, 0, st, qs, es, alive, seq_len, Hk, U, np_max, k_q, k_e,
                        sel, n_sel, c->dev_err);
    if (np_max <= 32 * 16)
      return launch_pdl(select_warp_kernel<16>, grid, block, 0, st, qs, es, alive, seq_len, Hk, U, np_max, k_q,
                        k_e, sel, n_sel, c->dev_err);
    return launch_pdl(select_warp_kernel<32>, grid, block, 0, st, qs, es, alive, seq_len, Hk, U, np_max, k_q, k_e,
                      sel, n_sel, c->dev_err);
  }
  const size_t smem = size_t(np_max) * 6;
  return launch_pdl(select_kernel, dim3(B * Hk), dim3(kSelThreads), smem, st, qs, es, alive, seq_len, Hk, np_max,
                    k_q, k_e, sel, n_sel, c->dev_err);
}

}  // namespace spkv
