// Warp form of the dual top-k page selection, shared by select_topk (select.cu) and the fused
// selection + residency kernel (fused.cu).
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1": dual selection
// (Gamma_e eviction head over the pages still alive, then Gamma_q over the rest), eviction
// policy (an alive candidate left out of Gamma_e dies), ED-DMA (pre-exp scores are ranked).
//
// One warp per unit with every score in registers: lane l holds pages r * 32 + l, r < R, so row
// r of the warp is alive word r.  Each top-k finds the k-th largest key by a 32-step bitwise
// search (one warp reduction per bit), then takes the keys above it and the first keys equal to
// it in page order -- the total order (score descending, page ascending) of the CTA form, so
// both forms give identical results.
#pragma once

#include "common.cuh"

namespace spkv {

// Per-lane bit masks over rows: bit r = page r * 32 + lane.  Keys of non-candidates must be 0:
// every trial below has its own bit set, so a zero key never matches one and the search counts
// candidates only without testing cand in every step.
template <int R>
__device__ __forceinline__ uint32_t warp_topk(const uint32_t (&key)[R], uint32_t cand, int k) {
  const int lane = threadIdx.x & 31;
  const int nc = __reduce_add_sync(0xffffffffu, __popc(cand));
  if (k <= 0) return 0u;
  if (nc <= k) return cand;
  // The k-th largest key starts with `prefix` (its bits under hmask), `remaining` of the
  // candidates that start with it are still to be taken, and `in_group` candidates do.  Once the
  // two are equal, every key of the group is taken and the search can stop.
  uint32_t prefix = 0, hmask = 0;
  int remaining = k, in_group = nc;
  for (int bit = 31; bit >= 0 && in_group != remaining; --bit) {
    const uint32_t trial = prefix | (1u << bit);
    const uint32_t hm = ~((1u << bit) - 1u);   // bits >= bit
    int c4[4] = {0, 0, 0, 0};   // four partial counts: short dependency chains
#pragma unroll
    for (int r = 0; r < R; ++r) c4[r & 3] += (key[r] & hm) == trial;
    const int c = __reduce_add_sync(0xffffffffu, (c4[0] + c4[1]) + (c4[2] + c4[3]));
    hmask = hm;
    if (c >= remaining) {
      prefix = trial;
      in_group = c;
    } else {
      remaining -= c;
      in_group -= c;
    }
  }
  // take every key above the group, and the first `remaining` of the group in page order (all of
  // it when the search stopped early; after all 32 bits the group is the keys equal to the k-th)
  uint32_t take = 0;
  int seen = 0;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool c = (cand >> r) & 1u;
    const uint32_t km = key[r] & hmask;
    const bool eq = c && km == prefix;
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    const bool pick = (c && km > prefix) || (eq && seen + __popc(bal & lt) < remaining);
    take |= static_cast<uint32_t>(pick) << r;
    seen += __popc(bal);
  }
  return take;
}

// Selection of unit u by one warp (np_max <= 32 R): writes sel[u][*], n_sel[u], updates the
// alive words, and, if ssel is not null, also writes the list (ascending pages, then the local
// page) to ssel[0 .. n_sel).  Returns n_sel.
template <int R>
__device__ __forceinline__ int warp_select_unit(const float* __restrict__ qs, const float* __restrict__ es,
                                                uint32_t* __restrict__ alive, const int32_t* __restrict__ seq_len,
                                                int u, int Hk, int np_max, int k_q, int k_e,
                                                int32_t* __restrict__ sel, int32_t* __restrict__ n_sel,
                                                int32_t* ssel, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const int b = u / Hk;
  const int words = (np_max + 31) / 32;
  const int64_t row = int64_t(u) * np_max;
  uint32_t* aw = alive + int64_t(u) * words;
  // every load first (one round trip), the checks after
  const int L = seq_len[b];
  uint32_t ek[R], qk[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = r * 32 + lane;
    ek[r] = i < np_max ? float_order_key(es[row + i]) : 0u;
    qk[r] = i < np_max ? float_order_key(qs[row + i]) : 0u;
  }
  const uint32_t my_word = lane < words ? aw[lane] : 0u;   // lane r holds alive word r
  const int local = L >= 1 ? (L - 1) / kPageTokens : 0;
  if (lane == 0 && (L < 1 || local >= np_max)) flag_error(err, SPKV_DEVERR_PAGE_ID);
  const int nc = min(local, np_max);
  uint32_t in_range = 0, cand_e = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool ok = r * 32 + lane < nc;
    const uint32_t word = __shfl_sync(0xffffffffu, my_word, r);
    in_range |= static_cast<uint32_t>(ok) << r;
    cand_e |= static_cast<uint32_t>(ok && ((word >> lane) & 1u)) << r;
  }
  // ---- Gamma_e, then every alive candidate outside it dies
#pragma unroll
  for (int r = 0; r < R; ++r) ek[r] = ((cand_e >> r) & 1u) ? ek[r] : 0u;
  const uint32_t in_e = warp_topk<R>(ek, cand_e, k_e);
  uint32_t my_clear = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const unsigned clr = __ballot_sync(0xffffffffu, ((cand_e & ~in_e) >> r) & 1u);
    if (lane == r) my_clear = clr;
  }
  if (lane < words && my_clear) aw[lane] = my_word & ~my_clear;
  // ---- Gamma_q over the candidates outside E
  const uint32_t cand_q = in_range & ~in_e;
#pragma unroll
  for (int r = 0; r < R; ++r) qk[r] = ((cand_q >> r) & 1u) ? qk[r] : 0u;
  const uint32_t in_q = warp_topk<R>(qk, cand_q, k_q);
  // ---- ascending union, then the local page
  const int stride = k_e + k_q + 1;
  int32_t* out = sel + int64_t(u) * stride;
  const uint32_t flag = in_e | in_q;
  const uint32_t lt = (1u << lane) - 1u;
  int total = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool f = (flag >> r) & 1u;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (f) {
      const int pos = total + __popc(bal & lt);
      out[pos] = r * 32 + lane;
      if (ssel) ssel[pos] = r * 32 + lane;
    }
    total += __popc(bal);
  }
  for (int i = total + 1 + lane; i < stride; i += 32) out[i] = -1;
  if (lane == 0) {
    out[total] = local;
    if (ssel) ssel[total] = local;
    n_sel[u] = total + 1;
  }
  return total + 1;
}

}  // namespace spkv
