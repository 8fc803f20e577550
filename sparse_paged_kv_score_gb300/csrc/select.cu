// Dual top-k page selection per (request, kv head) unit.
//
// [NOSA] "NOSA: Native and Offloadable Sparse Attention", section "Method 1": dual selection
// (query-aware Gamma_q with budget k_q, query-agnostic eviction head Gamma_e with budget k_e),
// eviction policy (a block not chosen by Gamma_e can never be chosen by it again), locality
// guarantee, and ED-DMA (blocks ranked on pre-exp eviction scores; exp is never applied).
//
// Up to 1024 pages per unit: one warp per unit, scores in registers (warp form, select_warp.cuh).
// Longer contexts: one CTA per unit, each thread holding R consecutive pages' keys in registers.
// Each top-k finds the k-th largest of the candidates' 32-bit order-preserving keys of the fp32
// scores four bits at a time (a 16-bin count of the next digit within the group that shares the
// digits found so far, summed over the block), then takes every key above that group and the
// first keys of the group in page order (a block-wide scan over the threads' page ranges): the
// total order (score descending, page ascending) of the warp form, so both forms give identical
// results.  The union is emitted in ascending page order by a block-wide scan, then the local
// page.
#include "common.cuh"
#include "internal.h"
#include "select_warp.cuh"

namespace spkv {
namespace {

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

struct SelShared {
  uint32_t part[2][32][8];   // [search step parity][warp]: 16 digit counts, two 16-bit fields per word
  int warp_tot[32];
};

// The k best candidates (bit r of cand: page p0 + r) among this thread's R keys, over the block:
// returns this thread's taken bits.  Best = larger key, ties broken by smaller page.
template <int R>
__device__ uint32_t block_topk_reg(const uint32_t (&key)[R], uint32_t cand, int k, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int nc;
  block_excl_scan(__popc(cand), sh.warp_tot, &nc);
  if (k <= 0) return 0u;
  if (nc <= k) return cand;
  // The k-th largest key starts with the digits of `prefix` above bit s; `remaining` of the
  // candidates that share them (`in_group`) are still to be taken.  Once the two are equal, the
  // whole group is taken and the search stops.
  uint32_t prefix = 0;
  int remaining = k, in_group = nc, s = 28;
  for (int step = 0;; ++step, s -= 4) {
    // this thread's counts of the next digit among the group, widened to 16-bit fields (a bin
    // holds at most np_max <= 32768 keys over the block): word j holds bins 2j and 2j + 1
    uint32_t wsum[8];
    if (R <= 8) {   // at most 8 per bin: 4-bit fields, bins 0-7 in lo and 8-15 in hi
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const bool in = ((cand >> r) & 1u) && (s == 28 || (key[r] >> (s + 4)) == (prefix >> (s + 4)));
        const uint32_t d = (key[r] >> s) & 15u;
        const uint32_t inc = in ? (1u << (4 * (d & 7u))) : 0u;
        if (d & 8u) hi += inc;
        else lo += inc;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t src = j < 4 ? lo : hi;
        const int q = 2 * (j & 3);
        wsum[j] = ((src >> (4 * q)) & 0xFu) | (((src >> (4 * q + 4)) & 0xFu) << 16);
      }
    } else {   // up to 32 per bin: 8-bit fields
      uint64_t lo = 0, hi = 0;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const bool in = ((cand >> r) & 1u) && (s == 28 || (key[r] >> (s + 4)) == (prefix >> (s + 4)));
        const uint32_t d = (key[r] >> s) & 15u;
        const uint64_t inc = in ? (1ull << (8 * (d & 7u))) : 0ull;
        if (d & 8u) hi += inc;
        else lo += inc;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint64_t src = j < 4 ? lo : hi;
        const int q = 2 * (j & 3);
        wsum[j] = static_cast<uint32_t>((src >> (8 * q)) & 0xFFu) |
                  (static_cast<uint32_t>((src >> (8 * q + 8)) & 0xFFu) << 16);
      }
    }
    // Warp sum of the 8 words, scattered: halving rounds leave lane l with the sum of word
    // 4 b4 + 2 b3 + b2 (b = the bits of l), then two rounds add over the lanes that share it.
    uint32_t a4[4], a2[2], a1;
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      a4[j] = (b4 ? wsum[j + 4] : wsum[j]) + __shfl_xor_sync(0xffffffffu, b4 ? wsum[j] : wsum[j + 4], 16);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      a2[j] = (b3 ? a4[j + 2] : a4[j]) + __shfl_xor_sync(0xffffffffu, b3 ? a4[j] : a4[j + 2], 8);
    a1 = (b2 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? a2[0] : a2[1], 4);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
    // each warp's counts to shared memory (a buffer per step parity: a warp writes this buffer again
    // two steps on, after every warp has passed the next step's barrier), then every warp adds
    // them all up and takes the same decision
    uint32_t(*part)[8] = sh.part[step & 1];
    if ((lane & 3) == 0) part[warp][(b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0)] = a1;
    __syncthreads();
    // The digit D of the k-th largest: lane d < 16 adds up bin d over the warps and takes the count
    // of bins d and above (a suffix scan); D is the highest d whose count from the top reaches
    // `remaining`, and the bins above it are taken whole.
    uint32_t tw = 0;
    if (lane < 16)
      for (int w = 0; w < nw; ++w) tw += part[w][lane >> 1];
    const int c = lane < 16 ? static_cast<int>((tw >> (16 * (lane & 1))) & 0xFFFFu) : 0;
    int suf = c;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const int y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 16) suf += y;
    }
    const uint32_t reach = __ballot_sync(0xffffffffu, lane < 16 && suf >= remaining);
    const int D = 31 - __clz(reach);   // bin 0's count from the top is the whole group, so reach != 0
    const int above = __shfl_sync(0xffffffffu, suf - c, D);   // the count of bins above D
    in_group = __shfl_sync(0xffffffffu, c, D);
    remaining -= above;
    prefix |= static_cast<uint32_t>(D) << s;
    if (in_group == remaining || s == 0) break;   // the same outcome in every thread
  }
  // every key above the group, and the first `remaining` of the group in page order
  const uint32_t pg = prefix >> s;
  uint32_t take = 0;
  int eq = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!((cand >> r) & 1u)) continue;
    const uint32_t kg = key[r] >> s;
    if (kg > pg) take |= 1u << r;
    else if (kg == pg) ++eq;
  }
  int tot;
  int rank = block_excl_scan(eq, sh.warp_tot, &tot);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (((cand >> r) & 1u) && (key[r] >> s) == pg) {
      if (rank < remaining) take |= 1u << r;
      ++rank;
    }
  }
  return take;
}

// One CTA of THREADS per unit; thread t holds pages R t .. R t + R - 1 (np_max <= THREADS R).
template <int R, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    select_kernel(const float* __restrict__ qs, const float* __restrict__ es, uint32_t* __restrict__ alive,
                  const int32_t* __restrict__ seq_len, int Hk, int np_max, int k_q, int k_e, int32_t* __restrict__ sel,
                  int32_t* __restrict__ n_sel, uint32_t* err) {
  static_assert(R == 4 || R == 8 || R == 16 || R == 32, "R pages per thread: a divisor of 32, at least 4");
  __shared__ SelShared sh;
  pdl_wait();
  pdl_trigger();

  const int u = blockIdx.x, b = u / Hk, tid = threadIdx.x;
  const int L = seq_len[b];
  int local = L >= 1 ? (L - 1) / kPageTokens : 0;
  if (tid == 0 && (L < 1 || local >= np_max)) flag_error(err, SPKV_DEVERR_PAGE_ID);
  const int nc = min(local, np_max);
  const int64_t row = int64_t(u) * np_max;
  uint32_t* aw = alive + int64_t(u) * ((np_max + 31) / 32);
  const int p0 = R * tid;

  // keys of this thread's pages (0 past np_max; those are never candidates); the query-score keys
  // load beside the eviction keys while registers allow (R <= 16), else after Gamma_e
  const bool vec = (np_max & 3) == 0 && ((reinterpret_cast<uintptr_t>(qs) | reinterpret_cast<uintptr_t>(es)) & 15u) == 0;
  auto load_keys = [&](const float* src, uint32_t (&key)[R]) {
    if (vec) {
#pragma unroll
      for (int r = 0; r < R; r += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p0 + r < np_max) v = *reinterpret_cast<const float4*>(src + row + p0 + r);
        key[r] = float_order_key(v.x);
        key[r + 1] = float_order_key(v.y);
        key[r + 2] = float_order_key(v.z);
        key[r + 3] = float_order_key(v.w);
      }
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) key[r] = p0 + r < np_max ? float_order_key(src[row + p0 + r]) : 0u;
    }
  };
  constexpr bool kEarlyQ = R <= 16;
  uint32_t ek[R], qk[R];
  load_keys(es, ek);
  if (kEarlyQ) load_keys(qs, qk);
  // pages below the local page, and which of them are alive (this thread's R bits of its word)
  const int nv = min(R, max(0, nc - p0));
  const uint32_t vmask = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
  const uint32_t word = p0 < np_max ? aw[p0 >> 5] : 0u;
  const uint32_t abits = R == 32 ? word : ((word >> (p0 & 31)) & ((1u << (R & 31)) - 1u));

  // ---- Gamma_e: top-k_e of the alive candidates by eviction score
  const uint32_t cand_e = abits & vmask;
  const uint32_t in_e = block_topk_reg<R>(ek, cand_e, k_e, sh);
  // alive candidates outside E die: the threads of one alive word combine their bits, and the
  // first of them writes it
  uint32_t kill = (cand_e & ~in_e) << (R == 32 ? 0 : (p0 & 31));
#pragma unroll
  for (int o = 1; o < 32 / R; o <<= 1) kill |= __shfl_xor_sync(0xffffffffu, kill, o);
  if ((p0 & 31) == 0 && kill) aw[p0 >> 5] = word & ~kill;
  // ---- Gamma_q: top-k_q of the candidates outside E by query score
  if (!kEarlyQ) load_keys(qs, qk);
  const uint32_t in_q = block_topk_reg<R>(qk, vmask & ~in_e, k_q, sh);

  // ---- ascending union, then the local page
  const int stride = k_e + k_q + 1;
  const uint32_t f = in_e | in_q;
  int total;
  int pos = block_excl_scan(__popc(f), sh.warp_tot, &total);
  int32_t* out = sel + int64_t(u) * stride;
#pragma unroll
  for (int r = 0; r < R; ++r)
    if ((f >> r) & 1u) out[pos++] = p0 + r;
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

cudaError_t select_init_attributes() { return cudaSuccess; }

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
  // CTA form: 512 threads of 4, 8, 16 or 32 pages up to 16384 pages, then 1024 threads of 32
  const dim3 grid(U);
  if (np_max <= 512 * 4)
    return launch_pdl(select_kernel<4, 512>, grid, dim3(512), 0, st, qs, es, alive, seq_len, Hk, np_max, k_q, k_e, sel,
                      n_sel, c->dev_err);
  if (np_max <= 512 * 8)
    return launch_pdl(select_kernel<8, 512>, grid, dim3(512), 0, st, qs, es, alive, seq_len, Hk, np_max, k_q, k_e, sel,
                      n_sel, c->dev_err);
  if (np_max <= 512 * 16)
    return launch_pdl(select_kernel<16, 512>, grid, dim3(512), 0, st, qs, es, alive, seq_len, Hk, np_max, k_q, k_e, sel,
                      n_sel, c->dev_err);
  if (np_max <= 512 * 32)
    return launch_pdl(select_kernel<32, 512>, grid, dim3(512), 0, st, qs, es, alive, seq_len, Hk, np_max, k_q, k_e, sel,
                      n_sel, c->dev_err);
  return launch_pdl(select_kernel<32, 1024>, grid, dim3(1024), 0, st, qs, es, alive, seq_len, Hk, np_max, k_q, k_e, sel,
                    n_sel, c->dev_err);
}

}  // namespace spkv
