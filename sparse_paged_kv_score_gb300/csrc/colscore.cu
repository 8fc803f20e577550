// Column score S of the last alpha prompt rows (the PyramidKV-style sparsification score), on the
// 5th-generation tensor cores.
//
// [FA] "How KV sparsity achieves 1.5x acceleration for vLLM", section "2. Attention
// modification": the score of key i is the sum of the softmax probabilities the last alpha
// query rows give it, S_i = sum_j A[j][i]; softmax needs each row's maximum and sum (rowmax and
// l) first, so the page computes them in a FlashAttention pass and then the probabilities
// p = exp(q k - rowmax) / l in a second pass, with the loop order turned to k-major so that the
// sum over rows stays in registers, and skips work the causal mask zeroes.
//
// With the rows' log-sum-exp given (the attention that produced rowmax and l returns it), the first
// pass is skipped and each row's LSE is read instead; the rest is the same.
//
// One CTA per (request b, query head hq) and launch; a launch covers one chunk of up to 128 window
// rows (one M 128 tile).  Every row's softmax is its own, so the chunks' column sums add: the first
// launch writes them, later launches add theirs.  Eighteen warps:
//   warp 0     TMA producer: the K rows of two consecutive pages (two 64 x 64 bf16 boxes each,
//              128-byte swizzle, stacked into 128-row tiles) into a 3-stage ring, once for each
//              pass;
//   warp 1     MMA issuer (one thread): S = Q K^T (M 128 query rows, N 64 or 128 keys) into one
//              of two TMEM buffers, in both passes; a stage is released as soon as its MMA
//              completes (V is never needed);
//   warps 2-17 four column groups of 32 keys (warps 2-5, 6-9, 10-13, 14-17), one warp per TMEM
//              lane quarter in each, so a thread owns query row r (TMEM lane r) on 32 keys of the
//              pair.  Pass 1 keeps its causal row maximum and sum over its keys in the log2
//              domain; the four groups merge into the row log-sum-exp once.  Pass 2 turns the S
//              row into probabilities 2^(s scale - lse) and sums them over the rows (the page's
//              k-major loop order, the transpose done in registers): a butterfly across the
//              warp's 32 lanes leaves lane l with the sum of key l over its 32 rows, and the four
//              lane quarters' sums are added in shared memory in a fixed order by whichever of
//              the group's four warps finishes the job last (a counter per group and ring slot),
//              so no warp waits for another.  Three ring slots suffice: a warp can only start job
//              j + 3 after the MMA of job j + 3, which waits for every warp to have read job
//              j + 1 from TMEM, i.e. to have finished job j.
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace spkv {
namespace {

constexpr int kCM = 128;                    // tile rows: the window's query rows
constexpr int kCStages = 4;
constexpr int kCThreads = 576;
constexpr int kMathThreads = 512;
constexpr int kGroups = 4;                  // column groups of 32 keys in a page pair
constexpr int kBox = 64 * 128;              // one page's 64 rows x 128 B (one d-half)
constexpr int kGBox = 2 * kBox;             // two pages' rows of one d-half
constexpr int kCStageBytes = 2 * kGBox;     // K half 0, K half 1 of a page pair
constexpr int kQBytes = 2 * kCM * 128;
constexpr uint32_t kTmemCols = 512;         // two 128-column buffers (four in the LSE-only mode)

struct ColSmem {
  uint64_t full[kCStages], empty[kCStages];
  uint64_t dfull[4], dfree[4];
  uint64_t drain;
  uint64_t mlready;                         // every group's (max, sum) rows are published
  uint32_t tmem_base;
  float ml[kGroups][2][kCM];                // pass 1 -> 2: (max, sum) of each column group per row
  float part[3][4][kCM];                    // pass 2: column sums of each lane quarter (32 rows), 3 slots
  int cnt[3][kGroups];                      // pass 2: warps of a group done with a slot
};

constexpr size_t kColSmem = 1024 + kQBytes + size_t(kCStages) * kCStageBytes + sizeof(ColSmem);
static_assert(kColSmem <= 232448, "column-score shared memory exceeds the per-CTA limit");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kCThreads, 1)
    colscore_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ ColScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* stages = base + kQBytes;
  ColSmem& S = *reinterpret_cast<ColSmem*>(stages + kCStages * kCStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hq = blockIdx.x, b = blockIdx.y;
  // the chunk of window rows: this launch's, or blockIdx.z's when both chunks share one grid
  const bool in_grid = p.chunks_in_grid > 1;
  const int row0 = in_grid ? 128 * static_cast<int>(blockIdx.z) : p.row0;
  const int rows = in_grid ? min(128, p.alpha - row0) : p.rows;
  const int h = hq / p.G;

  if (tid == 0) {
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&S.dfull[i], 1);
      // LSE-only mode: buffer i is read by the four warps of group i alone
      mbar_init(&S.dfree[i], p.lse_out ? 4 : kMathThreads / 32);
    }
    mbar_init(&S.drain, 1);
    mbar_init(&S.mlready, kMathThreads / 32);
    for (int i = 0; i < 3 * kGroups; ++i) (&S.cnt[0][0])[i] = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmk);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();
  const int n = p.seq_len[b];
  const int np_b = min(p.np_max, (max(n, 0) + kPageTokens - 1) / kPageTokens);
  if (tid == 0 && (n < p.alpha || n > p.np_max * kPageTokens)) flag_error(p.err, SPKV_DEVERR_PAGE_ID);
  // the Q tile: row r < alpha is query row r of this head (bf16, 128-byte swizzle), others zero
  for (int i = tid; i < kCM * 16; i += kCThreads) {
    const int r = i >> 4, c = i & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows)
      v = *reinterpret_cast<const uint4*>(p.q + ((int64_t(b) * p.alpha + row0 + r) * p.Hq + hq) * kHeadDim + 8 * c);
    *reinterpret_cast<uint4*>(sQ + (c >> 3) * (kCM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem_base;
  const bool valid_req = n >= p.alpha && n <= p.np_max * kPageTokens;
  const int ng = valid_req ? (np_b + 1) / 2 : 0;   // page pairs
  // pass 1 (each row's maximum and sum), then pass 2 (the probabilities); with the rows'
  // log-sum-exp given by the caller, pass 2 alone
  const int p1 = p.lse_in ? 0 : ng;
  const int n_jobs = p1 + (p.lse_out ? 0 : ng);   // lse_out: pass 1 alone

  if (warp == 0) {
    // ================================================================ TMA producer
    const uint64_t pol = l2_policy_evict_last();   // each pair is read twice, and by the group's other heads
    int j = 0;
    for (; j < n_jobs; ++j) {
      const int s = j % kCStages, g = j % ng;
      if (j >= kCStages && !warp_wait(&S.empty[s], ((j / kCStages) - 1) & 1)) {
        if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        uint32_t bytes = 0;
        int ph[2] = {-1, -1};
        for (int k = 0; k < 2; ++k) {
          const int pg = 2 * g + k;
          if (pg >= np_b) continue;
          const int v = p.page_table[int64_t(b) * p.np_max + pg];
          if (v < 0 || v >= p.n_phys) {
            if (j < ng) flag_error(p.err, SPKV_DEVERR_PHYS);
            continue;
          }
          ph[k] = v;
          bytes += 2 * kBox;
        }
        uint8_t* st = stages + s * kCStageBytes;
        if (bytes) {
          mbar_arrive_expect_tx(&S.full[s], bytes);
          for (int k = 0; k < 2; ++k) {
            if (ph[k] < 0) continue;
            const int z = static_cast<int>(int64_t(h) * p.n_phys + ph[k]);
            tma_load_3d(st + k * kBox, &tmk, &S.full[s], 0, 0, z, pol);
            tma_load_3d(st + kGBox + k * kBox, &tmk, &S.full[s], 64, 0, z, pol);
          }
        } else {
          mbar_arrive(&S.full[s]);
        }
      }
      __syncwarp();
    }
    for (int i = j > kCStages ? j - kCStages : 0; i < j; ++i) mbar_wait(&S.full[i % kCStages], (i / kCStages) & 1);
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t kId64 = umma_idesc_bf16(kCM, 64, false);
    constexpr uint32_t kId128 = umma_idesc_bf16(kCM, 128, false);
    const uint64_t q_desc = umma_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t k_desc = umma_desc_sw128(smem_u32(stages), 16, 1024);
    bool ok = true;
    const int nbuf = p.lse_out ? 4 : 2;               // accumulators in rotation
    for (int j = 0; j < n_jobs && ok; ++j) {
      const int s = j % kCStages, g = j % ng, bb = j % nbuf;
      const int size = 2 * g + 1 < np_b ? 2 : 1;
      if (!warp_wait(&S.full[s], (j / kCStages) & 1)) ok = false;
      else if (j >= nbuf && !warp_wait(&S.dfree[bb], ((j - nbuf) / nbuf) & 1)) ok = false;
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint64_t ka = k_desc + ((s * kCStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t qo = q_desc + (((k >> 2) * (kCM * 128) + (k & 3) * 32) >> 4);
          const uint64_t ko = ka + (((k >> 2) * kGBox + (k & 3) * 32) >> 4);
          umma_bf16(tbase + 128 * bb, qo, ko, size == 2 ? kId128 : kId64, k > 0);   // S = Q K^T
        }
        umma_commit(&S.dfull[bb]);
        umma_commit(&S.empty[s]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    if (lane == 0) umma_commit(&S.drain);
    __syncwarp();
    if (!warp_wait(&S.drain, 0) && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
  } else {
    // ================================================================ math warps
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;                 // column group: keys 32 grp .. 32 grp + 31 of the pair
    const int r = quarter * 32 + lane;               // TMEM lane: query row r
    const int t = (warp - 2) * 32 + lane;            // 0 .. 511
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + 32 * grp;
    const float scale = p.scale_log2;
    const int row_min = n - p.alpha + row0;          // position of the chunk's first row
    const int row_pos = row_min + r;                 // position of query row r
    float m = -CUDART_INF_F, l = 0.f, lse2 = CUDART_INF_F;
    if (p.lse_in && r < rows)      // the caller's natural-log LSE in the log2 domain of the scores
      lse2 = p.lse_in[(int64_t(b) * p.alpha + row0 + r) * p.Hq + hq] * 1.4426950408889634f;
    bool ok = true;
    float* srow = p.scores + (int64_t(b) * p.Hq + hq) * (int64_t(p.np_max) * kPageTokens);
    // the four groups' (max, sum) of row r merged into its log-sum-exp, log2 domain (+inf for rows
    // past the chunk or with nothing visible)
    auto merge_lse = [&]() -> float {
      float mm = -CUDART_INF_F;
#pragma unroll
      for (int q = 0; q < kGroups; ++q) mm = fmaxf(mm, S.ml[q][0][r]);
      float ll = 0.f;
#pragma unroll
      for (int q = 0; q < kGroups; ++q) {
        const float mq = S.ml[q][0][r];
        ll += mq == -CUDART_INF_F ? 0.f : S.ml[q][1][r] * fast_exp2(mq - mm);
      }
      return (r < rows && ll > 0.f) ? mm + log2f(ll) : CUDART_INF_F;
    };
    // One 32-key block of row r's scores (keys key0 ..) into its running maximum and sum (log2
    // domain), visible keys only.
    auto absorb = [&](const uint32_t (&sv)[32], int key0) {
      const bool full = key0 + 32 <= min(n, row_min + 1);   // every row of the chunk sees them
      // the row maximum over the visible keys first (raw S; scale > 0), then the sum
      float mx4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mx4[k] = -CUDART_INF_F;
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], __uint_as_float(sv[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int key = key0 + c;
          const bool vis = key < n && key <= row_pos;
          mx4[c & 3] = fmaxf(mx4[c & 3], vis ? __uint_as_float(sv[c]) : -CUDART_INF_F);
        }
      }
      const float mb = scale * fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_new = fmaxf(m, mb);
      if (m_new == -CUDART_INF_F) return;             // nothing visible yet
      float ls4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) ls4[k] = 0.f;
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {   // column pairs in packed f32x2 form
          float e0, e1;
          fma_f32x2(e0, e1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), scale, scale, -m_new, -m_new);
          add_f32x2(ls4[c & 3], ls4[(c + 1) & 3], fast_exp2(e0), fast_exp2(e1));   // c even: neighbouring sums
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int key = key0 + c;
          const bool vis = key < n && key <= row_pos;
          ls4[c & 3] += vis ? fast_exp2(fmaf(__uint_as_float(sv[c]), scale, -m_new)) : 0.f;
        }
      }
      l = l * fast_exp2(m - m_new) +                  // m = -inf gives 0
          ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
      m = m_new;
    };
    if (p.lse_out) {
      // LSE-only: group grp takes the pairs j with j % 4 == grp (accumulator grp), a thread all 128
      // keys of its row in each, 32 columns per tensor-memory wait, so the four groups work on
      // different pairs (one warp's load overlaps another's arithmetic)
      const uint32_t gaddr = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + 128 * grp;
      for (int j = grp; j < n_jobs; j += 4) {
        if (!warp_wait(&S.dfull[grp], (j >> 2) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kb = 2 * j * kPageTokens;           // the pair's first key
        const int rounds = min(4, max(0, (n - kb + 31) / 32));
        if (rounds == 0) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.dfree[grp]);
        }
        for (int rd = 0; rd < rounds; ++rd) {
          uint32_t sv[32];
          tmem_ld32(gaddr + 32 * rd, sv);
          tmem_wait_ld();
          if (rd == rounds - 1) {                     // this warp's last read of the accumulator
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.dfree[grp]);
          }
          absorb(sv, kb + 32 * rd);
        }
      }
    }
    for (int j = 0; j < (p.lse_out ? 0 : n_jobs); ++j) {
      const int g = j % ng, bb = j & 1;
      const bool pass2 = j >= p1;
      const int key0 = 2 * g * kPageTokens + 32 * grp;   // position of this warp's first key
      const bool live = key0 < n;                        // the pair's tail may lie past the prompt
      if (p1 > 0 && j == p1) {                           // pass 1 done: publish this group's (max, sum)
        S.ml[grp][0][r] = m;
        S.ml[grp][1][r] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.mlready);
      }
      // warps meet only through mbarriers, whose waits are bounded: a warp that gives up leaves alone
      bool got = warp_wait(&S.dfull[bb], (j >> 1) & 1);
      if (p1 > 0 && j == p1) got = warp_wait(&S.mlready, 0) && got;
      if (!got) {
        ok = false;
        break;
      }
      if (p1 > 0 && j == p1) lse2 = merge_lse();
      tc_fence_after();
      uint32_t sv[32];
      if (live) {
        tmem_ld32(lane_addr + 128 * bb, sv);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dfree[bb]);        // this warp's TMEM reads are done
      // every row of the chunk sees every key of this group (all but the causal tail)
      const bool full = key0 + 32 <= min(n, row_min + 1);
      if (!pass2) {
        if (live) absorb(sv, key0);
      } else {
        // row r's probabilities of these keys, summed over the warp's 32 rows by a butterfly:
        // each step keeps half of the columns (the half named by one lane bit) and adds the
        // partner lane's copy of them, so after five steps lane l holds key key0 + l
        if (live) {
          float v[32];                                     // rows past the chunk have lse2 = +inf
          if (full) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {   // column pairs in packed f32x2 form
              float e0, e1;
              fma_f32x2(e0, e1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), scale, scale, -lse2, -lse2);
              v[c] = fast_exp2(e0);
              v[c + 1] = fast_exp2(e1);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int key = key0 + c;
              const bool vis = key < n && key <= row_pos;
              const float e = fast_exp2(fmaf(__uint_as_float(sv[c]), scale, -lse2));
              v[c] = vis ? e : 0.f;
            }
          }
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) {              // w = values kept after this step
            const bool hi = (lane & w) != 0;
#pragma unroll
            for (int k = 0; k < w; ++k) {
              const float send = hi ? v[k] : v[k + w];
              const float keep = hi ? v[k + w] : v[k];
              v[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
          }
          const int slot = j % 3;
          S.part[slot][quarter][32 * grp + lane] = v[0];
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            __threadfence_block();                       // the partial sums before the count
            last = atomicAdd(&S.cnt[slot][grp], 1) == 3;
          }
          if (__shfl_sync(0xffffffffu, last, 0)) {      // the group's last warp adds the four quarters
            __threadfence_block();
            const int cc = 32 * grp + lane;
            const float sum = (S.part[slot][0][cc] + S.part[slot][1][cc]) + (S.part[slot][2][cc] + S.part[slot][3][cc]);
            const int key = key0 + lane;                 // keys from n on are zeroed below
            if (key < n) {
              if (in_grid) atomicAdd(&srow[key], sum);
              else srow[key] = p.accumulate ? srow[key] + sum : sum;
            }
            __syncwarp();
            if (lane == 0) S.cnt[slot][grp] = 0;        // reused three jobs later
          }
        }
      }
    }
    if (p.lse_out) {
      // pass 1 alone: each row's log-sum-exp (log2 domain) for a later probability pass
      S.ml[grp][0][r] = m;
      S.ml[grp][1][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.mlready);
      if (!warp_wait(&S.mlready, 0)) ok = false;
      else if (grp == 0 && r < rows) p.lse_out[(int64_t(b) * p.alpha + row0 + r) * p.Hq + hq] = merge_lse();
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    // positions from the prompt's end on (all of them for a rejected request) are zero
    if (!p.accumulate && !in_grid && !p.lse_out)
      for (int i = (valid_req ? n : 0) + t; i < p.np_max * kPageTokens; i += kMathThreads) srow[i] = 0.f;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Given-LSE form with the product turned around: S^T = K Q^T, the keys of a page pair as M (128
// TMEM lanes) and up to 256 window rows as N (TMEM columns).  A thread then owns one key and sums
// its probabilities over the rows in its own registers: per score one fused multiply-add, one exp2
// and one add, with no cross-lane reduction.  Both operands are the same K-major 128-byte-swizzled
// tiles as above, K from the paged pool by TMA and the window rows by one 4-D TMA load per
// (request, query head).  Every MMA is M 128 x N 256 (a pair with one page leaves lanes 64..127
// holding keys past the prompt, which are never read).
//
// Persistent: the (request, query head, page pair) tiles of all requests form one sequence (a
// table of per-request tile offsets in shared memory); CTA c takes a contiguous range of it, so
// the query heads of one kv head (the same pages) run side by side on neighbouring CTAs.  A tile's
// column sums are complete within the CTA (all the launch's rows are in one N 256 tile): the
// scores are plain stores (no atomic adds), bit-reproducible.  Eighteen warps:
//   warp 0     TMA producer: the page pairs into a 4-stage ring; each (request, head)'s rows' LSE
//              (log2 domain) into one of two shared buffers;
//   warp 1     MMA issuer: loads the window rows of each (request, head) once every MMA reading
//              the previous ones has completed, then 8 MMAs per pair into one of two 256-column
//              TMEM accumulators;
//   warps 2-17 two groups of eight, group q taking the pairs j with j % 2 == q (accumulator q),
//              each group one warp per (TMEM lane quarter: 32 keys, half of the rows: 128): a
//              thread reads its key's scores for its rows 32 columns at a time and sums them in a
//              fixed order; the two halves' sums meet in shared memory and the second to finish
//              adds them.  Four warps share each SM sub-partition, on two pairs in different
//              phases, so one computes while another waits for its tensor-memory load (a warp's
//              wait covers all its outstanding loads, so it cannot overlap its own).
constexpr int kTRows = 256;                       // window rows per launch (N)
constexpr int kTStages = 4;
constexpr int kTThreads = 576;
constexpr int kTMathWarps = 16;
constexpr int kRoundCols = 32;                    // TMEM columns a math thread reads per wait
constexpr int kTMaxB = 4096;                      // requests per launch (the tile table)
constexpr int kTQBytes = 2 * kTRows * 128;        // the rows' two 64-dim halves
constexpr uint32_t kTTmemCols = 512;              // two 256-column accumulators

struct ColTSmem {
  uint64_t full[kTStages], empty[kTStages];
  uint64_t dfull[2], dfree[2];
  uint64_t qfull, qfree;
  uint64_t lfull[2], lfree[2];
  uint64_t drain;
  uint32_t tmem_base;
  int scan[kTThreads / 32];
  alignas(16) float lse[2][kTRows];               // log2-domain LSE of each row, +inf past the chunk (read as float4)
  float part[2][3][2][128];                       // [group][slot][row half][key]: each half's sums
  int cnt[2][3][4];                               // [group][slot][lane quarter]: halves done
  int tile_pre[kTMaxB + 1];                       // Hq x (page pairs of the requests before b)
};

constexpr size_t kColTSmem = 1024 + kTQBytes + size_t(kTStages) * kCStageBytes + sizeof(ColTSmem);
static_assert(kColTSmem <= 232448, "column-score (given LSE) shared memory exceeds the per-CTA limit");
static_assert(offsetof(ColTSmem, lse) % 16 == 0, "the LSE rows are read as 16-byte vectors");

// Position in the tile sequence: request b, query head hq, pair g of the request's tb pairs.
struct TileWalk {
  int b = 0, hq = 0, g = 0, tb = 0;
  __device__ void start(const int* pre, int B, int Hq, int x) {
    int lo = 0, hi = B;                           // the last b with pre[b] <= x (then pre[b + 1] > x)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= x) lo = mid;
      else hi = mid;
    }
    b = lo;
    tb = (pre[b + 1] - pre[b]) / Hq;
    const int off = x - pre[b];
    hq = off / tb;
    g = off % tb;
  }
  __device__ void next(const int* pre, int B, int Hq) {
    if (++g < tb) return;
    g = 0;
    if (++hq < Hq) return;
    hq = 0;
    do {
      ++b;
    } while (b < B && pre[b + 1] == pre[b]);
    tb = b < B ? (pre[b + 1] - pre[b]) / Hq : 0;
  }
  // The page pair of step g: odd query heads take the request's pairs last to first, so a CTA that
  // moves on to the next head of the same kv head starts on the pages it read most recently (still
  // in L2).
  __device__ int pair() const { return (hq & 1) ? tb - 1 - g : g; }
};

__device__ __forceinline__ int request_pairs(const ColScoreParams& p, int b) {
  const int n = p.seq_len[b];
  if (n < p.alpha || n > p.np_max * kPageTokens) return 0;
  return ((n + kPageTokens - 1) / kPageTokens + 1) / 2;
}

// Sum over 32 rows (columns cb .. cb + 31 of this thread's key) of 2^(s scale - lse), rows before
// `thr` excluded (they precede the key).
__device__ __forceinline__ float key_rows_sum(const uint32_t (&sv)[32], const float* lse, int cb, int thr,
                                              float scale) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (thr <= cb) {
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const float4 l = *reinterpret_cast<const float4*>(lse + cb + c);
      float e0, e1, e2, e3;
      fma_f32x2(e0, e1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), scale, scale, -l.x, -l.y);
      fma_f32x2(e2, e3, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]), scale, scale, -l.z, -l.w);
      add_f32x2(a0, a1, fast_exp2(e0), fast_exp2(e1));
      add_f32x2(a2, a3, fast_exp2(e2), fast_exp2(e3));
    }
  } else if (thr < cb + 32) {
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const float4 l = *reinterpret_cast<const float4*>(lse + cb + c);
      const float lv[4] = {l.x, l.y, l.z, l.w};
      float e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        e[i] = cb + c + i >= thr ? fast_exp2(fmaf(__uint_as_float(sv[c + i]), scale, -lv[i])) : 0.f;
      add_f32x2(a0, a1, e[0], e[1]);
      add_f32x2(a2, a3, e[2], e[3]);
    }
  }
  return (a0 + a1) + (a2 + a3);
}

__global__ void __launch_bounds__(kTThreads, 1)
    colscore_lse_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ ColScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* stages = base + kTQBytes;
  ColTSmem& S = *reinterpret_cast<ColTSmem*>(stages + kTStages * kCStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.dfull[i], 1);
      mbar_init(&S.dfree[i], kTMathWarps / 2);   // the eight warps of group i
      mbar_init(&S.lfull[i], 32);
      mbar_init(&S.lfree[i], kTMathWarps);
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qfree, 1);
    mbar_init(&S.drain, 1);
    for (int i = 0; i < 2 * 3 * 4; ++i) (&S.cnt[0][0][0])[i] = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmq);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTTmemCols);
    tmem_relinquish();
  }
  pdl_wait();
  // tile table: tile_pre[b] = Hq x (page pairs of requests 0 .. b - 1), one slice of requests per thread
  {
    const int per = (p.B + kTThreads - 1) / kTThreads;
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const int t = request_pairs(p, b);
      if (t == 0 && blockIdx.x == 0) flag_error(p.err, SPKV_DEVERR_PAGE_ID);
      sum += p.Hq * t;
    }
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) S.scan[warp] = x;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += S.scan[w];
    int acc = wbase + x - sum;
    for (int b = b0; b < b1; ++b) {
      S.tile_pre[b] = acc;
      acc += p.Hq * request_pairs(p, b);
    }
    if (tid == kTThreads - 1) S.tile_pre[p.B] = wbase + x;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem_base;
  const int X = S.tile_pre[p.B];
  const int x0 = static_cast<int>(int64_t(blockIdx.x) * X / gridDim.x);
  const int x1 = static_cast<int>(int64_t(blockIdx.x + 1) * X / gridDim.x);
  const int njobs = x1 - x0;

  if (warp == 0) {
    // ================================================================ TMA producer
    const uint64_t pol = l2_policy_evict_last();   // the kv head's other query heads read the same pages
    TileWalk w;
    if (njobs > 0) w.start(S.tile_pre, p.B, p.Hq, x0);
    int k = -1, j = 0, np_b = 0;
    bool ok = true;
    for (; j < njobs; ++j, w.next(S.tile_pre, p.B, p.Hq)) {
      if (j == 0 || w.g == 0) {
        ++k;
        np_b = (p.seq_len[w.b] + kPageTokens - 1) / kPageTokens;
        if (k >= 2 && !warp_wait(&S.lfree[k & 1], ((k - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        for (int i = lane; i < kTRows; i += 32)
          S.lse[k & 1][i] = i < p.rows ? p.lse_in[(int64_t(w.b) * p.alpha + p.row0 + i) * p.Hq + w.hq] *
                                             (p.lse_is_log2 ? 1.f : 1.4426950408889634f)
                                       : CUDART_INF_F;
        mbar_arrive(&S.lfull[k & 1]);
      }
      const int s = j % kTStages;
      if (j >= kTStages && !warp_wait(&S.empty[s], ((j / kTStages) - 1) & 1)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        uint32_t bytes = 0;
        int ph[2] = {-1, -1};
        for (int q = 0; q < 2; ++q) {
          const int pg = 2 * w.pair() + q;
          if (pg >= np_b) continue;
          const int v = p.page_table[int64_t(w.b) * p.np_max + pg];
          if (v < 0 || v >= p.n_phys) {
            flag_error(p.err, SPKV_DEVERR_PHYS);
            continue;
          }
          ph[q] = v;
          bytes += 2 * kBox;
        }
        uint8_t* st = stages + s * kCStageBytes;
        const int h = w.hq / p.G;
        if (bytes) {
          mbar_arrive_expect_tx(&S.full[s], bytes);
          for (int q = 0; q < 2; ++q) {
            if (ph[q] < 0) continue;
            const int z = static_cast<int>(int64_t(h) * p.n_phys + ph[q]);
            tma_load_3d(st + q * kBox, &tmk, &S.full[s], 0, 0, z, pol);
            tma_load_3d(st + kGBox + q * kBox, &tmk, &S.full[s], 64, 0, z, pol);
          }
        } else {
          mbar_arrive(&S.full[s]);
        }
      }
      __syncwarp();
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    for (int i = j > kTStages ? j - kTStages : 0; i < j; ++i) mbar_wait(&S.full[i % kTStages], (i / kTStages) & 1);
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t kId = umma_idesc_bf16(128, kTRows, false);   // M = keys, N = rows
    const uint64_t q_desc = umma_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t k_desc = umma_desc_sw128(smem_u32(stages), 16, 1024);
    const uint64_t qpol = l2_policy_evict_first();
    TileWalk w;
    if (njobs > 0) w.start(S.tile_pre, p.B, p.Hq, x0);
    int k = -1;
    bool ok = true, q_pending = false;
    for (int j = 0; j < njobs && ok; ++j, w.next(S.tile_pre, p.B, p.Hq)) {
      if (j == 0 || w.g == 0) {
        ++k;
        if (k >= 1) {   // every MMA reading the previous rows completes before they are replaced
          if (lane == 0) umma_commit(&S.qfree);
          __syncwarp();
          if (!warp_wait(&S.qfree, (k - 1) & 1)) {
            ok = false;
            break;
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&S.qfull, kTQBytes);
          tma_load_4d(sQ, &tmq, &S.qfull, 0, w.hq, p.row0, w.b, qpol);
          tma_load_4d(sQ + kTQBytes / 2, &tmq, &S.qfull, 64, w.hq, p.row0, w.b, qpol);
        }
        q_pending = true;
        __syncwarp();
        if (!warp_wait(&S.qfull, k & 1)) {
          ok = false;
          break;
        }
        q_pending = false;
      }
      const int s = j % kTStages, bb = j & 1;
      if (!warp_wait(&S.full[s], (j / kTStages) & 1)) ok = false;
      else if (j >= 2 && !warp_wait(&S.dfree[bb], ((j - 2) >> 1) & 1)) ok = false;
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint64_t ka = k_desc + ((s * kCStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ko = ka + (((kk >> 2) * kGBox + (kk & 3) * 32) >> 4);
          const uint64_t qo = q_desc + (((kk >> 2) * (kTQBytes / 2) + (kk & 3) * 32) >> 4);
          umma_bf16(tbase + kTRows * bb, ko, qo, kId, kk > 0);   // S^T = K Q^T
        }
        umma_commit(&S.empty[s]);
        umma_commit(&S.dfull[bb]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    if (q_pending) mbar_wait(&S.qfull, k & 1);     // a row copy in flight lands before the CTA leaves
    if (lane == 0) umma_commit(&S.drain);
    __syncwarp();
    if (!warp_wait(&S.drain, 0) && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
  } else {
    // ================================================================ math warps
    const int mw = warp - 2;                       // 0 .. 15
    const int quarter = warp & 3;                  // TMEM lanes 32 quarter .. (keys of the pair)
    const int grp = mw >> 3;                       // pairs j with j % 2 == grp (accumulator grp)
    const int half = (mw >> 2) & 1;                // rows 128 half .. 128 half + 127
    const int kt = 32 * quarter + lane;            // this thread's key within the pair
    const int cb = 128 * half;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + kTRows * grp + cb;
    const float scale = p.scale_log2;
    const int rounds = min(128, max(0, p.rows - cb) + kRoundCols - 1) / kRoundCols;   // rounds holding rows
    TileWalk w;
    if (njobs > 0) w.start(S.tile_pre, p.B, p.Hq, x0);
    int k = -1, n = 0, first_pos = 0;
    float* srow = p.scores;
    bool ok = true;
    for (int j = 0; j < njobs; ++j, w.next(S.tile_pre, p.B, p.Hq)) {
      if (j == 0 || w.g == 0) {                    // every warp follows every (request, head) switch
        if (k >= 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.lfree[k & 1]);
        }
        ++k;
        if (!warp_wait(&S.lfull[k & 1], (k >> 1) & 1)) {
          ok = false;
          break;
        }
        n = p.seq_len[w.b];
        first_pos = n - p.alpha + p.row0;           // position of the launch's first row
        srow = p.scores + (int64_t(w.b) * p.Hq + w.hq) * (int64_t(p.np_max) * kPageTokens);
      }
      if ((j & 1) != grp) continue;
      if (!warp_wait(&S.dfull[grp], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key = 2 * w.pair() * kPageTokens + kt;
      const int thr = key - first_pos;             // rows before thr precede the key
      const float* lse = S.lse[k & 1];
      float sum = 0.f;
      if (rounds == 0) {                           // no rows of this launch in this half
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.dfree[grp]);
      }
      for (int rd = 0; rd < rounds; ++rd) {
        uint32_t sv[kRoundCols / 32][32];
#pragma unroll
        for (int i = 0; i < kRoundCols / 32; ++i) tmem_ld32(lane_addr + kRoundCols * rd + 32 * i, sv[i]);
        tmem_wait_ld();
        if (rd == rounds - 1) {                    // this warp's last read of the accumulator
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.dfree[grp]);
        }
        if (key < n) {
#pragma unroll
          for (int i = 0; i < kRoundCols / 32; ++i) sum += key_rows_sum(sv[i], lse, cb + kRoundCols * rd + 32 * i, thr, scale);
        }
      }
      // the two halves' sums of a key meet in shared memory; the second to arrive adds them in
      // order and stores the score
      const int slot = (j >> 1) % 3;
      S.part[grp][slot][half][kt] = sum;
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();                     // the partial sums before the count
        last = atomicAdd(&S.cnt[grp][slot][quarter], 1) == 1;
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence_block();
        const float tot = S.part[grp][slot][0][kt] + S.part[grp][slot][1][kt];
        if (key < n) srow[key] = p.accumulate ? srow[key] + tot : tot;
        else if (!p.accumulate && key < p.np_max * kPageTokens) srow[key] = 0.f;
        __syncwarp();
        if (lane == 0) S.cnt[grp][slot][quarter] = 0;   // reused three of the group's pairs later
      }
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    // positions past each (request, head)'s last pair (all of a rejected request's) are zero
    if (!p.accumulate) {
      const int t = tid - 64;
      for (int u = blockIdx.x; u < p.B * p.Hq; u += gridDim.x) {
        const int b = u / p.Hq;
        const int from = 2 * kPageTokens * ((S.tile_pre[b + 1] - S.tile_pre[b]) / p.Hq);
        float* row = p.scores + int64_t(u) * (int64_t(p.np_max) * kPageTokens);
        for (int i = from + t; i < p.np_max * kPageTokens; i += kTMathWarps * 32) row[i] = 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTTmemCols);
  }
}

}  // namespace

cudaError_t colscore_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(colscore_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kColSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(colscore_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kColTSmem));
}

int colscore_lse_max_requests() { return kTMaxB; }

cudaError_t launch_colscore_lse(const spkv_cache* c, const ColScoreParams& p, const CUtensorMap& tmq, int grid,
                                cudaStream_t st) {
  return launch_pdl(colscore_lse_kernel, dim3(grid), dim3(kTThreads), kColTSmem, st, c->tmap_k, tmq, p);
}

cudaError_t launch_colscore(const spkv_cache* c, const ColScoreParams& p, cudaStream_t st) {
  return launch_pdl(colscore_kernel, dim3(p.Hq, p.B, p.chunks_in_grid > 1 ? p.chunks_in_grid : 1), dim3(kCThreads),
                    kColSmem, st, c->tmap_k, p);
}

}  // namespace spkv
