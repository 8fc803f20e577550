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
// One CTA per (request b, query head hq); the alpha (<= 128) rows are one M 128 tile.  Six warps:
//   warp 0     TMA producer: the K rows of two consecutive pages (two 64 x 64 bf16 boxes each,
//              128-byte swizzle, stacked into 128-row tiles) into a 3-stage ring, once for each
//              pass;
//   warp 1     MMA issuer (one thread): S = Q K^T (M 128 query rows, N 64 or 128 keys) into one
//              of two TMEM buffers, in both passes; a stage is released as soon as its MMA
//              completes (V is never needed);
//   warps 2-5  thread r owns query row r (TMEM lane r).  Pass 1 keeps its causal row maximum and
//              sum in the log2 domain (the row log-sum-exp).  Pass 2 turns its S row into
//              probabilities 2^(s scale - lse) and writes them to a padded fp32 tile in shared
//              memory; then thread r sums column r of that tile (key r of the pair) over the
//              alpha rows -- the page's k-major loop order, with the transpose done in shared
//              memory.
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace spkv {
namespace {

constexpr int kCM = 128;                    // tile rows: the window's query rows
constexpr int kCStages = 3;
constexpr int kPRow = kCM + 1;              // padded row of the probability tile (conflict-free)
constexpr int kCThreads = 192;
constexpr int kBox = 64 * 128;              // one page's 64 rows x 128 B (one d-half)
constexpr int kGBox = 2 * kBox;             // two pages' rows of one d-half
constexpr int kCStageBytes = 2 * kGBox;     // K half 0, K half 1 of a page pair
constexpr int kQBytes = 2 * kCM * 128;
constexpr uint32_t kTmemCols = 256;         // two 128-column buffers

struct ColSmem {
  uint64_t full[kCStages], empty[kCStages];
  uint64_t dfull[2], dfree[2];
  uint64_t drain;
  uint32_t tmem_base;
  float prob[kCM * kPRow];                  // pass 2: probabilities [query row][key], padded rows
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
  const int h = hq / p.G;

  if (tid == 0) {
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.dfull[i], 1);
      mbar_init(&S.dfree[i], 4);
    }
    mbar_init(&S.drain, 1);
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
    if (r < p.alpha) v = *reinterpret_cast<const uint4*>(p.q + ((int64_t(b) * p.alpha + r) * p.Hq + hq) * kHeadDim + 8 * c);
    *reinterpret_cast<uint4*>(sQ + (c >> 3) * (kCM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem_base;
  const bool valid_req = n >= p.alpha && n <= p.np_max * kPageTokens;
  const int ng = valid_req ? (np_b + 1) / 2 : 0;   // page pairs
  const int n_jobs = 2 * ng;                       // pass 1, then pass 2

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
    for (int j = 0; j < n_jobs && ok; ++j) {
      const int s = j % kCStages, g = j % ng, bb = j & 1;
      const int size = 2 * g + 1 < np_b ? 2 : 1;
      if (!warp_wait(&S.full[s], (j / kCStages) & 1)) ok = false;
      else if (j >= 2 && !warp_wait(&S.dfree[bb], ((j - 2) >> 1) & 1)) ok = false;
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
    const int r = quarter * 32 + lane;               // TMEM lane: query row r
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float scale = p.scale_log2;
    const int row_pos = n - p.alpha + r;             // position of query row r
    float m = -CUDART_INF_F, l = 0.f, lse2 = CUDART_INF_F;
    bool ok = true;
    float* srow = p.scores + (int64_t(b) * p.Hq + hq) * (int64_t(p.np_max) * kPageTokens);
    for (int j = 0; j < n_jobs; ++j) {
      const int g = j % ng, bb = j & 1;
      const bool pass2 = j >= ng;
      const int size = 2 * g + 1 < np_b ? 2 : 1;
      const int key0 = 2 * g * kPageTokens;          // position of the pair's first key
      const int ncol = 64 * size;
      if (j == ng) lse2 = (r < p.alpha && l > 0.f) ? m + log2f(l) : CUDART_INF_F;   // pass 1 done
      // all four math warps leave together (pass 2 synchronises them on a named barrier)
      if (!named_bar_and(1, 128, warp_wait(&S.dfull[bb], (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float ls8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls8[k] = 0.f;
      if (!pass2) {
        // the row maximum over the visible keys of this pair first, then the sum
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -CUDART_INF_F;
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          uint32_t sv[32];
          tmem_ld32(lane_addr + 128 * bb + c0, sv);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int key = key0 + c0 + c;
            const bool vis = key < n && key <= row_pos;
            mx8[c & 7] = fmaxf(mx8[c & 7], vis ? __uint_as_float(sv[c]) * scale : -CUDART_INF_F);
          }
        }
        const float mb = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_new = fmaxf(m, mb);
        if (m_new != -CUDART_INF_F) {
          l *= fast_exp2(m - m_new);   // m = -inf gives 0
          m = m_new;
        }
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          uint32_t sv[32];
          tmem_ld32(lane_addr + 128 * bb + c0, sv);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int key = key0 + c0 + c;
            const bool vis = key < n && key <= row_pos && m != -CUDART_INF_F;
            ls8[c & 7] += vis ? fast_exp2(fmaf(__uint_as_float(sv[c]), scale, -m)) : 0.f;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.dfree[bb]);
        l += ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
      } else {
        // row r's probabilities of this pair into row r of the shared tile ...
        float* prow = S.prob + r * kPRow;
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          uint32_t sv[32];
          tmem_ld32(lane_addr + 128 * bb + c0, sv);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int key = key0 + c0 + c;
            const bool vis = key < n && key <= row_pos;   // rows >= alpha have lse2 = +inf
            const float e = fast_exp2(fmaf(__uint_as_float(sv[c]), scale, -lse2));
            prow[c0 + c] = vis ? e : 0.f;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.dfree[bb]);
        named_bar_sync(1, 128);
        // ... then thread r sums column r (key key0 + r) over the alpha rows
        if (r < ncol) {
#pragma unroll 8
          for (int row = 0; row < p.alpha; ++row) ls8[row & 7] += S.prob[row * kPRow + r];
          const float sum = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
          const int key = key0 + r;
          srow[key] = key < n ? sum : 0.f;
        }
        named_bar_sync(1, 128);   // the tile is rewritten by the next pair
      }
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    // positions past the request's pages (all of them for a rejected request) are zero
    for (int i = (valid_req ? np_b * kPageTokens : 0) + r; i < p.np_max * kPageTokens; i += kCM) srow[i] = 0.f;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t colscore_init_attributes() {
  return cudaFuncSetAttribute(colscore_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kColSmem));
}

cudaError_t launch_colscore(const spkv_cache* c, const ColScoreParams& p, cudaStream_t st) {
  return launch_pdl(colscore_kernel, dim3(p.Hq, p.B), dim3(kCThreads), kColSmem, st, c->tmap_k, p);
}

}  // namespace spkv
