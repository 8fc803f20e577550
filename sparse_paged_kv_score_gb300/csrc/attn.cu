// Split-K flash decoding over a list of KV pages per (request, kv head) unit, in two forms:
//   sparse : the page list is a selected subset (logical page ids -> page table), plain scores
//   lazy   : the page list is packed page words; the query is rotated with RoPE by the offset
//            between the query position and the page's document, once per document switch
//
// Computation: [FA] "How KV sparsity achieves 1.5x acceleration for vLLM", section "2. Attention
// modification": one pass over KV blocks with a running max, a running sum l and an output
// accumulator, O / l at the end; rowmax and l are kept and returned as LSE.  Lazy form:
// [LazyAttention] "Technical implementation 2. Decoding" and "Mathematical equivalence".
//
// GB300 design (one CTA per SM, persistent, six warps):
//   * Work balance: the pages of all units form one sequence of T pages.  Each CTA first streams
//     a static range (75% of the pages split evenly), then takes small chunks of the remaining
//     25% from an atomic counter, so SMs that stream faster take more and all finish together.
//     Static ranges and chunks ("segments") are numbered in page order; a unit split over
//     several segments leaves one fp32 partial (max, sum, unnormalised O) per segment in a
//     workspace slot (unit + segment), and a small second kernel (one CTA per unit, launched
//     with programmatic dependent launch) merges them and resets the chunk counter.
//   * Producer warp: streams each page's K and V (2 x 16 KiB, head-major, one contiguous page
//     each) with TMA tensor loads (128B swizzle) into a ring of shared-memory stages, and with
//     the first page of each unit a bulk copy of that unit's query rows; all complete on the
//     stage's mbarrier.  Consumers release stages on a second mbarrier.
//   * Four consumer warps each take 16 of the 64 tokens of every page.  Q.K^T runs on
//     mma.sync m16n8k16 with the 16 keys as M and the GQA group (padded to 8) as N, so the
//     group of query heads shares one tensor-core tile; P^T goes from the accumulator layout to
//     the B-operand layout with movmatrix; P.V runs with V^T (ldmatrix.trans) as A.  P (and the
//     rotated lazy query) is split into bf16 hi + lo parts so the weights keep ~17 bits.
//   * Epilogue warp: at each segment switch the consumers hand their (max, sum, O) to a shared
//     buffer and go on streaming; the epilogue warp merges the four states and writes the
//     output (unit within one segment) or the segment's partial, off the consumers' critical path.
//   * Launched with programmatic dependent launch: barrier set-up overlaps the previous kernel;
//     griddepcontrol.wait precedes the first read of its outputs.
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace spkv {
namespace {

constexpr int kBoxBytes = 8192;                // 64 tokens x 64 dims x bf16
constexpr int kKVBytes = 4 * kBoxBytes;        // K (2 boxes) + V (2 boxes) of one page-head
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDocRows = 16;                   // query rows of a document-major job

// Warps: kCons consumers, then the producer warp and the epilogue warp.  The document-major form
// runs two groups of four consumers over each page, one group per 8 of the job's 16 query rows, so
// every SM sub-partition has two consumer warps to switch between.
template <bool DOCS>
struct Cfg {
  static constexpr int kCons = DOCS ? 8 : 4;
  static constexpr int kThreads = (kCons + 2) * 32;
};
constexpr int kThreads = Cfg<false>::kThreads;

// Stage: K/V page image, then room for the query rows of the unit it starts.
template <int NT, bool DOCS = false>
__host__ __device__ constexpr int stage_bytes() { return kKVBytes + (DOCS ? kDocRows : NT * 8) * kHeadDim * 2; }

constexpr int kEnd = -2;   // StageMeta.unit of the stage that ends the CTA's page stream
constexpr int kMaxUnits = 4096;   // (request, kv head) units per call

struct __align__(16) StageMeta {
  int unit;     // unit of this page (-1: none, kEnd: no more pages)
  int valid;    // valid tokens (0 = skip the page)
  int rel;      // lazy: query position - document offset
  int ustart;   // position of the unit's first page in the global page sequence
  int ucount;   // pages of the unit
  int chunk;    // chunk of the global page sequence this page belongs to
  int pad0, pad1;
};

template <int NT, int KC, int NPREFIX = kMaxUnits + 1>
struct Smem {
  static constexpr int kG = NT * 8;
  // hand-off buffer from the consumer warps to the epilogue warp
  float cm[KC][kG];
  float cl[KC][kG];
  float co[KC][kG][kHeadDim + 4];   // rows padded: the consumers' stores are conflict-free
  int h_unit, h_chunk, h_ustart, h_ucount, h_last, h_pad[3];
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t cfull;     // consumers -> epilogue (count: the consumer warps)
  uint64_t cempty;    // epilogue -> consumers (count 1)
  StageMeta meta[8];
  int srel[8][16];          // document-major form: each query row's rotation offset, per stage
  int scan[kThreads];
  int prefix[NPREFIX];         // first global page position of every unit, then T (not used by DOCS)
};

template <int NT, int STAGES, bool DOCS = false>
constexpr size_t smem_bytes() {
  return 1024 /*align slack*/ + size_t(STAGES) * stage_bytes<NT, DOCS>() +
         sizeof(Smem<NT, Cfg<DOCS>::kCons, DOCS ? 1 : kMaxUnits + 1>);
}

__device__ __forceinline__ int unit_count(const AttnParams& p, bool lazy, int u) {
  if (lazy) {
    const int n = p.n_pages[u / p.Hk];
    return n < 0 ? 0 : (n > p.np_max ? p.np_max : n);
  }
  const int n = p.n_sel[u];
  return n < 0 ? 0 : (n > p.sel_stride ? p.sel_stride : n);
}

// Swizzled shared address of the 16-byte chunk `chunk` (0..15 across the 128 dims) of token
// row `row` inside one K or V page image made of two 128B-swizzled 64x64 boxes.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + ((chunk >> 3) * kBoxBytes) + row * 128 + ((((chunk & 7) ^ (row & 7))) << 4);
}

// PACK (groups of at most 4 query heads, NT == 1): the 8 columns of each MMA's query operand
// hold the group's heads twice.  Columns 4..7 carry the bf16 lo part of what columns 0..3 carry
// in hi (the rotated query in the lazy form, the probabilities P), so one MMA does the work of
// the hi MMA and the lo MMA; the halves are added where a full value is needed.
// DOCS (document-major lazy form, LAZY set): a unit is a job of the plan -- one document, one kv
// head and up to 16 / G of the requests that hold the document -- whose query rows (G per request,
// each with its own rotation offset) share every page of the document; jobs come from a queue, are
// never split, and leave one partial (max, sum, O) per query row, merged per request afterwards.
template <int NT, bool LAZY, bool PACK, int STAGES, bool DOCS = false>
__global__ void __launch_bounds__(Cfg<DOCS>::kThreads, 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ AttnParams p) {
  constexpr int kConsumers = Cfg<DOCS>::kCons;
  constexpr int kProducerWarp = kConsumers;
  constexpr int kEpilogueWarp = kConsumers + 1;
  constexpr int kStage = stage_bytes<NT, DOCS>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using SmemT = Smem<NT, kConsumers, DOCS ? 1 : kMaxUnits + 1>;
  SmemT& S = *reinterpret_cast<SmemT*>(stages + size_t(STAGES) * kStage);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = p.B * p.Hk;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumers);
    }
    mbar_init(&S.cfull, kConsumers);
    mbar_init(&S.cempty, 1);
    fence_mbar_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  // No warp touches a barrier before thread 0 has initialised it.
  __syncthreads();
  // The page lists and counts below are written by the previous kernel.  This kernel does not
  // trigger its dependent early: the combine kernel's CTAs would only sit on the SMs while the
  // pages stream (CTA exit triggers it).
  pdl_wait();

  const int N = gridDim.x;
  int T = 0, S0 = 0, D0 = 0, CH = 1, n_chunks = 0;
  if (!DOCS) {
    // ---- 1. unit prefix table: prefix[u] = first global page position of unit u, prefix[U] = T
    const int c0 = static_cast<int>(int64_t(tid) * U / kThreads);
    const int c1 = static_cast<int>(int64_t(tid + 1) * U / kThreads);
    int csum = 0;
    for (int u = c0; u < c1; ++u) csum += unit_count(p, LAZY, u);
    int x = csum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) S.scan[warp] = x;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += S.scan[w];
    {
      int acc = wbase + x - csum;  // exclusive prefix of this thread's slice
      for (int u = c0; u < c1; ++u) {
        S.prefix[u] = acc;
        acc += unit_count(p, LAZY, u);
      }
      if (c1 == U) S.prefix[U] = acc;
    }
    __syncthreads();
    T = S.prefix[U];

    // units with no pages get out = 0, lse = -inf (spread over the CTAs)
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
      if (S.prefix[u + 1] != S.prefix[u]) continue;
      const int b = u / p.Hk, h = u % p.Hk;
      for (int i = tid; i < p.G * kHeadDim; i += kThreads)
        p.out[(int64_t(b) * p.Hq + h * p.G) * kHeadDim + i] = 0.f;
      if (tid < p.G) p.lse[int64_t(b) * p.Hq + h * p.G + tid] = -CUDART_INF_F;
      if (tid == 0) p.ws_parts[2 * u] = p.ws_parts[2 * u + 1] = 0;
    }
    if (T == 0) return;
    // Segments: static ranges of S0 pages (one per CTA, none when they would be shorter than
    // min_chunk), then dynamic chunks of CH pages.  min_chunk bounds the partials of a unit
    // (about 250 at most); the chunk count stays within the workspace (max_chunks - N chunks).
    S0 = static_cast<int>(int64_t(T) * 3 / (4 * int64_t(N)));
    if (S0 < p.min_chunk) S0 = 0;
    D0 = S0 * N;
    const int T_dyn = T - D0;
    CH = max(max((T_dyn + 6 * N - 1) / (6 * N), (T_dyn + p.max_chunks - N - 1) / (p.max_chunks - N)), p.min_chunk);
    n_chunks = (T_dyn + CH - 1) / CH;
  }
  auto seg_of = [&](int x) { return x < D0 ? x / S0 : N + (x - D0) / CH; };
  const int qbytes = p.G * kHeadDim * 2;

  if (warp == kProducerWarp) {
    // ================================================================ producer warp
    const uint64_t pol = l2_policy_evict_first();   // each page is read once per call
    int last_unit = -1, last_chunk = -1, jl = 0;
    bool ok = true;
    // lane 0 keeps the next dynamic chunk index (DOCS: the next job) requested one segment ahead,
    // so the atomic's latency overlaps the streaming of the current segment
    int ahead = 0;
    if (lane == 0 && (DOCS || n_chunks > 0)) ahead = atomicAdd(&p.ws_ctl[0], 1);
    while (DOCS && ok) {
      const int job = __shfl_sync(0xffffffffu, ahead, 0);
      if (job >= p.n_jobs) break;
      if (lane == 0) ahead = atomicAdd(&p.ws_ctl[0], 1);
      const int4 jb = p.jobs[job];              // document, kv head, first occurrence, occurrences
      const int pg0 = p.doc_first[jb.x];
      const int npg = max(0, p.doc_first[jb.x + 1] - pg0);
      const int nrows = jb.w * p.G;
      // lane o < occurrences: occurrence o's request and rotation offset (query position minus
      // the document's placement in that request)
      int ob = 0, orel = 0;
      if (lane < jb.w) {
        const int2 oc = p.occ[jb.z + lane];     // request, document slot
        ob = oc.x;
        orel = p.qpos[oc.x] - p.doc_pos[int64_t(oc.x) * p.max_docs + oc.y];
      }
      const int row_rel = __shfl_sync(0xffffffffu, orel, min(lane / p.G, 31));   // query row = lane
      const int steps = max(npg, 1);            // a document without pages still hands over empty results
      for (int xb = 0; xb < steps && ok; xb += 32) {
        int phys = 0, valid = 0;
        if (xb + lane < npg) {
          const uint32_t w = p.doc_pages[pg0 + xb + lane];
          const int ph = static_cast<int>(w & 0x3FFFFu);
          if (ph >= p.n_phys) flag_error(p.err, SPKV_DEVERR_PHYS);
          else {
            phys = ph;
            valid = static_cast<int>((w >> 18) & 63u) + 1;
          }
        }
        const int cnt = min(32, steps - xb);
        for (int i = 0; i < cnt; ++i, ++jl) {
          const int s = jl % STAGES;
          const int bv = __shfl_sync(0xffffffffu, valid, i);
          const int bp = __shfl_sync(0xffffffffu, phys, i);
          if (jl >= STAGES) {
            if (!__all_sync(0xffffffffu, mbar_wait(&S.empty[s], ((jl / STAGES) - 1) & 1, p.wait_ns))) {
              if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
              ok = false;
              break;
            }
          }
          const bool first = xb + i == 0;
          uint8_t* dst = stages + size_t(s) * kStage;
          if (first && lane < 16) S.srel[s][lane] = row_rel;
          __syncwarp();
          if (lane == 0) {
            StageMeta m;
            m.unit = job;
            m.valid = bv;
            m.rel = xb + i;           // the page's index within the job
            m.ustart = 0;
            m.ucount = npg;
            m.chunk = 0;
            m.pad0 = nrows;
            m.pad1 = 0;
            S.meta[s] = m;
            mbar_arrive_expect_tx(&S.full[s], (bv > 0 ? kKVBytes : 0) + (first ? nrows * kHeadDim * 2 : 0));
          }
          __syncwarp();
          if (first && lane < jb.w)   // the G query rows of occurrence `lane`, one bulk copy each
            bulk_load(dst + kKVBytes + lane * p.G * kHeadDim * 2,
                      static_cast<const uint8_t*>(p.q) + (int64_t(ob) * p.Hq + jb.y * p.G) * (kHeadDim * 2),
                      p.G * kHeadDim * 2, &S.full[s]);
          if (lane == 0 && bv > 0) {
            const int z = static_cast<int>(int64_t(jb.y) * p.n_phys + bp);
            tma_load_3d(dst, &tmk, &S.full[s], 0, 0, z, pol);
            tma_load_3d(dst + kBoxBytes, &tmk, &S.full[s], 64, 0, z, pol);
            tma_load_3d(dst + 2 * kBoxBytes, &tmv, &S.full[s], 0, 0, z, pol);
            tma_load_3d(dst + 3 * kBoxBytes, &tmv, &S.full[s], 64, 0, z, pol);
          }
          __syncwarp();
        }
      }
    }
    for (int it = 0; !DOCS && ok; ++it) {
      int c, x0, x1;   // segment id and its page range
      if (it == 0 && S0 > 0) {
        c = blockIdx.x;
        x0 = blockIdx.x * S0;
        x1 = x0 + S0;
      } else {
        const int k = __shfl_sync(0xffffffffu, ahead, 0);
        if (n_chunks == 0 || k >= n_chunks) break;
        if (lane == 0) ahead = atomicAdd(&p.ws_ctl[0], 1);
        c = N + k;
        x0 = D0 + k * CH;
        x1 = min(T, x0 + CH);
      }
      for (int xb = x0; xb < x1 && ok; xb += 32) {
        const int xpos = xb + lane;
        const bool need = xpos < x1;
        // unit of page position xpos: the last u with prefix[u] <= xpos (skips empty units)
        int my_u = -1, my_k = 0, my_us = 0, my_uc = 0;
        if (need) {
          int lo = 0, hi = U;
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (S.prefix[mid] <= xpos) lo = mid;
            else hi = mid;
          }
          my_u = lo;
          my_us = S.prefix[lo];
          my_uc = S.prefix[lo + 1] - my_us;
          my_k = xpos - my_us;
        }
        int phys = 0, valid = 0, rel = 0, head = 0;
        if (need) {
          const int b = my_u / p.Hk;
          head = my_u % p.Hk;
          uint32_t bad = 0;
          if (!LAZY) {
            const int lp = p.sel[int64_t(my_u) * p.sel_stride + my_k];
            if (lp < 0 || lp >= p.np_max) {
              bad |= SPKV_DEVERR_PAGE_ID;
            } else {
              const int v = min(kPageTokens, p.seq_len[b] - kPageTokens * lp);
              int ph;
              if (p.slot) {
                // resident-slot form: the page sits in slot s of this request's slot range
                const int sl = p.slot[int64_t(my_u) * p.sel_stride + my_k];
                ph = sl >= 0 && sl < p.n_slots ? b * p.n_slots + sl : -1;
                if (ph < 0) bad |= SPKV_DEVERR_SLOT;
              } else {
                ph = page_lookup(p.page_table, p.np_max, p.pd, b, lp);
              }
              if (v <= 0) bad |= SPKV_DEVERR_PAGE_ID;
              else if (ph < 0 || ph >= p.n_phys) bad |= SPKV_DEVERR_PHYS;
              else { phys = ph; valid = v; }
            }
          } else {
            const int mh = p.meta_heads == 1 ? 0 : head;
            const uint32_t w = p.meta[(int64_t(b) * p.meta_heads + mh) * p.np_max + my_k];
            const int ph = static_cast<int>(w & 0x3FFFFu);
            const int v = static_cast<int>((w >> 18) & 63u) + 1;
            const int sl = static_cast<int>(w >> 24);
            if (ph >= p.n_phys) bad |= SPKV_DEVERR_PHYS;
            else if (sl >= p.max_docs) bad |= SPKV_DEVERR_SLOT;
            else {
              phys = ph;
              valid = v;
              rel = p.qpos[b] - p.doc_pos[int64_t(b) * p.max_docs + sl];
            }
          }
          flag_error(p.err, bad);
        }
        const int cnt = min(32, x1 - xb);
        for (int i = 0; i < cnt; ++i, ++jl) {
          const int s = jl % STAGES;
          const int bu = __shfl_sync(0xffffffffu, my_u, i);
          const int bv = __shfl_sync(0xffffffffu, valid, i);
          const int bp = __shfl_sync(0xffffffffu, phys, i);
          const int br = __shfl_sync(0xffffffffu, rel, i);
          const int bs = __shfl_sync(0xffffffffu, my_us, i);
          const int bc = __shfl_sync(0xffffffffu, my_uc, i);
          const int bh = __shfl_sync(0xffffffffu, head, i);
          if (jl >= STAGES) {
            // warp-uniform outcome even if lanes disagree at the time limit
            if (!__all_sync(0xffffffffu, mbar_wait(&S.empty[s], ((jl / STAGES) - 1) & 1, p.wait_ns))) {
              if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
              ok = false;
              break;
            }
          }
          if (lane == 0) {
            StageMeta m;
            m.unit = bu;
            m.valid = bv;
            m.rel = br;
            m.ustart = bs;
            m.ucount = bc;
            m.chunk = c;
            m.pad0 = m.pad1 = 0;
            S.meta[s] = m;
            uint8_t* dst = stages + size_t(s) * kStage;
            const bool new_seg = bu != last_unit || c != last_chunk;
            const uint32_t tx = (bv > 0 ? kKVBytes : 0) + (new_seg ? qbytes : 0);
            mbar_arrive_expect_tx(&S.full[s], tx);
            if (new_seg) {
              const int b = bu / p.Hk, h = bu % p.Hk;
              bulk_load(dst + kKVBytes,
                        static_cast<const uint8_t*>(p.q) + (int64_t(b) * p.Hq + h * p.G) * (kHeadDim * 2),
                        qbytes, &S.full[s]);
            }
            if (bv > 0) {
              const int z = static_cast<int>(int64_t(bh) * p.n_phys + bp);
              tma_load_3d(dst, &tmk, &S.full[s], 0, 0, z, pol);
              tma_load_3d(dst + kBoxBytes, &tmk, &S.full[s], 64, 0, z, pol);
              tma_load_3d(dst + 2 * kBoxBytes, &tmv, &S.full[s], 0, 0, z, pol);
              tma_load_3d(dst + 3 * kBoxBytes, &tmv, &S.full[s], 64, 0, z, pol);
            }
            last_unit = bu;
            last_chunk = c;
          }
          __syncwarp();
        }
      }
    }
    // end of this CTA's page stream
    if (ok) {
      const int s = jl % STAGES;
      bool free_stage = true;
      if (jl >= STAGES)
        free_stage = __all_sync(0xffffffffu, mbar_wait(&S.empty[s], ((jl / STAGES) - 1) & 1, p.wait_ns));
      if (free_stage) {
        if (lane == 0) {
          StageMeta m;
          m.unit = kEnd;
          m.valid = m.rel = m.ustart = m.ucount = m.chunk = m.pad0 = m.pad1 = 0;
          S.meta[s] = m;
          mbar_arrive(&S.full[s]);
        }
        ++jl;
      } else if (lane == 0) {
        flag_error(p.err, SPKV_DEVERR_TIMEOUT);
      }
    }
    // Before leaving, make sure no copy issued by this CTA is still in flight (always with the
    // full limit: the copies themselves complete in microseconds).
    for (int j = jl > STAGES ? jl - STAGES : 0; j < jl; ++j) mbar_wait(&S.full[j % STAGES], (j / STAGES) & 1);
    return;
  }

  if (warp == kEpilogueWarp) {
    // ================================================================ epilogue warp
    for (int k = 0;; ++k) {
      if (!__all_sync(0xffffffffu, mbar_wait(&S.cfull, k & 1, p.wait_ns))) {
        if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
        break;
      }
      const int u = S.h_unit, chunk = S.h_chunk, ustart = S.h_ustart, ucount = S.h_ucount, last = S.h_last;
      if (DOCS && u >= 0) {
        const int4 jb = p.jobs[u];
        for (int g = 0; g < jb.w * p.G; ++g) {
          // row g was handled by the four warps of group g / 8, in their column g % 8
          const int w0 = (g >> 3) * 4, col = g & 7;
          float M = -CUDART_INF_F;
#pragma unroll
          for (int w = 0; w < 4; ++w) M = fmaxf(M, S.cm[w0 + w][col]);
          float fw[4], L = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float mw = S.cm[w0 + w][col];
            fw[w] = mw == -CUDART_INF_F ? 0.f : exp2f(mw - M);
            L += fw[w] * S.cl[w0 + w][col];
          }
          // row of (occurrence, query head of the kv head's group) in the plan's partials
          const int64_t row = int64_t(jb.z + g / p.G) * p.Hq + jb.y * p.G + g % p.G;
#pragma unroll
          for (int i = 0; i < kHeadDim / 32; ++i) {
            const int d = lane + 32 * i;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) acc += fw[w] * S.co[w0 + w][col][d];
            p.part_o[row * kHeadDim + d] = acc;
          }
          if (lane == 0) {
            p.part_m[row] = M;
            p.part_l[row] = L;
          }
        }
      } else if (u >= 0) {
        const int b = u / p.Hk, h = u % p.Hk;
        const int first = seg_of(ustart);
        const int nparts = seg_of(ustart + ucount - 1) - first + 1;
        const int64_t orow = int64_t(b) * p.Hq + h * p.G;
        const int64_t slot = int64_t(u) + chunk;
        for (int g = 0; g < p.G; ++g) {
          float M = -CUDART_INF_F;
#pragma unroll
          for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, S.cm[w][g]);
          float fw[kConsumers], L = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumers; ++w) {
            const float mw = S.cm[w][g];
            fw[w] = mw == -CUDART_INF_F ? 0.f : exp2f(mw - M);
            L += fw[w] * S.cl[w][g];
          }
#pragma unroll
          for (int i = 0; i < kHeadDim / 32; ++i) {
            const int d = lane + 32 * i;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) acc += fw[w] * S.co[w][g][d];
            if (nparts == 1) p.out[(orow + g) * kHeadDim + d] = L > 0.f ? acc / L : 0.f;
            else p.ws_o[(slot * 16 + g) * kHeadDim + d] = acc;
          }
          if (lane == 0) {
            if (nparts == 1) {
              p.lse[orow + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
            } else {
              p.ws_m[slot * 16 + g] = M;
              p.ws_l[slot * 16 + g] = L;
            }
          }
        }
        // the unit's first segment records where the combine kernel finds its partials
        if (lane == 0 && chunk == first) {
          p.ws_parts[2 * u] = first;
          p.ws_parts[2 * u + 1] = nparts;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.cempty);
      if (last) break;
    }
    return;
  }

  // ================================================================== consumer warps
  const int r = lane >> 2, c = lane & 3;
  // tokens t0 .. t0 + 15 of every page; DOCS: consumer group `grp` takes query rows 8 grp .. 8 grp + 7
  const int t0 = (warp & 3) * 16;
  const int grp_row = DOCS ? (warp >> 2) * 8 : 0;
  const float scale = p.scale_log2;

  float m[NT][2], lsum[NT][2];
  float O[8][NT][4];
  uint32_t qh[8][NT][2];                  // B fragments of q (bf16 hi part)
  uint32_t ql[LAZY && !PACK ? 8 : 1][NT][2];   // lazy: bf16 lo part of the rotated query
  uint32_t qraw[LAZY ? 8 : 1][NT][2];     // lazy: unrotated query
  int cur_u = -1, cur_c = -1, cur_us = 0, cur_uc = 0, cur_rel = 0, n_flush = 0;
  int col_rel[NT];                        // rotation offset of each query column (DOCS: per row)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) col_rel[nt] = 0;
  bool have_rel = false;

  auto reset_state = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -CUDART_INF_F;
      lsum[nt][0] = lsum[nt][1] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[j][nt][e] = 0.f;
    }
  };

  // q fragments from the stage's query rows (rows g >= rows read as zero).
  auto load_q = [&](const uint8_t* qs, int rows) {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(qs);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = PACK ? (r & 3) : grp_row + nt * 8 + r;
      const bool live = g < rows;
      const int row = (live ? g : 0) * (kHeadDim / 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t w0 = live ? qw[row + ks * 8 + c] : 0u;
        const uint32_t w1 = live ? qw[row + ks * 8 + c + 4] : 0u;
        if (LAZY) {
          qraw[LAZY ? ks : 0][nt][0] = w0;
          qraw[LAZY ? ks : 0][nt][1] = w1;
        } else {
          qh[ks][nt][0] = w0;
          qh[ks][nt][1] = w1;
        }
      }
    }
  };

  // Lazy form: q_rot = R(rel) q for this thread's 32 dims, split into bf16 hi + lo.  The
  // angle of pair i is rel * theta_i; its fraction of a turn is formed exactly modulo 1 as a
  // 64-bit fixed-point product (phase accumulator), so the angle handed to __sincosf lies in
  // [-pi, pi) with ~1e-9 rad error however large rel * theta_i is.
  auto rotate_q = [&](const int (&rel)[NT]) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sn[2], cs[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 16 * ks + 2 * c + 8 * wi + e;   // pair index: dims i and i + 64
            const uint64_t ph = static_cast<uint64_t>(static_cast<int64_t>(rel[nt])) * p.phase_inc[i];
            const float ang = static_cast<float>(static_cast<int32_t>(ph >> 32)) * 1.4629180792671596e-09f;
            __sincosf(ang, &sn[e], &cs[e]);
          }
          const uint32_t wx = qraw[LAZY ? ks : 0][nt][wi], wy = qraw[LAZY ? ks + 4 : 0][nt][wi];
          const float x0 = bf16lo_to_f32(wx), x1 = bf16hi_to_f32(wx);
          const float y0 = bf16lo_to_f32(wy), y1 = bf16hi_to_f32(wy);
          float xh0, xl0, xh1, xl1, yh0, yl0, yh1, yl1;
          split_bf16(x0 * cs[0] - y0 * sn[0], xh0, xl0);
          split_bf16(x1 * cs[1] - y1 * sn[1], xh1, xl1);
          split_bf16(y0 * cs[0] + x0 * sn[0], yh0, yl0);
          split_bf16(y1 * cs[1] + x1 * sn[1], yh1, yl1);
          if (PACK) {   // columns 0..3 (r < 4) take the hi part, columns 4..7 the lo part
            const bool hi = r < 4;
            qh[ks][nt][wi] = pack_bf16x2(hi ? xh0 : xl0, hi ? xh1 : xl1);
            qh[ks + 4][nt][wi] = pack_bf16x2(hi ? yh0 : yl0, hi ? yh1 : yl1);
          } else {
            qh[ks][nt][wi] = pack_bf16x2(xh0, xh1);
            ql[LAZY && !PACK ? ks : 0][nt][wi] = pack_bf16x2(xl0, xl1);
            qh[ks + 4][nt][wi] = pack_bf16x2(yh0, yh1);
            ql[LAZY && !PACK ? ks + 4 : 0][nt][wi] = pack_bf16x2(yl0, yl1);
          }
        }
      }
    }
  };

  // Hands this warp's state for unit u to the epilogue warp (which merges the four warps).
  auto flush = [&](int u, int chunk, int ustart, int ucount, int last) {
    if (n_flush > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(&S.cempty, (n_flush - 1) & 1, p.wait_ns))) {
        if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
      }
    }
    if (PACK) {   // O = V^T P_hi (columns 0..3) + V^T P_lo (columns 4..7)
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[j][0][e] += __shfl_xor_sync(0xffffffffu, O[j][0][e], 2);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float l = lsum[nt][cc];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (r == 0) {
          S.cm[warp][nt * 8 + 2 * c + cc] = m[nt][cc];
          S.cl[warp][nt * 8 + 2 * c + cc] = l;
        }
      }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          S.co[warp][nt * 8 + 2 * c + (e & 1)][16 * j + r + ((e >> 1) << 3)] = O[j][nt][e];
    if (warp == 0 && lane == 0) {
      S.h_unit = u;
      S.h_chunk = chunk;
      S.h_ustart = ustart;
      S.h_ucount = ucount;
      S.h_last = last;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.cfull);
    ++n_flush;
  };

  const uint32_t stage0 = smem_u32(stages);
  if (DOCS) {
    // Document-major consumers take a job's pages two at a time (the last of an odd count alone,
    // its partner then the same stage with no valid token): one row max, one correction exp and
    // one rescale of O per 32 keys, and four independent Q.K^T chains and eight P.V chains.  The
    // job's query offsets are fixed, so its rotated query is formed once, at the job's start.
    reset_state();
    int cur_job = -1;
    int jl = 0;
    const int krow = t0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int vrow = t0 + (lane & 7) + ((lane >> 4) & 1) * 8;
    const int vsel = (lane >> 3) & 1;
    for (;;) {
      const int s = jl % STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s], (jl / STAGES) & 1, p.wait_ns))) {
        if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
        break;
      }
      const StageMeta mt = S.meta[s];
      if (mt.unit == kEnd) break;
      if (mt.unit != cur_job) {
        if (cur_job >= 0) flush(cur_job, 0, 0, 0, 0);
        cur_job = mt.unit;
        reset_state();
        load_q(stages + size_t(s) * kStage + kKVBytes, mt.pad0);
        col_rel[0] = S.srel[s][grp_row + r];
        rotate_q(col_rel);
      }
      const bool two = mt.rel + 1 < mt.ucount;   // the producer streams a job's pages in order
      const int s2 = two ? (jl + 1) % STAGES : s;
      int v2 = 0;
      if (two) {
        if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s2], ((jl + 1) / STAGES) & 1, p.wait_ns))) {
          if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
          break;
        }
        v2 = S.meta[s2].valid;
      }
      const int vld[2] = {mt.valid, v2};
      if (vld[0] > t0 || vld[1] > t0) {
        const uint32_t kb[2] = {stage0 + s * kStage, stage0 + s2 * kStage};
        // ---- S^T = K q^T for my 16 keys of both pages (even / odd k-steps in separate chains)
        float acc[2][2][4];
#pragma unroll
        for (int pg = 0; pg < 2; ++pg)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[pg][h][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
          for (int pg = 0; pg < 2; ++pg) {
            uint32_t a[4];
            ldsm_x4(swz(kb[pg], krow, 2 * ks + (lane >> 4)), a);
            mma_bf16_16816(acc[pg][ks & 1], a, qh[ks][0][0], qh[ks][0][1]);
            mma_bf16_16816(acc[pg][ks & 1], a, ql[LAZY && !PACK ? ks : 0][0][0],
                           ql[LAZY && !PACK ? ks : 0][0][1]);
          }
        }
        // ---- online softmax (log2 domain) over the 32 keys
        float sv[2][4];
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          const bool ok0 = t0 + r < vld[pg], ok1 = t0 + r + 8 < vld[pg];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x = (acc[pg][0][e] + acc[pg][1][e]) * scale;
            sv[pg][e] = (e < 2 ? ok0 : ok1) ? x : -CUDART_INF_F;
          }
        }
        float pv[2][4];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float mx = fmaxf(fmaxf(sv[0][cc], sv[0][cc + 2]), fmaxf(sv[1][cc], sv[1][cc + 2]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(m[0][cc], mx);   // finite: key t0 of one page is valid
          const float alpha = exp2f(m[0][cc] - mnew);
          m[0][cc] = mnew;
#pragma unroll
          for (int pg = 0; pg < 2; ++pg) {
            pv[pg][cc] = exp2f(sv[pg][cc] - mnew);
            pv[pg][cc + 2] = exp2f(sv[pg][cc + 2] - mnew);
          }
          lsum[0][cc] = lsum[0][cc] * alpha + ((pv[0][cc] + pv[0][cc + 2]) + (pv[1][cc] + pv[1][cc + 2]));
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            O[j][0][cc] *= alpha;
            O[j][0][cc + 2] *= alpha;
          }
        }
        uint32_t bh[2][2], bl[2][2];
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          float h0, l0, h1, l1, h2, l2, h3, l3;
          split_bf16(pv[pg][0], h0, l0);
          split_bf16(pv[pg][1], h1, l1);
          split_bf16(pv[pg][2], h2, l2);
          split_bf16(pv[pg][3], h3, l3);
          bh[pg][0] = movmatrix_trans(pack_bf16x2(h0, h1));
          bh[pg][1] = movmatrix_trans(pack_bf16x2(h2, h3));
          bl[pg][0] = movmatrix_trans(pack_bf16x2(l0, l1));
          bl[pg][1] = movmatrix_trans(pack_bf16x2(l2, l3));
        }
        // ---- O^T += V^T P^T for my 16 keys of both pages (rows past the valid count masked:
        // their P is 0, but the page image may hold any bits there)
        uint32_t mlo[2], mhi[2];
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          const int ta = t0 + 2 * c, tb = t0 + 8 + 2 * c;
          mlo[pg] = (ta < vld[pg] ? 0x0000FFFFu : 0u) | (ta + 1 < vld[pg] ? 0xFFFF0000u : 0u);
          mhi[pg] = (tb < vld[pg] ? 0x0000FFFFu : 0u) | (tb + 1 < vld[pg] ? 0xFFFF0000u : 0u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int pg = 0; pg < 2; ++pg) {
            uint32_t a[4];
            ldsm_x4_trans(swz(kb[pg] + 2 * kBoxBytes, vrow, 2 * j + vsel), a);
            a[0] &= mlo[pg];
            a[1] &= mlo[pg];
            a[2] &= mhi[pg];
            a[3] &= mhi[pg];
            mma_bf16_16816(O[j][0], a, bh[pg][0], bh[pg][1]);
            mma_bf16_16816(O[j][0], a, bl[pg][0], bl[pg][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.empty[s]);
        if (two) mbar_arrive(&S.empty[s2]);
      }
      jl += two ? 2 : 1;
    }
    flush(cur_job, 0, 0, 0, 1);
    return;
  }

  reset_state();
  for (int jl = 0;; ++jl) {
    const int s = jl % STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s], (jl / STAGES) & 1, p.wait_ns))) {
      if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
      break;
    }
    const StageMeta mt = S.meta[s];
    if (mt.unit == kEnd) break;
    if (mt.unit < 0) {  // defensive: a position the producer could not place
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
      continue;
    }
    if (mt.unit != cur_u || mt.chunk != cur_c) {
      if (cur_u >= 0) flush(cur_u, cur_c, cur_us, cur_uc, 0);
      cur_u = mt.unit;
      cur_c = mt.chunk;
      cur_us = mt.ustart;
      cur_uc = mt.ucount;
      reset_state();
      load_q(stages + size_t(s) * kStage + kKVBytes, DOCS ? mt.pad0 : p.G);
      if (DOCS) {   // the job's query rows each carry their own offset (one document: fixed for the job)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) col_rel[nt] = S.srel[s][grp_row + nt * 8 + r];
      }
      have_rel = false;
    }
    if (mt.valid > t0) {
      if (LAZY && (!have_rel || (!DOCS && mt.rel != cur_rel))) {
        if (!DOCS) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) col_rel[nt] = mt.rel;
        }
        rotate_q(col_rel);
        cur_rel = mt.rel;
        have_rel = true;
      }
      const uint32_t kb = stage0 + s * kStage;
      const uint32_t vb = kb + 2 * kBoxBytes;
      // ---- S^T = K q^T for my 16 keys.  Lazy form: even and odd k-steps accumulate
      // separately (two dependent MMA chains of half the length), then add; the stored-RoPE form
      // keeps one chain (it streams at the same rate either way)
      float acc[NT][4], acc2[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = acc2[nt][e] = 0.f;
      const int krow = t0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldsm_x4(swz(kb, krow, 2 * ks + (lane >> 4)), a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float (&d)[4] = (LAZY && (ks & 1)) ? acc2[nt] : acc[nt];
          mma_bf16_16816(d, a, qh[ks][nt][0], qh[ks][nt][1]);
          if (LAZY && !PACK) mma_bf16_16816(d, a, ql[LAZY && !PACK ? ks : 0][nt][0], ql[LAZY && !PACK ? ks : 0][nt][1]);
        }
      }
      if (LAZY) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
      }
      if (LAZY && PACK) {
        // hi-part scores (columns 0..3) + lo-part scores (columns 4..7), in both halves alike
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[0][e] += __shfl_xor_sync(0xffffffffu, acc[0][e], 2);
      }
      // ---- online softmax (log2 domain) on my 16 rows
      const bool row0_ok = t0 + r < mt.valid, row1_ok = t0 + r + 8 < mt.valid;
      uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float sv[4];
        sv[0] = row0_ok ? acc[nt][0] * scale : -CUDART_INF_F;
        sv[1] = row0_ok ? acc[nt][1] * scale : -CUDART_INF_F;
        sv[2] = row1_ok ? acc[nt][2] * scale : -CUDART_INF_F;
        sv[3] = row1_ok ? acc[nt][3] * scale : -CUDART_INF_F;
        float pv[4];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float mx = fmaxf(sv[cc], sv[cc + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(m[nt][cc], mx);
          const float alpha = exp2f(m[nt][cc] - mnew);
          m[nt][cc] = mnew;
          pv[cc] = exp2f(sv[cc] - mnew);
          pv[cc + 2] = exp2f(sv[cc + 2] - mnew);
          lsum[nt][cc] = lsum[nt][cc] * alpha + pv[cc] + pv[cc + 2];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            O[j][nt][cc] *= alpha;
            O[j][nt][cc + 2] *= alpha;
          }
        }
        float h0, l0, h1, l1, h2, l2, h3, l3;
        split_bf16(pv[0], h0, l0);
        split_bf16(pv[1], h1, l1);
        split_bf16(pv[2], h2, l2);
        split_bf16(pv[3], h3, l3);
        if (PACK) {   // both column halves hold the same P: columns 0..3 keep hi, 4..7 lo
          const bool hi = c < 2;
          bh[nt][0] = movmatrix_trans(pack_bf16x2(hi ? h0 : l0, hi ? h1 : l1));
          bh[nt][1] = movmatrix_trans(pack_bf16x2(hi ? h2 : l2, hi ? h3 : l3));
        } else {
          bh[nt][0] = movmatrix_trans(pack_bf16x2(h0, h1));
          bh[nt][1] = movmatrix_trans(pack_bf16x2(h2, h3));
          bl[nt][0] = movmatrix_trans(pack_bf16x2(l0, l1));
          bl[nt][1] = movmatrix_trans(pack_bf16x2(l2, l3));
        }
      }
      // ---- O^T += V^T P^T for my 16 keys
      const bool partial = mt.valid < t0 + 16;
      uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
      if (partial) {
        const int ta = t0 + 2 * c, tb = t0 + 8 + 2 * c;
        mlo = (ta < mt.valid ? 0x0000FFFFu : 0u) | (ta + 1 < mt.valid ? 0xFFFF0000u : 0u);
        mhi = (tb < mt.valid ? 0x0000FFFFu : 0u) | (tb + 1 < mt.valid ? 0xFFFF0000u : 0u);
      }
      const int vrow = t0 + (lane & 7) + ((lane >> 4) & 1) * 8;
      const int vsel = (lane >> 3) & 1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a[4];
        ldsm_x4_trans(swz(vb, vrow, 2 * j + vsel), a);
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16_16816(O[j][nt], a, bh[nt][0], bh[nt][1]);
          if (!PACK) mma_bf16_16816(O[j][nt], a, bl[nt][0], bl[nt][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
  // the last hand-off ends the epilogue warp (unit -1 when this warp saw no page)
  flush(cur_u, cur_c, cur_us, cur_uc, 1);
}

// Merges the split-K partials of every unit that spans several segments: one CTA per unit and
// group of up to four query heads (a group of five or more heads spreads over several CTAs instead
// of looping), one thread per (query head, output dimension); an online (max, sum) merge over
// batches of eight partials keeps eight independent loads in flight per thread.  Also resets the
// chunk counter for the next launch.
constexpr int kCombineHeads = 4;   // query heads per combine CTA (4 x 128 threads)
constexpr int kCombineBatch = 8;   // partials loaded per round

__global__ void __launch_bounds__(kCombineHeads * kHeadDim)
    attn_combine_kernel(const __grid_constant__ AttnParams p) {
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.x, d = threadIdx.x % kHeadDim;
  if (u == 0 && blockIdx.y == 0 && threadIdx.x == 0) p.ws_ctl[0] = 0;
  const int g = blockIdx.y * kCombineHeads + threadIdx.x / kHeadDim;
  const int first = p.ws_parts[2 * u], nparts = p.ws_parts[2 * u + 1];
  if (nparts <= 1 || g >= p.G) return;
  const int b = u / p.Hk, h = u % p.Hk;
  const int64_t orow = int64_t(b) * p.Hq + h * p.G;
  float M = -CUDART_INF_F, L = 0.f, acc = 0.f;
  for (int i0 = 0; i0 < nparts; i0 += kCombineBatch) {
    float mw[kCombineBatch], lw[kCombineBatch], ow[kCombineBatch];
#pragma unroll
    for (int q = 0; q < kCombineBatch; ++q) {
      if (i0 + q < nparts) {
        const int64_t sl = int64_t(u) + first + i0 + q;
        mw[q] = p.ws_m[sl * 16 + g];
        lw[q] = p.ws_l[sl * 16 + g];
        ow[q] = p.ws_o[(sl * 16 + g) * kHeadDim + d];
      } else {
        mw[q] = -CUDART_INF_F;
        lw[q] = ow[q] = 0.f;
      }
    }
    float mb = M;
#pragma unroll
    for (int q = 0; q < kCombineBatch; ++q) mb = fmaxf(mb, mw[q]);
    if (mb == -CUDART_INF_F) continue;
    const float r = exp2f(M - mb);     // M = -inf gives 0
    L *= r;
    acc *= r;
#pragma unroll
    for (int q = 0; q < kCombineBatch; ++q) {
      const float f = mw[q] == -CUDART_INF_F ? 0.f : exp2f(mw[q] - mb);
      L += f * lw[q];
      acc += f * ow[q];
    }
    M = mb;
  }
  p.out[(orow + g) * kHeadDim + d] = L > 0.f ? acc / L : 0.f;
  if (d == 0) p.lse[orow + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
}

// Document-major form: merges, for each request and query head, the partials its documents' jobs
// left (one per document slot, in slot order), and resets the job counter for the next launch.
__global__ void __launch_bounds__(kCombineHeads * kHeadDim)
    attn_docs_combine_kernel(const __grid_constant__ AttnParams p) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, d = threadIdx.x % kHeadDim;
  if (b == 0 && threadIdx.x == 0) p.ws_ctl[0] = 0;
  for (int hq = threadIdx.x / kHeadDim; hq < p.Hq; hq += kCombineHeads) {
    float M = -CUDART_INF_F, L = 0.f, acc = 0.f;
    for (int i0 = 0; i0 < p.max_docs; i0 += 8) {
      float mw[8], lw[8], ow[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int o = i0 + k < p.max_docs ? p.req_occ[int64_t(b) * p.max_docs + i0 + k] : -1;
        if (o >= 0) {
          const int64_t row = int64_t(o) * p.Hq + hq;
          mw[k] = p.part_m[row];
          lw[k] = p.part_l[row];
          ow[k] = p.part_o[row * kHeadDim + d];
        } else {
          mw[k] = -CUDART_INF_F;
          lw[k] = ow[k] = 0.f;
        }
      }
      float mb = M;
#pragma unroll
      for (int k = 0; k < 8; ++k) mb = fmaxf(mb, mw[k]);
      if (mb == -CUDART_INF_F) continue;
      const float r = exp2f(M - mb);     // M = -inf gives 0
      L *= r;
      acc *= r;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float f = mw[k] == -CUDART_INF_F ? 0.f : exp2f(mw[k] - mb);
        L += f * lw[k];
        acc += f * ow[k];
      }
      M = mb;
    }
    p.out[(int64_t(b) * p.Hq + hq) * kHeadDim + d] = L > 0.f ? acc / L : 0.f;
    if (d == 0) p.lse[int64_t(b) * p.Hq + hq] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
  }
}

template <int NT, bool LAZY, bool PACK, int STAGES, bool DOCS = false>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(attn_split_kernel<NT, LAZY, PACK, STAGES, DOCS>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem_bytes<NT, STAGES, DOCS>()));
}

template <int NT, bool LAZY, bool PACK, int STAGES>
cudaError_t launch_one(const spkv_cache* c, const AttnParams& p, int grid, cudaStream_t st) {
  cudaError_t e = launch_pdl(attn_split_kernel<NT, LAZY, PACK, STAGES>, dim3(grid), dim3(kThreads),
                             smem_bytes<NT, STAGES>(), st, c->tmap_k, c->tmap_v, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel, dim3(p.B * p.Hk, (p.G + kCombineHeads - 1) / kCombineHeads),
                    dim3(kCombineHeads * kHeadDim), 0, st, p);
}

constexpr int kStages1 = 5;   // G <= 8: 5 stages of 34 KiB
constexpr int kStages2 = 4;   // G <= 16: 4 stages of 36 KiB
constexpr int kStagesD = 5;   // document-major: 5 stages of 36 KiB (16 query rows), eight consumer warps

}  // namespace

cudaError_t attn_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<1, true, true, kStages1>()) != cudaSuccess) return e;
  if ((e = set_attr<1, false, false, kStages1>()) != cudaSuccess) return e;
  if ((e = set_attr<1, true, false, kStages1>()) != cudaSuccess) return e;
  if ((e = set_attr<2, false, false, kStages2>()) != cudaSuccess) return e;
  if ((e = set_attr<1, true, false, kStagesD, true>()) != cudaSuccess) return e;
  return set_attr<2, true, false, kStages2>();
}

cudaError_t launch_attn_docs(const spkv_cache* c, const AttnParams& p, int grid, cudaStream_t st) {
  cudaError_t e = launch_pdl(attn_split_kernel<1, true, false, kStagesD, true>, dim3(grid),
                             dim3(Cfg<true>::kThreads), smem_bytes<1, kStagesD, true>(), st, c->tmap_k, c->tmap_v, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_docs_combine_kernel, dim3(p.B), dim3(kCombineHeads * kHeadDim), 0, st, p);
}

cudaError_t launch_attn(const spkv_cache* c, const AttnParams& p, bool lazy, int grid, cudaStream_t st) {
  // PACK only in the lazy form: it saves the lo MMAs of the rotated query and of P, and there
  // the consumer arithmetic shows in the time; the stored-RoPE form streams at the same rate
  // with or without it.
  if (lazy && p.G <= 4) return launch_one<1, true, true, kStages1>(c, p, grid, st);
  if (p.G <= 8) {
    return lazy ? launch_one<1, true, false, kStages1>(c, p, grid, st)
                : launch_one<1, false, false, kStages1>(c, p, grid, st);
  }
  return lazy ? launch_one<2, true, false, kStages2>(c, p, grid, st)
              : launch_one<2, false, false, kStages2>(c, p, grid, st);
}

}  // namespace spkv
