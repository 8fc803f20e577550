// LazyAttention prefill over cached documents, on the 5th-generation tensor cores.
//
// [Lazy] "LazyAttention", sections "Core idea: deferred positional encoding", "Technical
// implementation 1. Prefilling" and "Mathematical equivalence": cached keys carry only their
// document-local rotation, and a query at absolute position n scores the keys of document i
// (placed at offset P_i) after one relative rotation by n - P_i; the result equals attention over
// keys re-rotated to their absolute positions.  A tile of M = 128 query rows shares each K/V
// page, so the rotation is a small cost next to the M x 64 x 128 products per page.
//
// The pages rotate the key block; here each query row is rotated instead, once per document
// switch (a document spans tens of pages, so this is cheaper still, and the key tiles stay as
// TMA wrote them).  Both give the same scores.
//
// One CTA per (request b, kv head h, pair of query heads of its group, tile of 128 query
// rows): the two query heads are two 128-row tiles that share every K/V page.  Consecutive pages
// of one document are taken in groups of two, so that a QK^T product is one N = 128 MMA tile.
// Ten warps:
//   warp 0     TMA producer: K and V of the group's pages (64 x 64 bf16 boxes, 128-byte swizzle;
//              the two pages' rows stacked so each d-half is one 128-row tile) into a 2-slot
//              ring whose K and V halves fill and free on their own (a slot's K is reloaded once
//              both tiles' QK have read it, its V once both PVs have), and L2 prefetches of the
//              pages beyond it;
//   warp 1     MMA issuer (one thread), per tile x in turn: O_x += P_x V_(g-1) (M 128, N 128,
//              P read from tensor memory, V from shared memory as an MN-major operand), then
//              S_x = Q_x K_g^T (M 128, N 64 or 128) into the same tensor-memory columns -- MMAs
//              of one thread execute in issue order, so the PV has read P before the QK writes
//              S; it also zeroes the V rows of a partial page so that P = 0 never meets garbage;
//   warps 2-5, 6-9  softmax of tile 0 and tile 1: thread r owns query row r (TMEM lane r):
//              it rotates its query row on document switches, reads its S row from TMEM,
//              runs the online softmax in the log2 domain, writes its P row (bf16 pairs) back
//              over its S row as the A operand of the next PV MMA, and rescales its O row in
//              TMEM only when the row maximum has grown by more than 2^8 since the last
//              rescale; at the end it normalises O and writes out and lse.  While one tile's
//              warps run their softmax, the tensor cores work on the other tile.
// Tensor memory holds all 512 columns: O of both tiles and one S/P buffer of 128 per tile.
// Hand-offs are mbarriers; every wait is bounded (SPKV_DEVERR_TIMEOUT), and the MMA issuer
// drains its MMAs before TMEM is released.
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace spkv {
namespace {

constexpr int kPM = 128;                      // query rows per tile (TMEM lanes)
constexpr int kTiles = 2;                     // query heads (tiles) per CTA
constexpr int kStages = 2;                    // page-group ring slots (K and V halves freed apart)
constexpr int kPrefetch = 8;                  // pages beyond the ring fetched into L2
constexpr int kPThreads = 64 + kTiles * 128;
constexpr int kBox = 64 * 128;                // one page's 64 rows x 128 B (one d-half), bytes
constexpr int kGBox = 2 * kBox;               // the group's rows of one d-half
constexpr int kStageBytes = 4 * kGBox;        // K half 0, K half 1, V half 0, V half 1
constexpr int kQBytes = 2 * kPM * 128;        // Q tile: two d-halves of 128 rows x 128 B
constexpr uint32_t kTmemCols = 512;           // O of tile x at 128 x; S / P of tile x at 256 + 128 x
constexpr float kRescaleLog2 = 8.f;           // row-max growth (log2) tolerated before O is rescaled
constexpr float kLn2 = 0.69314718055994530942f;

__host__ __device__ constexpr uint32_t o_col(int x) { return 128u * x; }
__host__ __device__ constexpr uint32_t s_col(int x) { return 256u + 128u * x; }

struct PrefillSmem {
  // K and V halves of each ring slot fill and free on their own: a slot's K is free once both
  // tiles' QK have read it, its V once both tiles' PV have
  uint64_t fullK[kStages], emptyK[kStages], fullV[kStages], emptyV[kStages];
  uint64_t sfull[kTiles], pready[kTiles], pvdone[kTiles], qready[kTiles];
  uint64_t drain;
  uint32_t tmem_base;
};

constexpr size_t kPrefillSmem =
    1024 + size_t(kTiles) * kQBytes + size_t(kStages) * kStageBytes + sizeof(PrefillSmem);
static_assert(kPrefillSmem <= 232448, "prefill shared memory exceeds the per-CTA limit");

struct PageInfo {
  int phys, valid, slot;
};

__device__ __forceinline__ PageInfo page_info(const PrefillParams& p, int b, int h, int j) {
  const int mh = p.meta_heads == 1 ? 0 : h;
  const uint32_t w = p.meta[(int64_t(b) * p.meta_heads + mh) * p.np_max + j];
  PageInfo r;
  r.phys = static_cast<int>(w & 0x3FFFFu);
  r.valid = static_cast<int>((w >> 18) & 63u) + 1;
  r.slot = static_cast<int>(w >> 24);
  if (r.phys >= p.n_phys || r.slot >= p.max_docs) {   // skipped page (flagged by the producer)
    r.phys = 0;
    r.valid = 0;
    r.slot = 0;
  }
  return r;
}

// Page j and, when it exists and belongs to the same document, page j + 1.
struct Group {
  PageInfo a, b;
  int size;
};

__device__ __forceinline__ Group group_at(const PrefillParams& p, int b, int h, int j, int n) {
  Group g;
  g.a = page_info(p, b, h, j);
  g.size = 1;
  g.b.phys = g.b.valid = g.b.slot = 0;
  if (j + 1 < n) {
    const PageInfo nb = page_info(p, b, h, j + 1);
    if (nb.slot == g.a.slot) {
      g.b = nb;
      g.size = 2;
    }
  }
  return g;
}

// Bounded wait with one outcome for the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ALIBI: keys carry no rotation and the query rows are written once; each score gets the
// linear bias -slope * (n - m), m = doc_pos[slot] + page_start + column.
template <bool ALIBI>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                            // tile x at x * kQBytes
  uint8_t* stages = base + kTiles * kQBytes;
  PrefillSmem& S = *reinterpret_cast<PrefillSmem*>(stages + kStages * kStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, b = blockIdx.z;
  const int pairs = (p.G + 1) / 2;
  const int h = blockIdx.y / pairs, hq0 = h * p.G + 2 * (blockIdx.y % pairs);
  const int n_tiles = min(kTiles, h * p.G + p.G - hq0);   // the last pair of an odd group has one head

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.fullK[s], 1);
      mbar_init(&S.emptyK[s], 1);
      mbar_init(&S.fullV[s], 1);
      mbar_init(&S.emptyV[s], 1);
    }
    for (int x = 0; x < kTiles; ++x) {
      mbar_init(&S.sfull[x], 1);
      mbar_init(&S.pready[x], 4);
      mbar_init(&S.pvdone[x], 1);
      mbar_init(&S.qready[x], 4);
    }
    mbar_init(&S.drain, 1);
    fence_mbar_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem_base;
  pdl_wait();
  const int n = max(0, min(p.n_pages[b], p.np_max));

  if (warp == 0) {
    // ================================================================ TMA producer
    const uint64_t pol = l2_policy_evict_last();   // the group's other query heads and other requests reuse pages
    auto prefetch = [&](int jj) {
      const PageInfo pi = page_info(p, b, h, jj);
      if (pi.valid == 0) return;
      const int z = static_cast<int>(int64_t(h) * p.n_phys + pi.phys);
      tma_prefetch_l2_3d(&tmk, 0, 0, z);
      tma_prefetch_l2_3d(&tmk, 64, 0, z);
      tma_prefetch_l2_3d(&tmv, 0, 0, z);
      tma_prefetch_l2_3d(&tmv, 64, 0, z);
    };
    // K (v = false) or V (v = true) rows of one page into the slot's half for page a or b
    auto load_page = [&](uint8_t* st, int half_off, const PageInfo& pi, uint64_t* bar, bool v) {
      const int z = static_cast<int>(int64_t(h) * p.n_phys + pi.phys);
      uint8_t* dst = st + (v ? 2 * kGBox : 0) + half_off;
      tma_load_3d(dst, v ? &tmv : &tmk, bar, 0, 0, z, pol);
      tma_load_3d(dst + kGBox, v ? &tmv : &tmk, bar, 64, 0, z, pol);
    };
    if (lane == 0) {
      for (int jj = 0; jj < n; ++jj) {   // flag malformed page words once
        const int mh = p.meta_heads == 1 ? 0 : h;
        const uint32_t w = p.meta[(int64_t(b) * p.meta_heads + mh) * p.np_max + jj];
        if (static_cast<int64_t>(w & 0x3FFFFu) >= p.n_phys) flag_error(p.err, SPKV_DEVERR_PHYS);
        else if (static_cast<int>(w >> 24) >= p.max_docs) flag_error(p.err, SPKV_DEVERR_SLOT);
      }
      for (int jj = 2 * kStages; jj < min(n, 2 * kStages + kPrefetch); ++jj) prefetch(jj);
    }
    int g = 0, j = 0;
    for (; j < n; ++g) {
      const Group gr = group_at(p, b, h, j, n);
      const int s = g % kStages;
      uint8_t* st = stages + s * kStageBytes;
      const uint32_t bytes = (gr.a.valid > 0 ? 2 * kBox : 0) + (gr.size == 2 && gr.b.valid > 0 ? 2 * kBox : 0);
      // K of the group, once both tiles' QK of the slot's previous group have completed
      if (g >= kStages && !warp_wait(&S.emptyK[s], ((g / kStages) - 1) & 1)) {
        if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        for (int jj = j + 2 * kStages + kPrefetch; jj < min(n, j + gr.size + 2 * kStages + kPrefetch); ++jj)
          prefetch(jj);
        if (bytes) {
          mbar_arrive_expect_tx(&S.fullK[s], bytes);
          if (gr.a.valid > 0) load_page(st, 0, gr.a, &S.fullK[s], false);
          if (gr.size == 2 && gr.b.valid > 0) load_page(st, kBox, gr.b, &S.fullK[s], false);
        } else {
          mbar_arrive(&S.fullK[s]);
        }
      }
      __syncwarp();
      // V of the group, once both tiles' PV of the slot's previous group have completed
      if (g >= kStages && !warp_wait(&S.emptyV[s], ((g / kStages) - 1) & 1)) {
        if (lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
        mbar_wait(&S.fullK[s], (g / kStages) & 1);   // this group's K copy must not be in flight at exit
        break;
      }
      if (lane == 0) {
        if (bytes) {
          mbar_arrive_expect_tx(&S.fullV[s], bytes);
          if (gr.a.valid > 0) load_page(st, 0, gr.a, &S.fullV[s], true);
          if (gr.size == 2 && gr.b.valid > 0) load_page(st, kBox, gr.b, &S.fullV[s], true);
        } else {
          mbar_arrive(&S.fullV[s]);
        }
      }
      __syncwarp();
      j += gr.size;
    }
    // no copy of this CTA may still be in flight when it exits
    for (int i = g > kStages ? g - kStages : 0; i < g; ++i) {
      mbar_wait(&S.fullK[i % kStages], (i / kStages) & 1);
      mbar_wait(&S.fullV[i % kStages], (i / kStages) & 1);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t kIdS64 = umma_idesc_bf16(kPM, 64, false);
    constexpr uint32_t kIdS128 = umma_idesc_bf16(kPM, 128, false);
    constexpr uint32_t kIdO = umma_idesc_bf16(kPM, 128, true);
    // Operand descriptors are formed once; a k step adds its byte offset / 16 to the start
    // address field (every address here is below 256 KiB, so the field never overflows).
    const uint64_t q_desc = umma_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t k_desc = umma_desc_sw128(smem_u32(stages), 16, 1024);
    const uint64_t v_desc = umma_desc_sw128(smem_u32(stages + 2 * kGBox), kGBox, 1024);
    bool ok = true;
    int prev_slot = -1, n_docs = 0, prev_size = 0, g = 0;
    // O_x += P_x V of group gg (size sz): P in the first 32 sz columns of S_x
    auto issue_pv = [&](int x, int gg, int sz) -> bool {
      if (!warp_wait(&S.pready[x], gg & 1)) return false;
      if (lane == 0) {
        tc_fence_after();
        const uint64_t va = v_desc + (((gg % kStages) * kStageBytes) >> 4);
        for (int k = 0; k < 4 * sz; ++k)
          umma_bf16_tmem_a(tbase + o_col(x), tbase + s_col(x) + 8 * k, va + 128 * k, kIdO, gg > 0 || k > 0);
        umma_commit(&S.pvdone[x]);
      }
      __syncwarp();
      return true;
    };
    // V of group gg (pages of gp) in its slot; rows past a page's valid tokens are multiplied by
    // P = 0, so they are made exact zeros first
    auto wait_v = [&](int gg, const Group& gp) -> bool {
      if (!warp_wait(&S.fullV[gg % kStages], (gg / kStages) & 1)) return false;
      for (int pg = 0; pg < gp.size; ++pg) {
        const int valid = pg == 0 ? gp.a.valid : gp.b.valid;
        if (valid == 64) continue;
        uint8_t* vt = stages + (gg % kStages) * kStageBytes + 2 * kGBox + pg * kBox;
        for (int i = lane; i < (64 - valid) * 16; i += 32) {
          const int row = valid + (i >> 4), c = i & 15;
          *reinterpret_cast<uint4*>(vt + (c >> 3) * kGBox + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      return true;
    };
    Group prev_gr{};
    for (int j = 0; j < n && ok; ++g) {
      const Group gr = group_at(p, b, h, j, n);
      const int s = g % kStages;
      if (!warp_wait(&S.fullK[s], (g / kStages) & 1)) {
        ok = false;
        break;
      }
      const bool new_doc = ALIBI ? g == 0 : gr.a.slot != prev_slot;
      prev_slot = gr.a.slot;
      for (int x = 0; x < n_tiles && ok; ++x) {
        // PV of the previous group reads P_x from the columns the QK below overwrites; MMAs of
        // one thread run in issue order
        if (g >= 1 && ((x == 0 && !wait_v(g - 1, prev_gr)) || !issue_pv(x, g - 1, prev_size))) {
          ok = false;
          break;
        }
        if (new_doc && !warp_wait(&S.qready[x], n_docs & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint64_t qa = q_desc + ((x * kQBytes) >> 4), ka = k_desc + ((s * kStageBytes) >> 4);
          const uint32_t id = gr.size == 2 ? kIdS128 : kIdS64;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma_bf16(tbase + s_col(x), qa + (((k >> 2) * (kPM * 128) + (k & 3) * 32) >> 4),
                      ka + (((k >> 2) * kGBox + (k & 3) * 32) >> 4), id, k > 0);
          umma_commit(&S.sfull[x]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        umma_commit(&S.emptyK[s]);                                 // both tiles' QK of group g
        if (g >= 1) umma_commit(&S.emptyV[(g - 1) % kStages]);    // both tiles' PV of group g - 1
      }
      __syncwarp();
      if (new_doc) ++n_docs;
      prev_gr = gr;
      prev_size = gr.size;
      j += gr.size;
    }
    if (ok && g > 0) {
      ok = wait_v(g - 1, prev_gr);
      for (int x = 0; x < n_tiles && ok; ++x) ok = issue_pv(x, g - 1, prev_size);
      if (ok && lane == 0) umma_commit(&S.emptyV[(g - 1) % kStages]);
    }
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    // every MMA issued has completed before TMEM is released
    if (lane == 0) umma_commit(&S.drain);
    __syncwarp();
    if (!warp_wait(&S.drain, 0) && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
  } else if ((warp - 2) / 4 < n_tiles) {
    // ================================================================ softmax warps of tile x
    const int x = (warp - 2) / 4;
    const int hq = hq0 + x;
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;         // query row of the tile
    const int t = mt * kPM + r;
    const bool live = t < p.T;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint16_t* qrow = p.q + ((int64_t(b) * p.T + (live ? t : 0)) * p.Hq + hq) * kHeadDim;
    uint8_t* qtile = sQ + x * kQBytes;
    const int pos = p.qpos0[b] + t;
    const float scale = p.scale_log2;
    const float slope_l2 = ALIBI ? p.slopes[hq] * 1.4426950408889634f : 0.f;   // bias slope, log2 units
    float cslope[ALIBI ? 32 : 1];   // ALiBi: c slope for the 32 columns of a block
#pragma unroll
    for (int c = 0; c < (ALIBI ? 32 : 1); ++c) cslope[c] = static_cast<float>(c) * slope_l2;
    const int64_t ps_row = (int64_t(b) * p.meta_heads + (p.meta_heads == 1 ? 0 : h)) * p.np_max;
    float m = -CUDART_INF_F, l = 0.f;
    int prev_slot = -1, g = 0;
    bool ok = true;
    for (int j = 0; j < n; ++g) {
      const Group gr = group_at(p, b, h, j, n);
      // columns of each page this row attends: its valid tokens, and with page positions known
      // (ALiBi, or the RoPE step) only keys at positions m <= pos: column c of a page whose first
      // token sits at m0 is visible while m0 + c <= pos (cached documents precede every row; the
      // rows' own document, placed at qpos0, is the causal part)
      int va = gr.a.valid, vb = gr.size == 2 ? gr.b.valid : 0;
      // ALiBi: the bias of column 0 of each page of the group (log2 units), slope (m - n)
      float cb_a = 0.f, cb_b = 0.f;
      if (ALIBI || p.causal) {
        const int dp = p.doc_pos[int64_t(b) * p.max_docs + gr.a.slot];
        const int m0a = dp + p.page_start[ps_row + j];
        const int m0b = gr.size == 2 ? dp + p.page_start[ps_row + j + 1] : 0;
        if (ALIBI) {
          cb_a = slope_l2 * static_cast<float>(m0a - pos);
          if (gr.size == 2) cb_b = slope_l2 * static_cast<float>(m0b - pos);
        }
        va = min(va, max(0, pos - m0a + 1));
        if (gr.size == 2) vb = min(vb, max(0, pos - m0b + 1));
      }
      j += gr.size;
      if (ALIBI ? g == 0 : gr.a.slot != prev_slot) {
        // Document switch: every MMA that read the previous rotation has completed (its S
        // row was read in the previous iteration), so row r of Q is rewritten as
        // R(pos - doc_pos[slot]) q in bf16 (ALiBi: q itself, once).
        prev_slot = gr.a.slot;
        const int rel = ALIBI ? 0 : pos - p.doc_pos[int64_t(b) * p.max_docs + gr.a.slot];
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint4 xa = make_uint4(0, 0, 0, 0), ya = make_uint4(0, 0, 0, 0);
          if (live) {
            xa = *reinterpret_cast<const uint4*>(qrow + 8 * cc);
            ya = *reinterpret_cast<const uint4*>(qrow + 64 + 8 * cc);
          }
          const uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w}, yw[4] = {ya.x, ya.y, ya.z, ya.w};
          uint32_t xo[4], yo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float sn[2], cs[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int i = 8 * cc + 2 * e + k;   // pair index: dims i and i + 64
              const uint64_t ph = static_cast<uint64_t>(static_cast<int64_t>(rel)) * p.phase_inc[i];
              const float ang = static_cast<float>(static_cast<int32_t>(ph >> 32)) * 1.4629180792671596e-09f;
              __sincosf(ang, &sn[k], &cs[k]);
            }
            const float x0 = bf16lo_to_f32(xw[e]), x1 = bf16hi_to_f32(xw[e]);
            const float y0 = bf16lo_to_f32(yw[e]), y1 = bf16hi_to_f32(yw[e]);
            xo[e] = pack_bf16x2(x0 * cs[0] - y0 * sn[0], x1 * cs[1] - y1 * sn[1]);
            yo[e] = pack_bf16x2(y0 * cs[0] + x0 * sn[0], y1 * cs[1] + x1 * sn[1]);
          }
          const int off = r * 128 + ((cc ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(qtile + off) = make_uint4(xo[0], xo[1], xo[2], xo[3]);
          *reinterpret_cast<uint4*>(qtile + kPM * 128 + off) = make_uint4(yo[0], yo[1], yo[2], yo[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.qready[x]);
      }
      if (!warp_wait(&S.sfull[x], g & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S columns: page a in 0..63, page b in 64..127 (a group of one page fills only the first
      // 64).  Two passes over tensor memory keep 32 columns in registers at a time: the row
      // maximum first, then p, the row sum and P (bf16 pairs written over the columns already
      // read: block k's 16 words land on columns 16 k .. 16 k + 15 <= 32 k).
      const bool full = va == 64 && vb == 64;
      const int nblk = 2 * gr.size;
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = -CUDART_INF_F;
#pragma unroll 1
      for (int k = 0; k < nblk; ++k) {
        uint32_t sv[32];
        tmem_ld32(lane_addr + s_col(x) + 32 * k, sv);
        tmem_wait_ld();
        const int lim = (k < 2 ? va : vb) - 32 * (k & 1);   // valid columns of this block
        if (ALIBI) {   // the maximum of s scale + bias: of s scale + c slope, plus the block's cb
          const float cb = (k < 2 ? cb_a : cb_b) + slope_l2 * static_cast<float>(32 * (k & 1));
          float bm8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) bm8[e] = -CUDART_INF_F;
          if (full) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              bm8[c & 7] = fmaxf(bm8[c & 7], fmaf(__uint_as_float(sv[c]), scale, cslope[ALIBI ? c : 0]));
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float a = fmaf(__uint_as_float(sv[c]), scale, cslope[ALIBI ? c : 0]);
              bm8[c & 7] = fmaxf(bm8[c & 7], c < lim ? a : -CUDART_INF_F);
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], bm8[e] + cb);
        } else if (full) {   // the maximum of s (scale > 0 is applied once below); every column valid
#pragma unroll
          for (int c = 0; c < 32; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(sv[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            mx8[c & 7] = fmaxf(mx8[c & 7], c < lim ? __uint_as_float(sv[c]) : -CUDART_INF_F);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_grp = ALIBI ? mx : mx * scale;
      bool rescale = false;
      float alpha = 1.f;
      if (m == -CUDART_INF_F) {
        m = m_grp;   // nothing accumulated yet (O holds zeros or nothing)
      } else if (m_grp > m + kRescaleLog2) {
        rescale = true;
        alpha = fast_exp2(m - m_grp);
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O holds every PV issued before this group's QK (issue order): they have completed
        // once S arrived, but wait for the previous group's PV explicitly
        if (!warp_wait(&S.pvdone[x], (g - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < 128; cb += 32) {
          uint32_t o[32];
          tmem_ld32(lane_addr + o_col(x) + cb, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(lane_addr + o_col(x) + cb, o);
        }
        tmem_wait_st();
        if (rescale) {
          l *= alpha;
          m = m_grp;
        }
      }
      // p = 2^(s * scale - m), zero past the valid columns (and everywhere while m is -inf)
      const bool have_m = m != -CUDART_INF_F;
      const float mneg = have_m ? -m : 0.f;
      float ls8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls8[k] = 0.f;
#pragma unroll 1
      for (int k = 0; k < nblk; ++k) {
        uint32_t sv[32];
        tmem_ld32(lane_addr + s_col(x) + 32 * k, sv);
        tmem_wait_ld();
        const int lim = have_m ? (k < 2 ? va : vb) - 32 * (k & 1) : 0;
        // ALiBi: column c adds c slope to the block's bias; RoPE: no bias
        const float cbm = ALIBI ? (k < 2 ? cb_a : cb_b) + slope_l2 * static_cast<float>(32 * (k & 1)) + mneg : mneg;
        uint32_t pw[16];
        if (full && have_m) {   // every column valid: no masking; column pairs in packed f32x2 form
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float b0 = mneg, b1 = mneg, e0, e1;
            if (ALIBI)
              fma_f32x2(b0, b1, static_cast<float>(c), static_cast<float>(c + 1), slope_l2, slope_l2, cbm, cbm);
            fma_f32x2(e0, e1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), scale, scale, b0, b1);
            const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
            add_f32x2(ls8[c & 7], ls8[(c + 1) & 7], p0, p1);   // c even: two neighbouring sums
            pw[c >> 1] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float b0 = ALIBI ? fmaf(static_cast<float>(c), slope_l2, cbm) : mneg;
            const float b1 = ALIBI ? fmaf(static_cast<float>(c + 1), slope_l2, cbm) : mneg;
            const float e0 = fast_exp2(fmaf(__uint_as_float(sv[c]), scale, b0));
            const float e1 = fast_exp2(fmaf(__uint_as_float(sv[c + 1]), scale, b1));
            const float p0 = (have_m && c < lim) ? e0 : 0.f;
            const float p1 = (have_m && c + 1 < lim) ? e1 : 0.f;
            ls8[c & 7] += p0;
            ls8[(c + 1) & 7] += p1;
            pw[c >> 1] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(lane_addr + s_col(x) + 16 * k, pw);
      }
      l += ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pready[x]);
    }
    if (ok && g > 0) ok = warp_wait(&S.pvdone[x], (g - 1) & 1);
    if (!ok && lane == 0) flag_error(p.err, SPKV_DEVERR_TIMEOUT);
    tc_fence_after();
    float* orow = p.out + ((int64_t(b) * p.T + (live ? t : 0)) * p.Hq + hq) * kHeadDim;
    const bool have = ok && g > 0 && l > 0.f;
    const float inv_l = have ? 1.f / l : 0.f;
#pragma unroll 1
    for (int cb = 0; cb < 128; cb += 32) {
      uint32_t o[32] = {};
      if (ok && g > 0) {   // TMEM holds O only once a PV has run
        tmem_ld32(lane_addr + o_col(x) + cb, o);
        tmem_wait_ld();
      }
      if (live) {
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float4 w;
          w.x = have ? __uint_as_float(o[c]) * inv_l : 0.f;
          w.y = have ? __uint_as_float(o[c + 1]) * inv_l : 0.f;
          w.z = have ? __uint_as_float(o[c + 2]) * inv_l : 0.f;
          w.w = have ? __uint_as_float(o[c + 3]) * inv_l : 0.f;
          *reinterpret_cast<float4*>(orow + cb + c) = w;
        }
      }
    }
    if (live) p.lse[(int64_t(b) * p.T + t) * p.Hq + hq] = have ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t prefill_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kPrefillSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kPrefillSmem));
}

cudaError_t launch_prefill(const spkv_cache* c, const PrefillParams& p, cudaStream_t st) {
  const int pairs = (p.G + 1) / 2;
  const dim3 grid((p.T + kPM - 1) / kPM, p.Hk * pairs, p.B);
  return launch_pdl(p.slopes ? prefill_kernel<true> : prefill_kernel<false>, grid, dim3(kPThreads), kPrefillSmem, st,
                    c->tmap_k, c->tmap_v, p);
}

}  // namespace spkv
