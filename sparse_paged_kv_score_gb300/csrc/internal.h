// Host-side handle and the launch functions each kernel file exports to api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/spkv.h"

struct spkv_cache {
  spkv_desc d;
  int device = 0;
  int sm_count = 0;
  CUtensorMap tmap_k;   // K pool as [Hk*n_phys][64 tok][128 d] bf16, box 64x64, 128B swizzle
  CUtensorMap tmap_v;
  uint32_t* dev_err = nullptr;   // device error word
  float* ws_m = nullptr;         // split-K partial row max   [slots][16]
  float* ws_l = nullptr;         // split-K partial row sum   [slots][16]
  float* ws_o = nullptr;         // split-K partial outputs   [slots][16][128]
  int32_t* ws_cnt = nullptr;     // per unit (first segment, segments) [2 * max_units], then the chunk counter
  int64_t ws_slots = 0;
  int32_t max_units = 0;
  int attn_grid = 0;             // CTAs of the split-K attention kernel (one per SM)
  int max_chunks = 0;            // chunks the attention kernel may cut its page sequence into
  uint64_t wait_ns = 1000000000ull;   // limit of the attention kernel's bounded hand-off waits
  const void* host_k = nullptr;  // last host pool given to retrieve_pages and its device address
  const void* host_v = nullptr;
  const void* host_k_dev = nullptr;
  const void* host_v_dev = nullptr;
};

namespace spkv {

// Device view of a two-level page directory (spkv_page_dir); dir == nullptr means the call uses a
// flat page table instead.
struct PageDir {
  const int32_t* dir;            // [B][n_dir]: >= 0 device segment, <= -2 host segment -2 - e, -1 unmapped
  const int32_t* dev;            // device-tier segments [n_dev][1 << shift]
  const int32_t* const* chunks;  // device addresses of the host chunks, each [1 << chunk_shift][1 << shift]
  int n_dir, shift, n_dev, chunk_shift;
  int64_t n_host;
};

// Launches `k` with programmatic stream serialisation: the kernel may start while the previous
// kernel of the stream finishes; every kernel of this library calls pdl_wait() before it reads
// anything an earlier kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// Sets the dynamic shared-memory limits of every kernel once (at handle creation), so that no
// launch path calls cudaFuncSetAttribute and every call can be captured in a CUDA graph.
cudaError_t init_kernel_attributes();

// Parameters of the split-K attention kernel (sparse and lazy forms).
struct AttnParams {
  const void* q;
  float* out;
  float* lse;
  int B, Hq, Hk, G;
  int64_t n_phys;
  uint32_t* err;
  float* ws_m;
  float* ws_l;
  float* ws_o;
  int32_t* ws_parts;             // per unit: first segment and number of segments (partials)
  int32_t* ws_ctl;               // [0] next chunk to hand out; 0 between calls
  int max_chunks;                // chunks of the page sequence at most (workspace slots = units + this)
  int min_chunk;                 // smallest segment length (keeps a unit's partials <= 256)
  // sparse form
  const int32_t* page_table;
  int np_max;
  const int32_t* sel;
  const int32_t* n_sel;
  int sel_stride;
  const int32_t* seq_len;
  PageDir pd;                    // two-level page directory (pd.dir null: page_table)
  const int32_t* slot;           // resident-slot form: slot of each selected page (else null)
  int n_slots;                   // slots per (request, kv head); page = b * n_slots + slot
  // lazy form
  const int32_t* qpos;
  const uint32_t* meta;
  int meta_heads;
  const int32_t* n_pages;
  const int32_t* doc_pos;
  int max_docs;
  // document-major lazy form (a plan's jobs)
  const int4* jobs;              // [n_jobs]: document, kv head, first occurrence, occurrences
  int n_jobs;
  const int2* occ;               // [occurrences]: request, document slot
  const int32_t* req_occ;        // [B][max_docs]: occurrence of each (request, slot), -1 for none
  const uint32_t* doc_pages;     // page words (phys | (valid - 1) << 18) of every document, by document
  const int32_t* doc_first;      // [documents + 1]: first page word of each document
  float* part_m;                 // [occurrences][Hq] row max (log2 domain), sum and unnormalised O
  float* part_l;
  float* part_o;
  float scale_log2;              // log2(e) / sqrt(128)
  uint64_t wait_ns;              // limit of each intra-CTA hand-off wait (0: give up unless complete)
  uint64_t phase_inc[64];        // RoPE pair j: turns per position, 2^-64 fixed point
};

// Parameters of the LazyAttention prefill kernel (tcgen05).
struct PrefillParams {
  const uint16_t* q;             // bf16 [B][T][Hq][128]
  float* out;                    // [B][T][Hq][128]
  float* lse;                    // [B][T][Hq]
  int B, T, Hq, Hk, G;
  int64_t n_phys;
  const int32_t* qpos0;
  const uint32_t* meta;
  int meta_heads;
  const int32_t* n_pages;
  int np_max;
  const int32_t* doc_pos;
  int max_docs;
  float scale_log2;
  uint32_t* err;
  uint64_t phase_inc[64];
  const int32_t* page_start;     // ALiBi form and RoPE step: document-local start of each listed page
  const float* slopes;           // ALiBi form: [Hq] bias slopes (natural-log units); null for RoPE
  int causal;                    // RoPE step: keys at positions after a row are masked (needs page_start);
                                 // the ALiBi form always masks them
};

// Parameters of the column-score kernel (PyramidKV-style score S).
struct ColScoreParams {
  const uint16_t* q;             // bf16 [B][alpha][Hq][128]: the last alpha rows of each prompt
  float* scores;                 // [B][Hq][np_max * 64]
  int B, alpha, Hq, Hk, G;
  int row0, rows;                // this launch's chunk: window rows row0 .. row0 + rows - 1 (rows <= 128;
                                 // <= 256 in the given-LSE kernel)
  int accumulate;                // 0: write the chunk's sums (first chunk), 1: add them
  int chunks_in_grid;            // 2: blockIdx.z is the chunk (rows 128 z ..), sums added atomically
                                 // onto a zeroed row (two addends onto zero: order-independent)
  int64_t n_phys;
  const int32_t* page_table;     // [B][np_max]
  int np_max;
  const int32_t* seq_len;        // prompt length n per request
  const float* lse_in;           // [B][alpha][Hq] natural-log LSE of each window row, or null (pass 1 runs)
  int lse_is_log2;               // lse_in holds log2-domain values (written by a pass-1 launch)
  float* lse_out;                // colscore_kernel: pass 1 alone, each row's log2-domain LSE to [B][alpha][Hq]
  float scale_log2;
  uint32_t* err;
};

cudaError_t launch_summary_build(const spkv_cache* c, cudaStream_t st);
cudaError_t launch_append(const spkv_cache* c, const int32_t* phys, const int32_t* tok, const void* k_new,
                          const void* v_new, int n_rows, cudaStream_t st);
// The fused decode append's pointers (k_new, v_new: bf16 [B][Hk][128] as 32-bit words).
struct AppendRows {
  uint32_t* kpool;
  uint32_t* vpool;
  int32_t* page_cnt;
  const uint32_t* k_new;
  const uint32_t* v_new;
};

// k_new == nullptr: scores only; else the decode append of each request's new row is fused in.
cudaError_t launch_score(const spkv_cache* c, const void* q, int B, int Hq, const int32_t* page_table,
                         int np_max, const int32_t* seq_len, float* scores, cudaStream_t st,
                         const void* k_new = nullptr, const void* v_new = nullptr, const PageDir* pd = nullptr);
cudaError_t launch_select(const spkv_cache* c, const float* qs, const float* es, uint32_t* alive, int B,
                          int np_max, const int32_t* seq_len, int k_q, int k_e, int32_t* sel, int32_t* n_sel,
                          cudaStream_t st);
cudaError_t launch_attn(const spkv_cache* c, const AttnParams& p, bool lazy, int grid, cudaStream_t st);
cudaError_t launch_attn_docs(const spkv_cache* c, const AttnParams& p, int grid, cudaStream_t st);
cudaError_t launch_setdiff(uint32_t* err, const int32_t* resident, int n_slots, const int32_t* sel,
                           const int32_t* n_sel, int sel_stride, int n_units, int32_t* missing,
                           int32_t* n_missing, int32_t* slot, cudaStream_t st);
cudaError_t launch_retrieve(const spkv_cache* c, const void* k_host, const void* v_host, int64_t n_host_pages,
                            const int32_t* page_table, int np_max, int B, const int32_t* missing,
                            const int32_t* n_missing, const int32_t* victims, int32_t* slot, const int32_t* n_sel,
                            int sel_stride, int n_slots, cudaStream_t st, const PageDir* pd = nullptr);
cudaError_t launch_lru(uint32_t* err, int32_t* resident, int32_t* ts, int n_slots, const int32_t* slot,
                       const int32_t* n_sel, const int32_t* missing, const int32_t* n_missing, int sel_stride,
                       int n_units, int32_t t_now, int bucket_width, int32_t* victims, int32_t* hist,
                       cudaStream_t st);

cudaError_t launch_select_resident(const spkv_cache* c, const float* qs, const float* es, uint32_t* alive, int B,
                                   int np_max, const int32_t* seq_len, int k_q, int k_e, int32_t* sel,
                                   int32_t* n_sel, int32_t* resident, int32_t* ts, int n_slots, int32_t t_now,
                                   int W, int32_t* missing, int32_t* n_missing, int32_t* slot, int32_t* victims,
                                   int32_t* hist, cudaStream_t st);
bool fused_supported(int np_max);

// Shared-memory bytes the attention kernel needs for a group size (used for limits checks).
cudaError_t attn_init_attributes();
cudaError_t select_init_attributes();
cudaError_t resid_init_attributes();
cudaError_t fused_init_attributes();
cudaError_t prefill_init_attributes();
cudaError_t colscore_init_attributes();
cudaError_t launch_colscore(const spkv_cache* c, const ColScoreParams& p, cudaStream_t st);
// Given-LSE column scores, keys as M: rows row0 .. row0 + rows - 1 (rows <= 256) of the window,
// tmq the window rows [B][alpha][Hq][128] as a 4-D tensor (d, hq, row, b), box 64 x 1 x 256 x 1,
// 128-byte swizzle; grid persistent CTAs.  At most colscore_lse_max_requests() requests.
int colscore_lse_max_requests();
cudaError_t launch_colscore_lse(const spkv_cache* c, const ColScoreParams& p, const CUtensorMap& tmq, int grid,
                                cudaStream_t st);
cudaError_t launch_prefill(const spkv_cache* c, const PrefillParams& p, cudaStream_t st);

}  // namespace spkv
