// Host side of the C ABI declared in include/spkv.h: argument checks, the handle, tensor-map
// encoding and kernel launches.  No entry point synchronises except spkv_get_device_error.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <new>

#include "internal.h"

using spkv::AttnParams;

namespace {

constexpr int kMaxGroup = 16;
constexpr int kMaxColumnRows = 1024;   // window rows of attn_column_scores (eight 128-row launches)
constexpr int kMaxUnitsDefault = 4096;

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int status_of(cudaError_t e) { return e == cudaSuccess ? SPKV_OK : SPKV_ECUDA; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Pool [n_page_heads][64 tok][128 d] bf16 as a 3-D tensor (d, tok, page-head); box 64 x 64 x 1
// with 128-byte swizzle (a 128-byte row of the box is one token's 64 dims).
bool encode_pool(CUtensorMap* m, void* base, int64_t n_page_heads) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, 64, static_cast<cuuint64_t>(n_page_heads)};
  cuuint64_t strides[2] = {256, 16384};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Window rows [B][alpha][Hq][128] bf16 as a 4-D tensor (d, hq, row, b); box 64 x 1 x 256 x 1 with
// 128-byte swizzle (one box is 256 rows of one head's 64-dim half, rows past alpha read as zero).
bool encode_rows(CUtensorMap* m, const void* q, int B, int alpha, int Hq) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(alpha), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {256, static_cast<cuuint64_t>(Hq) * 256, static_cast<cuuint64_t>(alpha) * Hq * 256};
  cuuint32_t box[4] = {64, 1, 256, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int check_group(spkv_cache_t c, int B, int Hq) {
  if (!c || B < 0 || Hq <= 0) return SPKV_EINVAL;
  const int Hk = c->d.n_kv_heads;
  if (Hq % Hk != 0) return SPKV_EINVAL;
  const int G = Hq / Hk;
  if (G < 1 || G > kMaxGroup) return SPKV_EUNSUPPORTED;
  if (int64_t(B) * Hk > c->max_units) return SPKV_EINVAL;
  return SPKV_OK;
}

void fill_common(AttnParams& p, spkv_cache_t c, const void* q, int B, int Hq, float* out, float* lse) {
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hk = c->d.n_kv_heads;
  p.G = Hq / p.Hk;
  p.n_phys = c->d.n_phys_pages;
  p.err = c->dev_err;
  p.ws_m = c->ws_m;
  p.ws_l = c->ws_l;
  p.ws_o = c->ws_o;
  p.ws_parts = c->ws_cnt;
  p.ws_ctl = c->ws_cnt + 2 * c->max_units;
  p.max_chunks = c->max_chunks;
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(128.0));
  p.wait_ns = c->wait_ns;
}

}  // namespace

namespace spkv {
cudaError_t init_kernel_attributes() {
  cudaError_t e;
  if ((e = attn_init_attributes()) != cudaSuccess) return e;
  if ((e = select_init_attributes()) != cudaSuccess) return e;
  if ((e = fused_init_attributes()) != cudaSuccess) return e;
  if ((e = prefill_init_attributes()) != cudaSuccess) return e;
  if ((e = colscore_init_attributes()) != cudaSuccess) return e;
  return resid_init_attributes();
}
}  // namespace spkv

extern "C" {

const char* spkv_status_string(int s) {
  switch (s) {
    case SPKV_OK: return "SPKV_OK";
    case SPKV_EINVAL: return "SPKV_EINVAL: invalid argument";
    case SPKV_ENOMEM: return "SPKV_ENOMEM: allocation failed";
    case SPKV_ECUDA: return "SPKV_ECUDA: CUDA call or launch failed";
    case SPKV_EDEVICE: return "SPKV_EDEVICE: device data out of range (see error bits)";
    case SPKV_ETIMEOUT: return "SPKV_ETIMEOUT: a bounded device wait gave up";
    case SPKV_EUNSUPPORTED: return "SPKV_EUNSUPPORTED: shape outside the supported sizes";
    default: return "unknown status";
  }
}

int paged_kv_create(const spkv_desc* desc, void* stream, spkv_cache_t* out) {
  if (!desc || !out) return SPKV_EINVAL;
  *out = nullptr;
  const spkv_desc& d = *desc;
  if (d.head_dim != 128 || d.page_tokens != 64 || d.subblock != 16) return SPKV_EUNSUPPORTED;
  if (d.n_kv_heads <= 0 || d.n_phys_pages <= 0 || d.max_units < 0 || d.max_units > 4096) return SPKV_EINVAL;
  if (!d.k_pool || !d.v_pool || !d.ksum != !d.page_cnt) return SPKV_EINVAL;
  if (d.ksum_bf16 != 0 && d.ksum_bf16 != 1) return SPKV_EINVAL;
  if (!aligned(d.k_pool, 16) || !aligned(d.v_pool, 16) || !aligned(d.ksum, 16)) return SPKV_EINVAL;
  const int64_t n_ph = int64_t(d.n_kv_heads) * d.n_phys_pages;
  if (n_ph >= (int64_t(1) << 31)) return SPKV_EUNSUPPORTED;

  spkv_cache* c = new (std::nothrow) spkv_cache();
  if (!c) return SPKV_ENOMEM;
  c->d = d;
  c->max_units = d.max_units > 0 ? d.max_units : kMaxUnitsDefault;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return SPKV_ECUDA;
  }
  c->attn_grid = c->sm_count;
  if (spkv::init_kernel_attributes() != cudaSuccess) {
    delete c;
    return SPKV_ECUDA;
  }
  if (!encode_pool(&c->tmap_k, d.k_pool, n_ph) || !encode_pool(&c->tmap_v, d.v_pool, n_ph)) {
    delete c;
    return SPKV_ECUDA;
  }
  c->max_chunks = 16 * c->attn_grid;
  c->ws_slots = int64_t(c->max_chunks) + c->max_units;
  bool ok = cudaMalloc(&c->dev_err, sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(&c->ws_m, sizeof(float) * 16 * c->ws_slots) == cudaSuccess &&
            cudaMalloc(&c->ws_l, sizeof(float) * 16 * c->ws_slots) == cudaSuccess &&
            cudaMalloc(&c->ws_o, sizeof(float) * 16 * 128 * c->ws_slots) == cudaSuccess &&
            cudaMalloc(&c->ws_cnt, sizeof(int32_t) * (2 * c->max_units + 2)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    paged_kv_destroy(c);
    return SPKV_ENOMEM;
  }
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(c->dev_err, 0, sizeof(uint32_t), st) != cudaSuccess ||
      cudaMemsetAsync(c->ws_cnt, 0, sizeof(int32_t) * (2 * c->max_units + 2), st) != cudaSuccess ||
      (d.ksum && spkv::launch_summary_build(c, st) != cudaSuccess)) {
    paged_kv_destroy(c);
    return SPKV_ECUDA;
  }
  *out = c;
  return SPKV_OK;
}

int paged_kv_destroy(spkv_cache_t c) {
  if (!c) return SPKV_EINVAL;
  cudaFree(c->dev_err);
  cudaFree(c->ws_m);
  cudaFree(c->ws_l);
  cudaFree(c->ws_o);
  cudaFree(c->ws_cnt);
  delete c;
  return SPKV_OK;
}

int spkv_sm_count(spkv_cache_t c) { return c ? c->sm_count : SPKV_EINVAL; }

int spkv_set_wait_limit(spkv_cache_t c, uint64_t ns) {
  if (!c || ns > 10000000000ull) return SPKV_EINVAL;
  c->wait_ns = ns;
  return SPKV_OK;
}

int paged_kv_append(spkv_cache_t c, const int32_t* phys_page, const int32_t* tok_in_page, const void* k_new,
                    const void* v_new, int n_rows, void* stream) {
  if (!c || !c->d.ksum || n_rows < 0) return SPKV_EINVAL;
  if (n_rows == 0) return SPKV_OK;
  if (!phys_page || !tok_in_page || !k_new || !v_new || !aligned(k_new, 4) || !aligned(v_new, 4)) return SPKV_EINVAL;
  return status_of(spkv::launch_append(c, phys_page, tok_in_page, k_new, v_new, n_rows, as_stream(stream)));
}

int score_blocks(spkv_cache_t c, const void* q, int B, int Hq, const int32_t* page_table, int np_max,
                 const int32_t* seq_len, float* scores, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (!c->d.ksum) return SPKV_EINVAL;
  if (B == 0) return SPKV_OK;
  if (!q || !page_table || !seq_len || !scores || np_max <= 0 || !aligned(q, 8)) return SPKV_EINVAL;
  return status_of(spkv::launch_score(c, q, B, Hq, page_table, np_max, seq_len, scores, as_stream(stream)));
}

int decode_append_score(spkv_cache_t c, const void* k_new, const void* v_new, const void* q, int B, int Hq,
                        const int32_t* page_table, int np_max, const int32_t* seq_len, float* scores, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (!c->d.ksum) return SPKV_EINVAL;
  if (B == 0) return SPKV_OK;
  if (!q || !page_table || !seq_len || !scores || np_max <= 0 || !aligned(q, 8)) return SPKV_EINVAL;
  if (!k_new || !v_new || !aligned(k_new, 4) || !aligned(v_new, 4)) return SPKV_EINVAL;
  return status_of(spkv::launch_score(c, q, B, Hq, page_table, np_max, seq_len, scores, as_stream(stream), k_new,
                                      v_new));
}

int select_topk(spkv_cache_t c, const float* q_scores, const float* evict_scores, uint32_t* alive, int B, int np_max,
                const int32_t* seq_len, int k_q, int k_e, int32_t* sel, int32_t* n_sel, void* stream) {
  if (!c || B < 0) return SPKV_EINVAL;
  if (int64_t(B) * c->d.n_kv_heads > 65535) return SPKV_EINVAL;
  if (B == 0) return SPKV_OK;
  if (!q_scores || !evict_scores || !alive || !seq_len || !sel || !n_sel) return SPKV_EINVAL;
  if (np_max <= 0 || np_max > 32768 || k_q < 0 || k_e < 0 || k_q + k_e + 1 > 4096) return SPKV_EINVAL;
  return status_of(spkv::launch_select(c, q_scores, evict_scores, alive, B, np_max, seq_len, k_q, k_e, sel, n_sel,
                                       as_stream(stream)));
}

int sparse_decode_attn(spkv_cache_t c, const void* q, int B, int Hq, const int32_t* page_table, int np_max,
                       const int32_t* sel, const int32_t* n_sel, int sel_stride, const int32_t* seq_len, float* out,
                       float* lse, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (B == 0) return SPKV_OK;
  if (!q || !page_table || !sel || !n_sel || !seq_len || !out || !lse || np_max <= 0 || sel_stride <= 0 ||
      !aligned(q, 16))
    return SPKV_EINVAL;
  AttnParams p;
  fill_common(p, c, q, B, Hq, out, lse);
  p.page_table = page_table;
  p.np_max = np_max;
  p.sel = sel;
  p.n_sel = n_sel;
  p.sel_stride = sel_stride;
  p.seq_len = seq_len;
  p.min_chunk = (sel_stride + 125) / 126;
  const int64_t t_max = int64_t(B) * c->d.n_kv_heads * sel_stride;
  const int grid = static_cast<int>(t_max < c->attn_grid ? t_max : c->attn_grid);
  return status_of(spkv::launch_attn(c, p, false, grid, as_stream(stream)));
}

int sparse_decode_attn_slots(spkv_cache_t c, const void* q, int B, int Hq, const int32_t* sel, const int32_t* slot,
                             const int32_t* n_sel, int sel_stride, int n_slots, const int32_t* seq_len, float* out,
                             float* lse, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (B == 0) return SPKV_OK;
  if (!q || !sel || !slot || !n_sel || !seq_len || !out || !lse || sel_stride <= 0 || n_slots <= 0 ||
      !aligned(q, 16))
    return SPKV_EINVAL;
  if (int64_t(B) * n_slots > c->d.n_phys_pages) return SPKV_EINVAL;
  AttnParams p;
  fill_common(p, c, q, B, Hq, out, lse);
  p.np_max = 1 << 25;   // bounds the logical page id (64 * id stays within int); no page table here
  p.sel = sel;
  p.n_sel = n_sel;
  p.sel_stride = sel_stride;
  p.seq_len = seq_len;
  p.slot = slot;
  p.n_slots = n_slots;
  p.min_chunk = (sel_stride + 125) / 126;
  const int64_t t_max = int64_t(B) * c->d.n_kv_heads * sel_stride;
  const int grid = static_cast<int>(t_max < c->attn_grid ? t_max : c->attn_grid);
  return status_of(spkv::launch_attn(c, p, false, grid, as_stream(stream)));
}

int lazy_rope_decode_attn(spkv_cache_t c, const void* q, int B, int Hq, const int32_t* qpos, const uint32_t* meta,
                          int meta_heads, const int32_t* n_pages, int np_max, const int32_t* doc_pos, int max_docs,
                          float theta, float* out, float* lse, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (B == 0) return SPKV_OK;
  if (!q || !qpos || !meta || !n_pages || !doc_pos || !out || !lse || np_max <= 0 || max_docs <= 0 ||
      !aligned(q, 16))
    return SPKV_EINVAL;
  if (meta_heads != 1 && meta_heads != c->d.n_kv_heads) return SPKV_EINVAL;
  if (!(theta > 1.0f) || !std::isfinite(theta)) return SPKV_EINVAL;
  AttnParams p;
  fill_common(p, c, q, B, Hq, out, lse);
  p.np_max = np_max;
  p.qpos = qpos;
  p.meta = meta;
  p.meta_heads = meta_heads;
  p.n_pages = n_pages;
  p.doc_pos = doc_pos;
  p.max_docs = max_docs;
  p.min_chunk = (np_max + 125) / 126;
  // turns per position of pair j: theta^(-2j/128) / (2 pi), as a 2^-64 fixed-point fraction
  for (int j = 0; j < 64; ++j) {
    const double f = std::pow(static_cast<double>(theta), -2.0 * j / 128.0) / (2.0 * 3.14159265358979323846);
    p.phase_inc[j] = static_cast<uint64_t>(std::ldexp(f, 64));
  }
  const int64_t t_max = int64_t(B) * c->d.n_kv_heads * np_max;
  const int grid = static_cast<int>(t_max < c->attn_grid ? t_max : c->attn_grid);
  return status_of(spkv::launch_attn(c, p, true, grid, as_stream(stream)));
}

static int rope_prefill(spkv_cache_t c, const void* q, int B, int T, int Hq, const int32_t* qpos0,
                        const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                        const int32_t* page_start, const int32_t* doc_pos, int max_docs, float theta, float* out,
                        float* lse, void* stream) {
  if (!c || B < 0 || T < 0 || Hq <= 0) return SPKV_EINVAL;
  const int Hk = c->d.n_kv_heads;
  if (Hq % Hk != 0) return SPKV_EINVAL;
  if (Hq / Hk > kMaxGroup) return SPKV_EUNSUPPORTED;
  if (B == 0 || T == 0) return SPKV_OK;
  if (!q || !qpos0 || !meta || !n_pages || !doc_pos || !out || !lse || np_max <= 0 || max_docs <= 0 ||
      !aligned(q, 16) || !aligned(out, 16))
    return SPKV_EINVAL;
  if (meta_heads != 1 && meta_heads != Hk) return SPKV_EINVAL;
  if (!(theta > 1.0f) || !std::isfinite(theta)) return SPKV_EINVAL;
  if (B > 65535 || Hq > 65535) return SPKV_EINVAL;
  spkv::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hk = Hk;
  p.G = Hq / Hk;
  p.n_phys = c->d.n_phys_pages;
  p.qpos0 = qpos0;
  p.meta = meta;
  p.meta_heads = meta_heads;
  p.n_pages = n_pages;
  p.np_max = np_max;
  p.doc_pos = doc_pos;
  p.max_docs = max_docs;
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(128.0));
  p.err = c->dev_err;
  p.page_start = page_start;
  p.causal = page_start != nullptr;
  for (int j = 0; j < 64; ++j) {
    const double f = std::pow(static_cast<double>(theta), -2.0 * j / 128.0) / (2.0 * 3.14159265358979323846);
    p.phase_inc[j] = static_cast<uint64_t>(std::ldexp(f, 64));
  }
  return status_of(spkv::launch_prefill(c, p, as_stream(stream)));
}

int lazy_rope_prefill_attn(spkv_cache_t c, const void* q, int B, int T, int Hq, const int32_t* qpos0,
                           const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                           const int32_t* doc_pos, int max_docs, float theta, float* out, float* lse, void* stream) {
  return rope_prefill(c, q, B, T, Hq, qpos0, meta, meta_heads, n_pages, np_max, nullptr, doc_pos, max_docs, theta,
                      out, lse, stream);
}

int lazy_rope_prefill_step(spkv_cache_t c, const void* q, int B, int T, int Hq, const int32_t* qpos0,
                           const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                           const int32_t* page_start, const int32_t* doc_pos, int max_docs, float theta, float* out,
                           float* lse, void* stream) {
  if (!page_start) return SPKV_EINVAL;
  return rope_prefill(c, q, B, T, Hq, qpos0, meta, meta_heads, n_pages, np_max, page_start, doc_pos, max_docs,
                      theta, out, lse, stream);
}

int lazy_alibi_prefill_attn(spkv_cache_t c, const void* q, int B, int T, int Hq, const int32_t* qpos0,
                            const uint32_t* meta, int meta_heads, const int32_t* n_pages, int np_max,
                            const int32_t* page_start, const int32_t* doc_pos, int max_docs, const float* slopes,
                            float* out, float* lse, void* stream) {
  if (!c || B < 0 || T < 0 || Hq <= 0) return SPKV_EINVAL;
  const int Hk = c->d.n_kv_heads;
  if (Hq % Hk != 0) return SPKV_EINVAL;
  if (Hq / Hk > kMaxGroup) return SPKV_EUNSUPPORTED;
  if (B == 0 || T == 0) return SPKV_OK;
  if (!q || !qpos0 || !meta || !n_pages || !page_start || !doc_pos || !slopes || !out || !lse || np_max <= 0 ||
      max_docs <= 0 || !aligned(q, 16) || !aligned(out, 16))
    return SPKV_EINVAL;
  if (meta_heads != 1 && meta_heads != Hk) return SPKV_EINVAL;
  if (B > 65535 || Hq > 65535) return SPKV_EINVAL;
  spkv::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hk = Hk;
  p.G = Hq / Hk;
  p.n_phys = c->d.n_phys_pages;
  p.qpos0 = qpos0;
  p.meta = meta;
  p.meta_heads = meta_heads;
  p.n_pages = n_pages;
  p.np_max = np_max;
  p.doc_pos = doc_pos;
  p.max_docs = max_docs;
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(128.0));
  p.err = c->dev_err;
  p.page_start = page_start;
  p.slopes = slopes;   // phase_inc stays zero: the query is never rotated
  return status_of(spkv::launch_prefill(c, p, as_stream(stream)));
}

static int column_scores(spkv_cache_t c, const void* q, const float* lse_in, int B, int alpha, int Hq,
                  const int32_t* page_table, int np_max, const int32_t* seq_len, float* scores, void* stream) {
  if (!c || B < 0 || Hq <= 0 || alpha < 0) return SPKV_EINVAL;
  const int Hk = c->d.n_kv_heads;
  if (Hq % Hk != 0) return SPKV_EINVAL;
  if (alpha > kMaxColumnRows || Hq / Hk > kMaxGroup) return SPKV_EUNSUPPORTED;
  if (B == 0) return SPKV_OK;
  if (!q || !page_table || !seq_len || !scores || np_max <= 0 || alpha == 0 || !aligned(q, 16)) return SPKV_EINVAL;
  if (B > 65535 || Hq > 65535) return SPKV_EINVAL;
  spkv::ColScoreParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.scores = scores;
  p.B = B;
  p.alpha = alpha;
  p.Hq = Hq;
  p.Hk = Hk;
  p.G = Hq / Hk;
  p.n_phys = c->d.n_phys_pages;
  p.page_table = page_table;
  p.np_max = np_max;
  p.seq_len = seq_len;
  p.lse_in = lse_in;
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(128.0));
  p.err = c->dev_err;
  // The keys-as-M probability kernel, 256 window rows per launch (later launches add in order),
  // from the caller's LSE or, without one, from a pass-1 launch of the row-major kernel that writes
  // each row's log2-domain LSE into the handle's split-K workspace (one stream per handle).  The
  // tile table of a launch lives in shared memory and counts tiles in 32 bits.
  const bool ws_fits = int64_t(B) * alpha * Hq <= int64_t(16) * 128 * c->ws_slots;
  if ((lse_in || ws_fits) && B <= spkv::colscore_lse_max_requests() &&
      int64_t(B) * Hq * ((int64_t(np_max) + 1) / 2) < (int64_t(1) << 31)) {
    CUtensorMap tmq;
    if (!encode_rows(&tmq, q, B, alpha, Hq)) return SPKV_ECUDA;
    if (!lse_in) {
      spkv::ColScoreParams p1 = p;
      p1.lse_out = c->ws_o;
      p1.row0 = 0;
      p1.rows = std::min(128, alpha);
      p1.chunks_in_grid = (alpha + 127) / 128;
      const int st = status_of(spkv::launch_colscore(c, p1, as_stream(stream)));
      if (st != SPKV_OK) return st;
      p.lse_in = c->ws_o;
      p.lse_is_log2 = 1;
    }
    const int64_t tiles = int64_t(B) * Hq * ((int64_t(np_max) + 1) / 2);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles, c->sm_count)));
    for (int r0 = 0; r0 < alpha; r0 += 256) {
      p.row0 = r0;
      p.rows = std::min(256, alpha - r0);
      p.accumulate = r0 > 0;
      const int st = status_of(spkv::launch_colscore_lse(c, p, tmq, grid, as_stream(stream)));
      if (st != SPKV_OK) return st;
    }
    return SPKV_OK;
  }
  // each row's softmax is its own, so the column sums of 128-row chunks of the window add.  Two
  // chunks run in one grid, adding atomically onto a zeroed result (two addends onto zero give
  // the same sum in either order); more run as one launch per chunk, later ones adding in order.
  if (alpha > 128 && alpha <= 256) {
    const size_t bytes = size_t(B) * Hq * size_t(np_max) * 64 * sizeof(float);
    if (cudaMemsetAsync(scores, 0, bytes, as_stream(stream)) != cudaSuccess) return SPKV_ECUDA;
    p.chunks_in_grid = 2;
    return status_of(spkv::launch_colscore(c, p, as_stream(stream)));
  }
  for (int r0 = 0; r0 < alpha; r0 += 128) {
    p.row0 = r0;
    p.rows = std::min(128, alpha - r0);
    p.accumulate = r0 > 0;
    const int st = status_of(spkv::launch_colscore(c, p, as_stream(stream)));
    if (st != SPKV_OK) return st;
  }
  return SPKV_OK;
}

int attn_column_scores(spkv_cache_t c, const void* q, int B, int alpha, int Hq, const int32_t* page_table,
                       int np_max, const int32_t* seq_len, float* scores, void* stream) {
  return column_scores(c, q, nullptr, B, alpha, Hq, page_table, np_max, seq_len, scores, stream);
}

int attn_column_scores_lse(spkv_cache_t c, const void* q, const float* lse, int B, int alpha, int Hq,
                           const int32_t* page_table, int np_max, const int32_t* seq_len, float* scores,
                           void* stream) {
  if (!lse) return SPKV_EINVAL;
  return column_scores(c, q, lse, B, alpha, Hq, page_table, np_max, seq_len, scores, stream);
}

int resident_setdiff(spkv_cache_t c, const int32_t* resident, int n_slots, const int32_t* sel, const int32_t* n_sel,
                     int sel_stride, int n_units, int32_t* missing, int32_t* n_missing, int32_t* slot, void* stream) {
  if (!c || n_units < 0) return SPKV_EINVAL;
  if (n_units == 0) return SPKV_OK;
  if (!resident || !sel || !n_sel || !missing || !n_missing || !slot) return SPKV_EINVAL;
  if (n_slots <= 0 || n_slots > 16384 || sel_stride <= 0 || sel_stride > 4096 || n_units > 65535) return SPKV_EINVAL;
  return status_of(spkv::launch_setdiff(c->dev_err, resident, n_slots, sel, n_sel, sel_stride, n_units, missing,
                                        n_missing, slot, as_stream(stream)));
}

int lru_bucket_update(spkv_cache_t c, int32_t* resident, int32_t* ts, int n_slots, const int32_t* slot,
                      const int32_t* n_sel, const int32_t* missing, const int32_t* n_missing, int sel_stride,
                      int n_units, int32_t t_now, int bucket_width, int32_t* victims, int32_t* hist, void* stream) {
  if (!c || n_units < 0) return SPKV_EINVAL;
  if (n_units == 0) return SPKV_OK;
  if (!resident || !ts || !slot || !n_sel || !missing || !n_missing || !victims || !hist) return SPKV_EINVAL;
  if (n_slots <= 0 || n_slots > 16384 || sel_stride <= 0 || sel_stride > 4096 || n_units > 65535 || bucket_width < 1)
    return SPKV_EINVAL;
  return status_of(spkv::launch_lru(c->dev_err, resident, ts, n_slots, slot, n_sel, missing, n_missing, sel_stride,
                                    n_units, t_now, bucket_width, victims, hist, as_stream(stream)));
}

static int retrieve_common(spkv_cache_t c, const void* k_host, const void* v_host, int64_t n_host_pages,
                           const int32_t* page_table, const spkv::PageDir* pd, int np_max, int B,
                           const int32_t* missing, const int32_t* n_missing, const int32_t* victims, int32_t* slot,
                           const int32_t* n_sel, int sel_stride, int n_slots, void* stream) {
  if (!c || B < 0) return SPKV_EINVAL;
  if (B == 0) return SPKV_OK;
  if (!k_host || !v_host || (!page_table && !pd) || !missing || !n_missing || !victims || !slot || !n_sel)
    return SPKV_EINVAL;
  if (!aligned(k_host, 16) || !aligned(v_host, 16)) return SPKV_EINVAL;
  if (n_host_pages <= 0 || np_max <= 0 || sel_stride <= 0 || sel_stride > 4096 || n_slots <= 0) return SPKV_EINVAL;
  if (int64_t(B) * c->d.n_kv_heads > c->max_units) return SPKV_EINVAL;
  if (int64_t(B) * n_slots > c->d.n_phys_pages) return SPKV_EINVAL;
  // device address of the mapped host pool (the same address under unified addressing);
  // looked up once per pool, so later calls (e.g. under stream capture) make no CUDA query
  if (k_host != c->host_k || v_host != c->host_v) {
    void* dk = nullptr;
    void* dv = nullptr;
    if (cudaHostGetDevicePointer(&dk, const_cast<void*>(k_host), 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&dv, const_cast<void*>(v_host), 0) != cudaSuccess) {
      cudaGetLastError();
      return SPKV_EINVAL;   // not pinned, device-mapped host memory
    }
    c->host_k = k_host;
    c->host_v = v_host;
    c->host_k_dev = dk;
    c->host_v_dev = dv;
  }
  return status_of(spkv::launch_retrieve(c, c->host_k_dev, c->host_v_dev, n_host_pages, page_table, np_max, B, missing, n_missing,
                                         victims, slot, n_sel, sel_stride, n_slots, as_stream(stream), pd));
}

int retrieve_pages(spkv_cache_t c, const void* k_host, const void* v_host, int64_t n_host_pages,
                   const int32_t* page_table, int np_max, int B, const int32_t* missing, const int32_t* n_missing,
                   const int32_t* victims, int32_t* slot, const int32_t* n_sel, int sel_stride, int n_slots,
                   void* stream) {
  if (!page_table) return SPKV_EINVAL;
  return retrieve_common(c, k_host, v_host, n_host_pages, page_table, nullptr, np_max, B, missing, n_missing, victims,
                         slot, n_sel, sel_stride, n_slots, stream);
}

int select_resident_update(spkv_cache_t c, const float* q_scores, const float* evict_scores, uint32_t* alive, int B,
                           int np_max, const int32_t* seq_len, int k_q, int k_e, int32_t* sel, int32_t* n_sel,
                           int32_t* resident, int32_t* ts, int n_slots, int32_t t_now, int bucket_width,
                           int32_t* missing, int32_t* n_missing, int32_t* slot, int32_t* victims, int32_t* hist,
                           void* stream) {
  if (!c || B < 0) return SPKV_EINVAL;
  const int64_t U = int64_t(B) * c->d.n_kv_heads;
  if (U > 65535) return SPKV_EINVAL;
  if (B == 0) return SPKV_OK;
  if (!q_scores || !evict_scores || !alive || !seq_len || !sel || !n_sel || !resident || !ts || !missing ||
      !n_missing || !slot || !victims || !hist)
    return SPKV_EINVAL;
  if (np_max <= 0 || np_max > 32768 || k_q < 0 || k_e < 0 || k_q + k_e + 1 > 4096) return SPKV_EINVAL;
  if (n_slots <= 0 || n_slots > 16384 || bucket_width < 1) return SPKV_EINVAL;
  cudaStream_t st = as_stream(stream);
  const int stride = k_q + k_e + 1;
  if (spkv::fused_supported(np_max))
    return status_of(spkv::launch_select_resident(c, q_scores, evict_scores, alive, B, np_max, seq_len, k_q, k_e,
                                                  sel, n_sel, resident, ts, n_slots, t_now, bucket_width, missing,
                                                  n_missing, slot, victims, hist, st));
  // longer contexts: the three kernels in turn (same results)
  cudaError_t e = spkv::launch_select(c, q_scores, evict_scores, alive, B, np_max, seq_len, k_q, k_e, sel, n_sel, st);
  if (e == cudaSuccess)
    e = spkv::launch_setdiff(c->dev_err, resident, n_slots, sel, n_sel, stride, static_cast<int>(U), missing,
                             n_missing, slot, st);
  if (e == cudaSuccess)
    e = spkv::launch_lru(c->dev_err, resident, ts, n_slots, slot, n_sel, missing, n_missing, stride,
                         static_cast<int>(U), t_now, bucket_width, victims, hist, st);
  return status_of(e);
}

// Checks a directory description and converts it to the kernels' view.
static int dir_view(const spkv_page_dir* d, int np_max, spkv::PageDir* out) {
  if (!d || !d->dir || d->seg_shift < 4 || d->seg_shift > 12 || d->chunk_shift < 0 || d->chunk_shift > 16 ||
      d->n_dev_segs < 0 || d->n_host_segs < 0 || (d->n_dev_segs > 0 && !d->dev_segs) ||
      (d->n_host_segs > 0 && !d->host_chunks))
    return SPKV_EINVAL;
  if (int64_t(d->n_dir) << d->seg_shift < np_max) return SPKV_EINVAL;   // the directory must cover np_max pages
  out->dir = d->dir;
  out->dev = d->dev_segs;
  out->chunks = d->host_chunks;
  out->n_dir = d->n_dir;
  out->shift = d->seg_shift;
  out->n_dev = d->n_dev_segs;
  out->chunk_shift = d->chunk_shift;
  out->n_host = d->n_host_segs;
  return SPKV_OK;
}

int score_blocks_dir(spkv_cache_t c, const void* q, int B, int Hq, const spkv_page_dir* dir, int np_max,
                     const int32_t* seq_len, float* scores, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (!c->d.ksum) return SPKV_EINVAL;
  if (B == 0) return SPKV_OK;
  if (!q || !seq_len || !scores || np_max <= 0 || !aligned(q, 8)) return SPKV_EINVAL;
  spkv::PageDir pd;
  if ((st = dir_view(dir, np_max, &pd)) != SPKV_OK) return st;
  return status_of(spkv::launch_score(c, q, B, Hq, nullptr, np_max, seq_len, scores, as_stream(stream), nullptr,
                                      nullptr, &pd));
}

int sparse_decode_attn_dir(spkv_cache_t c, const void* q, int B, int Hq, const spkv_page_dir* dir, int np_max,
                           const int32_t* sel, const int32_t* n_sel, int sel_stride, const int32_t* seq_len,
                           float* out, float* lse, void* stream) {
  int st = check_group(c, B, Hq);
  if (st != SPKV_OK) return st;
  if (B == 0) return SPKV_OK;
  if (!q || !sel || !n_sel || !seq_len || !out || !lse || np_max <= 0 || sel_stride <= 0 || !aligned(q, 16))
    return SPKV_EINVAL;
  AttnParams p;
  fill_common(p, c, q, B, Hq, out, lse);
  if ((st = dir_view(dir, np_max, &p.pd)) != SPKV_OK) return st;
  p.np_max = np_max;
  p.sel = sel;
  p.n_sel = n_sel;
  p.sel_stride = sel_stride;
  p.seq_len = seq_len;
  p.min_chunk = (sel_stride + 125) / 126;
  const int64_t t_max = int64_t(B) * c->d.n_kv_heads * sel_stride;
  const int grid = static_cast<int>(t_max < c->attn_grid ? t_max : c->attn_grid);
  return status_of(spkv::launch_attn(c, p, false, grid, as_stream(stream)));
}

int retrieve_pages_dir(spkv_cache_t c, const void* k_host, const void* v_host, int64_t n_host_pages,
                       const spkv_page_dir* dir, int np_max, int B, const int32_t* missing, const int32_t* n_missing,
                       const int32_t* victims, int32_t* slot, const int32_t* n_sel, int sel_stride, int n_slots,
                       void* stream) {
  spkv::PageDir pd;
  const int st = dir_view(dir, np_max, &pd);
  if (st != SPKV_OK) return st;
  return retrieve_common(c, k_host, v_host, n_host_pages, nullptr, &pd, np_max, B, missing, n_missing, victims, slot,
                         n_sel, sel_stride, n_slots, stream);
}

int spkv_pack_page_words(const int32_t* phys, const int32_t* valid, const int32_t* doc_slot, int64_t n,
                         uint32_t* words) {
  if (n < 0 || (n > 0 && (!phys || !valid || !doc_slot || !words))) return SPKV_EINVAL;
  for (int64_t i = 0; i < n; ++i) {
    if (phys[i] < 0 || phys[i] >= (1 << 18) || valid[i] < 1 || valid[i] > 64 || doc_slot[i] < 0 || doc_slot[i] > 255)
      return SPKV_EINVAL;
    words[i] = static_cast<uint32_t>(phys[i]) | (static_cast<uint32_t>(valid[i] - 1) << 18) |
               (static_cast<uint32_t>(doc_slot[i]) << 24);
  }
  return SPKV_OK;
}

int spkv_get_device_error(spkv_cache_t c, void* stream, uint32_t* bits) {
  if (!c || !bits) return SPKV_EINVAL;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return SPKV_ECUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, c->dev_err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SPKV_ECUDA;
  if (v && cudaMemset(c->dev_err, 0, sizeof(v)) != cudaSuccess) return SPKV_ECUDA;
  *bits = v;
  if (v & SPKV_DEVERR_TIMEOUT) return SPKV_ETIMEOUT;
  return v ? SPKV_EDEVICE : SPKV_OK;
}

}  // extern "C"
