// Document-major schedule of lazy-RoPE decode attention over shared cached documents.
//
// [Lazy] "LazyAttention", sections "Core idea: deferred positional encoding" (a cached document is
// reused at any position) and "Technical implementation 2. Decoding" (the query is rotated once per
// document by its relative offset).  When many requests hold the same cached document, attention
// per request reads that document's pages once per request; grouped by document, a job streams
// the pages once for the query rows of up to 16 / G requests (each rotated by its own offset), so
// the bytes read fall from one copy per (request, head) towards one copy per (document, head).
//
// The plan depends only on which documents each request holds, so it is built once on the host
// for a batch composition and reused by every decode step of that batch:
//   occurrences  every (request b, document slot i) with a document, grouped by document;
//   jobs         per document, per kv head, chunks of up to 16 / G occurrences; documents with
//                more pages first, so the longest jobs start early;
//   partials     one (max, sum, O) record per (occurrence, query head), merged per request.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "internal.h"

struct spkv_doc_plan {
  int B = 0, Hq = 0, Hk = 0, G = 0, max_docs = 0, n_docs = 0, n_jobs = 0, n_occ = 0;
  int4* jobs = nullptr;
  int2* occ = nullptr;
  int32_t* req_occ = nullptr;
  float* part_m = nullptr;
  float* part_l = nullptr;
  float* part_o = nullptr;
  int32_t* ctl = nullptr;
};

namespace {

void release(spkv_doc_plan* pl) {
  cudaFree(pl->jobs);
  cudaFree(pl->occ);
  cudaFree(pl->req_occ);
  cudaFree(pl->part_m);
  cudaFree(pl->part_l);
  cudaFree(pl->part_o);
  cudaFree(pl->ctl);
  delete pl;
}

}  // namespace

extern "C" {

int lazy_docs_plan_create(spkv_cache_t c, int B, int Hq, const int32_t* req_docs, int max_docs, int n_docs,
                          const int32_t* doc_first, spkv_doc_plan_t* out) {
  if (!out) return SPKV_EINVAL;
  *out = nullptr;
  if (!c || B <= 0 || Hq <= 0 || max_docs <= 0 || n_docs <= 0 || !req_docs || !doc_first) return SPKV_EINVAL;
  const int Hk = c->d.n_kv_heads;
  if (Hq % Hk != 0) return SPKV_EINVAL;
  const int G = Hq / Hk;
  if (G > 16) return SPKV_EUNSUPPORTED;
  if (int64_t(B) * max_docs > (int64_t(1) << 24)) return SPKV_EINVAL;
  for (int d = 0; d < n_docs; ++d)
    if (doc_first[d] < 0 || doc_first[d + 1] < doc_first[d]) return SPKV_EINVAL;
  std::vector<int32_t> count(n_docs, 0);
  for (int64_t k = 0; k < int64_t(B) * max_docs; ++k) {
    const int d = req_docs[k];
    if (d < -1 || d >= n_docs) return SPKV_EINVAL;
    if (d >= 0) ++count[d];
  }
  // occurrences grouped by document, (request, slot) ascending inside a document
  std::vector<int32_t> first(n_docs + 1, 0);
  for (int d = 0; d < n_docs; ++d) first[d + 1] = first[d] + count[d];
  const int n_occ = first[n_docs];
  std::vector<int2> occ(std::max(n_occ, 1));
  std::vector<int32_t> req_occ(int64_t(B) * max_docs, -1);
  std::vector<int32_t> fill(first.begin(), first.end() - 1);
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < max_docs; ++i) {
      const int d = req_docs[int64_t(b) * max_docs + i];
      if (d < 0) continue;
      const int o = fill[d]++;
      occ[o] = make_int2(b, i);
      req_occ[int64_t(b) * max_docs + i] = o;
    }
  // jobs: documents with more pages first; per document, kv head major, chunks of opj occurrences
  const int opj = std::max(1, 16 / G);
  std::vector<int> order(n_docs);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return doc_first[a + 1] - doc_first[a] > doc_first[b + 1] - doc_first[b];
  });
  std::vector<int4> jobs;
  for (int d : order) {
    if (count[d] == 0) continue;
    for (int h = 0; h < Hk; ++h)
      for (int o = 0; o < count[d]; o += opj) jobs.push_back(make_int4(d, h, first[d] + o, std::min(opj, count[d] - o)));
  }
  spkv_doc_plan* pl = new (std::nothrow) spkv_doc_plan();
  if (!pl) return SPKV_ENOMEM;
  pl->B = B;
  pl->Hq = Hq;
  pl->Hk = Hk;
  pl->G = G;
  pl->max_docs = max_docs;
  pl->n_docs = n_docs;
  pl->n_jobs = static_cast<int>(jobs.size());
  pl->n_occ = n_occ;
  const size_t rows = size_t(std::max(n_occ, 1)) * Hq;
  bool ok = cudaMalloc(&pl->jobs, std::max<size_t>(jobs.size(), 1) * sizeof(int4)) == cudaSuccess &&
            cudaMalloc(&pl->occ, occ.size() * sizeof(int2)) == cudaSuccess &&
            cudaMalloc(&pl->req_occ, req_occ.size() * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&pl->part_m, rows * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&pl->part_l, rows * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&pl->part_o, rows * 128 * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&pl->ctl, 2 * sizeof(int32_t)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release(pl);
    return SPKV_ENOMEM;
  }
  if ((!jobs.empty() && cudaMemcpy(pl->jobs, jobs.data(), jobs.size() * sizeof(int4), cudaMemcpyHostToDevice) !=
                            cudaSuccess) ||
      cudaMemcpy(pl->occ, occ.data(), occ.size() * sizeof(int2), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(pl->req_occ, req_occ.data(), req_occ.size() * sizeof(int32_t), cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemset(pl->ctl, 0, 2 * sizeof(int32_t)) != cudaSuccess) {
    release(pl);
    return SPKV_ECUDA;
  }
  *out = pl;
  return SPKV_OK;
}

int lazy_docs_plan_jobs(spkv_doc_plan_t pl) { return pl ? pl->n_jobs : SPKV_EINVAL; }

int lazy_docs_plan_destroy(spkv_doc_plan_t pl) {
  if (!pl) return SPKV_EINVAL;
  release(pl);
  return SPKV_OK;
}

int lazy_rope_decode_attn_docs(spkv_cache_t c, spkv_doc_plan_t pl, const void* q, const int32_t* qpos,
                               const uint32_t* doc_pages, const int32_t* doc_first, const int32_t* doc_pos,
                               float theta, float* out, float* lse, void* stream) {
  if (!c || !pl || !q || !qpos || !doc_pages || !doc_first || !doc_pos || !out || !lse) return SPKV_EINVAL;
  if (pl->Hk != c->d.n_kv_heads || (reinterpret_cast<uintptr_t>(q) % 16) != 0) return SPKV_EINVAL;
  if (!(theta > 1.0f) || !std::isfinite(theta)) return SPKV_EINVAL;
  spkv::AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.B = pl->B;
  p.Hq = pl->Hq;
  p.Hk = pl->Hk;
  p.G = pl->G;
  p.n_phys = c->d.n_phys_pages;
  p.err = c->dev_err;
  p.ws_ctl = pl->ctl;
  p.qpos = qpos;
  p.doc_pos = doc_pos;
  p.max_docs = pl->max_docs;
  p.jobs = pl->jobs;
  p.n_jobs = pl->n_jobs;
  p.occ = pl->occ;
  p.req_occ = pl->req_occ;
  p.doc_pages = doc_pages;
  p.doc_first = doc_first;
  p.part_m = pl->part_m;
  p.part_l = pl->part_l;
  p.part_o = pl->part_o;
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(128.0));
  p.wait_ns = c->wait_ns;
  for (int j = 0; j < 64; ++j) {
    const double f = std::pow(static_cast<double>(theta), -2.0 * j / 128.0) / (2.0 * 3.14159265358979323846);
    p.phase_inc[j] = static_cast<uint64_t>(std::ldexp(f, 64));
  }
  const int grid = std::max(1, std::min(pl->n_jobs, c->attn_grid));
  return spkv::launch_attn_docs(c, p, grid, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPKV_OK : SPKV_ECUDA;
}

}  // extern "C"
