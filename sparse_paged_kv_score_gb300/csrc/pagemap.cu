// Host-side manager of a two-level page directory.
//
// [Spin] "Unifying Sparse Attention with Hierarchical Memory for Scalable Long-Context LLM Serving",
// section 2C "Hierarchical metadata management": a small top-level directory stays on the GPU and
// points to second-level segments allocated on demand in CPU memory, so metadata follows the pages in
// use instead of the logical address space; latency-critical metadata stays on the GPU (the directory
// and a cache of hot segments) and bulk metadata lives in host memory (tier separation).
//
// State:
//   * a pinned host mirror of the directory, [B][n_dir] entries in the encoding of spkv_page_dir
//     (>= 0 device slot, <= -2 host segment -2 - e, -1 unmapped); it is the authoritative copy and
//     spkv_pagemap_sync copies it to the device directory;
//   * host segments: every mapped segment has one, in pinned host memory mapped into the device
//     address space, allocated in chunks of 2^chunk_shift segments the first time a page of the
//     segment's range is mapped; the kernels read host-tier segments in place;
//   * device slots: n_dev_segs segments of device memory holding copies of promoted segments; a
//     slot whose host segment changed (or that was just promoted) is copied again at the next sync.
// Nothing here runs on the GPU except the copies that spkv_pagemap_sync enqueues.
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"

struct spkv_pagemap {
  int B = 0, np_max = 0, shift = 0, seg = 0, n_dir = 0, n_dev = 0, chunk_shift = 6;
  int32_t* h_dir = nullptr;           // pinned host mirror [B][n_dir]
  int32_t* d_dir = nullptr;           // device directory [B][n_dir]
  int32_t* d_segs = nullptr;          // device slots [n_dev][seg]
  int32_t** d_chunks = nullptr;       // device chunk table [max_chunks]
  int32_t** h_chunk_dev = nullptr;    // pinned host copy of the chunk table (device addresses)
  int max_chunks = 0;
  std::vector<int32_t*> chunks;       // host addresses of the chunks
  int64_t n_host = 0;                 // host segments handed out
  std::vector<int32_t> host_of;       // [B * n_dir]: host segment of (b, s), -1 if unmapped
  std::vector<int32_t> owner;         // [n_dev]: b * n_dir + s held by the slot, or -1
  std::vector<int64_t> stamp;         // [n_dev]: promotion time (the oldest slot is reused first)
  std::vector<char> dirty;            // [n_dev]: copy the host segment into the slot at the next sync
  bool dir_dirty = true, chunks_dirty = false;
  int64_t clock = 0;
};

namespace {

int32_t* host_segment(spkv_pagemap* pm, int64_t h) {
  return pm->chunks[h >> pm->chunk_shift] + ((h & ((int64_t(1) << pm->chunk_shift) - 1)) << pm->shift);
}

void release(spkv_pagemap* pm) {
  cudaFreeHost(pm->h_dir);
  cudaFreeHost(pm->h_chunk_dev);
  cudaFree(pm->d_dir);
  cudaFree(pm->d_segs);
  cudaFree(pm->d_chunks);
  for (int32_t* c : pm->chunks) cudaFreeHost(c);
  delete pm;
}

// Host segment of (b, s), allocated (filled with -1, i.e. unmapped pages) when it has none yet.
int64_t ensure_host_segment(spkv_pagemap* pm, int b, int s) {
  const int64_t key = int64_t(b) * pm->n_dir + s;
  if (pm->host_of[key] >= 0) return pm->host_of[key];
  const int64_t h = pm->n_host;
  if ((h >> pm->chunk_shift) >= static_cast<int64_t>(pm->chunks.size())) {
    if (static_cast<int>(pm->chunks.size()) >= pm->max_chunks) return -1;
    void* p = nullptr;
    const size_t bytes = (size_t(1) << pm->chunk_shift) * pm->seg * sizeof(int32_t);
    if (cudaHostAlloc(&p, bytes, cudaHostAllocMapped) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, p, 0) != cudaSuccess) {
      cudaGetLastError();
      cudaFreeHost(p);
      return -1;
    }
    pm->h_chunk_dev[pm->chunks.size()] = static_cast<int32_t*>(dp);
    pm->chunks.push_back(static_cast<int32_t*>(p));
    pm->chunks_dirty = true;
  }
  ++pm->n_host;
  int32_t* seg = host_segment(pm, h);
  for (int i = 0; i < pm->seg; ++i) seg[i] = -1;
  pm->host_of[key] = static_cast<int32_t>(h);
  if (pm->h_dir[key] == -1) {
    pm->h_dir[key] = static_cast<int32_t>(-2 - h);
    pm->dir_dirty = true;
  }
  return h;
}

}  // namespace

extern "C" {

int spkv_pagemap_create(int B, int np_max, int seg_shift, int n_dev_segs, spkv_pagemap_t* out) {
  if (!out) return SPKV_EINVAL;
  *out = nullptr;
  if (B <= 0 || np_max <= 0 || seg_shift < 4 || seg_shift > 12 || n_dev_segs < 0) return SPKV_EINVAL;
  spkv_pagemap* pm = new (std::nothrow) spkv_pagemap();
  if (!pm) return SPKV_ENOMEM;
  pm->B = B;
  pm->np_max = np_max;
  pm->shift = seg_shift;
  pm->seg = 1 << seg_shift;
  pm->n_dir = (np_max + pm->seg - 1) / pm->seg;
  pm->n_dev = n_dev_segs;
  const int64_t entries = int64_t(B) * pm->n_dir;
  // host segments are numbered in 31 bits (directory entry -2 - h); chunks cover all of them
  pm->max_chunks = static_cast<int>((entries + (int64_t(1) << pm->chunk_shift) - 1) >> pm->chunk_shift);
  try {
    pm->host_of.assign(entries, -1);
    pm->owner.assign(n_dev_segs, -1);
    pm->stamp.assign(n_dev_segs, 0);
    pm->dirty.assign(n_dev_segs, 0);
  } catch (...) {
    delete pm;
    return SPKV_ENOMEM;
  }
  bool ok = cudaHostAlloc(reinterpret_cast<void**>(&pm->h_dir), entries * sizeof(int32_t), cudaHostAllocDefault) ==
                cudaSuccess &&
            cudaHostAlloc(reinterpret_cast<void**>(&pm->h_chunk_dev), pm->max_chunks * sizeof(int32_t*),
                          cudaHostAllocDefault) == cudaSuccess &&
            cudaMalloc(&pm->d_dir, entries * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&pm->d_chunks), pm->max_chunks * sizeof(int32_t*)) == cudaSuccess &&
            (n_dev_segs == 0 ||
             cudaMalloc(&pm->d_segs, size_t(n_dev_segs) * pm->seg * sizeof(int32_t)) == cudaSuccess);
  if (!ok) {
    cudaGetLastError();
    release(pm);
    return SPKV_ENOMEM;
  }
  for (int64_t i = 0; i < entries; ++i) pm->h_dir[i] = -1;
  std::memset(pm->h_chunk_dev, 0, pm->max_chunks * sizeof(int32_t*));
  *out = pm;
  return SPKV_OK;
}

int spkv_pagemap_map(spkv_pagemap_t pm, int b, int first_page, int n, const int32_t* phys) {
  if (!pm || b < 0 || b >= pm->B || first_page < 0 || n < 0 || int64_t(first_page) + n > pm->np_max) return SPKV_EINVAL;
  if (n > 0 && !phys) return SPKV_EINVAL;
  for (int i = 0; i < n; ++i) {
    const int p = first_page + i;
    const int s = p >> pm->shift;
    const int64_t key = int64_t(b) * pm->n_dir + s;
    if (phys[i] < 0 && pm->host_of[key] < 0) continue;   // unmapping a page of an unmapped segment
    const int64_t h = ensure_host_segment(pm, b, s);
    if (h < 0) return SPKV_ENOMEM;
    host_segment(pm, h)[p & (pm->seg - 1)] = phys[i] < 0 ? -1 : phys[i];
    const int32_t e = pm->h_dir[key];
    if (e >= 0) pm->dirty[e] = 1;                        // its device copy is refreshed at the next sync
  }
  return SPKV_OK;
}

int spkv_pagemap_promote(spkv_pagemap_t pm, int b, int page) {
  if (!pm || b < 0 || b >= pm->B || page < 0 || page >= pm->np_max) return SPKV_EINVAL;
  const int64_t key = int64_t(b) * pm->n_dir + (page >> pm->shift);
  if (pm->host_of[key] < 0 || pm->n_dev == 0) return SPKV_EINVAL;
  const int32_t e = pm->h_dir[key];
  if (e >= 0) {
    pm->stamp[e] = ++pm->clock;
    return SPKV_OK;
  }
  int slot = -1;
  for (int i = 0; i < pm->n_dev && slot < 0; ++i)
    if (pm->owner[i] < 0) slot = i;
  if (slot < 0) {   // reuse the slot promoted longest ago; its segment returns to the host tier
    slot = 0;
    for (int i = 1; i < pm->n_dev; ++i)
      if (pm->stamp[i] < pm->stamp[slot]) slot = i;
    const int64_t old = pm->owner[slot];
    pm->h_dir[old] = static_cast<int32_t>(-2 - int64_t(pm->host_of[old]));
  }
  pm->owner[slot] = static_cast<int32_t>(key);
  pm->stamp[slot] = ++pm->clock;
  pm->dirty[slot] = 1;
  pm->h_dir[key] = slot;
  pm->dir_dirty = true;
  return SPKV_OK;
}

int spkv_pagemap_sync(spkv_pagemap_t pm, void* stream) {
  if (!pm) return SPKV_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < pm->n_dev && e == cudaSuccess; ++i) {
    if (!pm->dirty[i] || pm->owner[i] < 0) continue;
    e = cudaMemcpyAsync(pm->d_segs + size_t(i) * pm->seg, host_segment(pm, pm->host_of[pm->owner[i]]),
                        pm->seg * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  }
  if (e == cudaSuccess && pm->chunks_dirty)
    e = cudaMemcpyAsync(pm->d_chunks, pm->h_chunk_dev, pm->chunks.size() * sizeof(int32_t*), cudaMemcpyHostToDevice,
                        st);
  if (e == cudaSuccess && pm->dir_dirty)
    e = cudaMemcpyAsync(pm->d_dir, pm->h_dir, int64_t(pm->B) * pm->n_dir * sizeof(int32_t), cudaMemcpyHostToDevice,
                        st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SPKV_ECUDA;
  }
  for (int i = 0; i < pm->n_dev; ++i) pm->dirty[i] = 0;
  pm->dir_dirty = pm->chunks_dirty = false;
  return SPKV_OK;
}

int spkv_pagemap_view(spkv_pagemap_t pm, spkv_page_dir* out) {
  if (!pm || !out) return SPKV_EINVAL;
  out->dir = pm->d_dir;
  out->dev_segs = pm->d_segs;
  out->host_chunks = pm->d_chunks;
  out->n_dir = pm->n_dir;
  out->seg_shift = pm->shift;
  out->n_dev_segs = pm->n_dev;
  out->chunk_shift = pm->chunk_shift;
  out->n_host_segs = pm->n_host;
  return SPKV_OK;
}

int spkv_pagemap_bytes(spkv_pagemap_t pm, int64_t* device_bytes, int64_t* host_bytes) {
  if (!pm || !device_bytes || !host_bytes) return SPKV_EINVAL;
  *device_bytes = int64_t(pm->B) * pm->n_dir * 4 + int64_t(pm->n_dev) * pm->seg * 4 +
                  int64_t(pm->max_chunks) * static_cast<int64_t>(sizeof(int32_t*));
  *host_bytes = static_cast<int64_t>(pm->chunks.size()) * (int64_t(1) << pm->chunk_shift) * pm->seg * 4;
  return SPKV_OK;
}

int spkv_pagemap_destroy(spkv_pagemap_t pm) {
  if (!pm) return SPKV_EINVAL;
  release(pm);
  return SPKV_OK;
}

}  // extern "C"
