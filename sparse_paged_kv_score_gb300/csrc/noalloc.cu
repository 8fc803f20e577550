// sparse_decode_attn_noalloc: the split-K sparse decode attention of sparse_decode_attn, for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is unavailable or not allowed -- for example an
// inference engine that hands the library a fixed memory budget and forbids allocation after
// start-up, a host runtime whose allocator is owned by another framework, or a caller that
// must not create a library handle (paged_kv_create allocates the handle's workspace).  Such a
// caller still owns and passes every input and output; the only memory this entry point needs
// beyond them is the split-K scratch (per-CTA partial results and per-unit arrival counters),
// and that lives in the fixed-size device array below, which exists from the moment the library
// is loaded on a device until the process exits.
//
// Contract (also stated in include/spkv.h):
//   * at most SPKV_NOALLOC_MAX_UNITS (request, kv head) units and group size <= 16; larger calls
//     return SPKV_EUNSUPPORTED before launching anything;
//   * the first call on a device looks up the array's device address (cudaGetSymbolAddress)
//     with that device current, so make that first call before any stream capture;
//   * all calls on a device share the one array and it keeps the last call's contents; the
//     chunk counter is cleared at the start of every call, and every call rewrites the per-unit
//     partial records before reading them;
//     two calls whose kernels overlap on the GPU (different streams, no ordering) race on it;
//   * the caller's error word is required: a page id or physical page out of range is skipped
//     and reported only there, so a call that could not report it would hand back wrong
//     results with SPKV_OK;
//   * every device pointer must belong to the current device (checked with
//     cudaPointerGetAttributes, a lookup that allocates nothing): the scratch address, kernel
//     attributes and tensor maps all follow the current device;
//   * nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kSlots = int64_t(2 * SPKV_NOALLOC_MAX_CTAS) + SPKV_NOALLOC_MAX_UNITS;
// Byte layout of the scratch array (each region 256-byte aligned).
constexpr int64_t kOffCtl = 0;     // the chunk counter (first word); the rest of the region is unused
constexpr int64_t kOffCnt = 256;
constexpr int64_t kOffM = kOffCnt + ((SPKV_NOALLOC_MAX_UNITS * 8 + 255) / 256) * 256;
constexpr int64_t kOffL = kOffM + kSlots * 16 * 4;
constexpr int64_t kOffO = kOffL + kSlots * 16 * 4;
constexpr int64_t kScratchBytes = kOffO + kSlots * 16 * 128 * 4;
static_assert(kScratchBytes == SPKV_NOALLOC_SCRATCH_BYTES, "header constant out of date");

}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the device object; the
// kernel gets the device address found by cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `dev` (looked up once per device, `dev` current); the
// same first call sets the attention kernel's shared-memory limit on that device.
cudaError_t scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    cudaError_t e = spkv::attn_init_attributes();
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_addr[dev]);
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// True when p is device (or managed) memory of device `dev`.  Host memory, unregistered or
// pinned, and another device's memory are refused.
bool on_device(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev;
}

bool encode(CUtensorMap* m, const void* base, int64_t n_page_heads) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, 64, static_cast<cuuint64_t>(n_page_heads)};
  cuuint64_t strides[2] = {256, 16384};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int sparse_decode_attn_noalloc(const void* k_pool, const void* v_pool, int n_kv_heads,
                                          int64_t n_phys_pages, const void* q, int B, int Hq,
                                          const int32_t* page_table, int np_max, const int32_t* sel,
                                          const int32_t* n_sel, int sel_stride, const int32_t* seq_len,
                                          float* out, float* lse, uint32_t* dev_err, void* stream) {
  if (!k_pool || !v_pool || !q || !page_table || !sel || !n_sel || !seq_len || !out || !lse || !dev_err)
    return SPKV_EINVAL;
  if (n_kv_heads <= 0 || n_phys_pages <= 0 || B < 0 || Hq <= 0 || np_max <= 0 || sel_stride <= 0)
    return SPKV_EINVAL;
  if (Hq % n_kv_heads != 0) return SPKV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(q) % 16 != 0)
    return SPKV_EINVAL;
  const int G = Hq / n_kv_heads;
  const int64_t n_ph = int64_t(n_kv_heads) * n_phys_pages;
  if (G > 16 || int64_t(B) * n_kv_heads > SPKV_NOALLOC_MAX_UNITS || n_ph >= (int64_t(1) << 31))
    return SPKV_EUNSUPPORTED;
  if (B == 0) return SPKV_OK;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPKV_ECUDA;
  for (const void* ptr : {k_pool, v_pool, q, static_cast<const void*>(page_table), static_cast<const void*>(sel),
                          static_cast<const void*>(n_sel), static_cast<const void*>(seq_len),
                          static_cast<const void*>(out), static_cast<const void*>(lse),
                          static_cast<const void*>(dev_err)})
    if (!on_device(ptr, dev)) return SPKV_EINVAL;
  unsigned char* base = nullptr;
  if (scratch_address(dev, &base) != cudaSuccess) return SPKV_ECUDA;

  spkv_cache c;  // host-side description only (tensor maps); owns no memory
  std::memset(&c.d, 0, sizeof(c.d));
  c.d.n_kv_heads = n_kv_heads;
  c.d.n_phys_pages = n_phys_pages;
  if (!encode(&c.tmap_k, k_pool, n_ph) || !encode(&c.tmap_v, v_pool, n_ph)) return SPKV_ECUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* cnt = reinterpret_cast<int32_t*>(base + kOffCnt);
  const int64_t units = int64_t(B) * n_kv_heads;
  if (cudaMemsetAsync(base + kOffCtl, 0, 2 * sizeof(int32_t), st) != cudaSuccess) return SPKV_ECUDA;

  spkv::AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hk = n_kv_heads;
  p.G = G;
  p.n_phys = n_phys_pages;
  p.err = dev_err;
  p.ws_m = reinterpret_cast<float*>(base + kOffM);
  p.ws_l = reinterpret_cast<float*>(base + kOffL);
  p.ws_o = reinterpret_cast<float*>(base + kOffO);
  p.ws_parts = cnt;
  p.ws_ctl = reinterpret_cast<int32_t*>(base + kOffCtl);
  p.max_chunks = 2 * SPKV_NOALLOC_MAX_CTAS;
  p.min_chunk = (sel_stride + 125) / 126;
  p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(128.0));
  p.wait_ns = 1000000000ull;
  p.page_table = page_table;
  p.np_max = np_max;
  p.sel = sel;
  p.n_sel = n_sel;
  p.sel_stride = sel_stride;
  p.seq_len = seq_len;
  const int64_t t_max = units * sel_stride;
  int64_t grid = sms < SPKV_NOALLOC_MAX_CTAS ? sms : SPKV_NOALLOC_MAX_CTAS;
  if (t_max < grid) grid = t_max;
  return spkv::launch_attn(&c, p, false, static_cast<int>(grid), st) == cudaSuccess ? SPKV_OK : SPKV_ECUDA;
}
