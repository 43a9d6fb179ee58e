// sta_decode_splitkv_noalloc: split-KV decode for callers that cannot allocate
// device memory. The partial results live in one fixed array in the library's
// own device memory instead of a caller workspace; everything else is the
// ordinary split-KV decode path (same kernels, same plan).
#include <mutex>

#include "internal.h"

namespace sta {
namespace {

// Scratch for the partial outputs and LSEs: 16 MiB, resident on every GPU that
// loads the library until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, looked up once per device (with that
// device current) and cached. In host code the array's name only stands in for
// the symbol; the address a kernel may use comes from cudaGetSymbolAddress.
sta_status noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return STA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return STA_ERR_CUDA;
    cached[dev] = p;
  }
  *ptr = cached[dev];
  return STA_OK;
}

inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace sta

using namespace sta;

extern "C" sta_status sta_decode_splitkv_noalloc(const void* q, const void* k, const void* v,
                                                 const int32_t* kv_indptr_dev, const int32_t* kv_indptr_host,
                                                 int n_req, int Hq, int Hkv, int d, sta_dtype dtype, float scale,
                                                 int num_splits, void* o, float* lse, sta_stream stream) {
  if (!(scale > 0.f) || !isfinite(scale)) return STA_ERR_INVALID_ARG;
  DecodeArgs a;
  int64_t T = 0;
  sta_status st = decode_setup(kv_indptr_host, n_req, Hq, Hkv, d, dtype, num_splits, a, T);
  if (st != STA_OK) return st;
  const size_t slots = decode_slots(a);
  const size_t o_bytes = round256(slots * (size_t)Hq * d * sizeof(float));
  const size_t need = o_bytes + round256(slots * (size_t)Hq * sizeof(float));
  if (need > kNoAllocScratchBytes) return STA_ERR_WORKSPACE;  // beyond the fixed scratch
  if (!q || !kv_indptr_dev || !o) return STA_ERR_INVALID_ARG;
  if (T > 0 && (!k || !v)) return STA_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15u) || ((uintptr_t)k & 15u) || ((uintptr_t)v & 15u) || ((uintptr_t)o & 15u))
    return STA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != STA_OK) return st;
  a.q = q; a.k = k; a.v = v; a.kv_indptr = kv_indptr_dev; a.o = o; a.lse = lse;
  a.part_o = static_cast<float*>(scratch);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(scratch) + o_bytes);
  a.scale_log2 = scale * kLog2e;
  a.err = device_error_word();
  return launch_decode(a, (cudaStream_t)stream);
}
