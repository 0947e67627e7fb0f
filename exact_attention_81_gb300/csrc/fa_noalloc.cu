// fa_noalloc.cu -- split-KV decode for callers that cannot allocate device memory.
//
// fa_fwd_kvcache needs a caller-owned workspace for the per-split partial outputs.  Some
// callers have no way to provide one: code running as a plugin inside another runtime that
// hands it no workspace, or a serving loop that keeps cudaMalloc (which can synchronise
// the whole device) out of its decode step and has no buffer set aside for this call.
// fa_fwd_kvcache_noalloc serves them by writing the partials to a scratch array compiled
// into the library instead.
//
// The scratch is a file-scope __device__ array of FA_NOALLOC_SCRATCH_BYTES.  Host code
// cannot use the array's name as a device address, so on the first call on each device
// (with that device current) the address is looked up once with cudaGetSymbolAddress and
// cached per device; that first call should therefore be made before any stream capture.
// Every call on a device shares the one array and finds the previous call's contents in
// it.  Nothing in it has to start at zero -- every partial a call reads was written by the
// same call -- but two calls that overlap on the GPU race on it.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
fa_status scratch_for_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_fwd_kvcache_noalloc(const void *q, const void *k_cache,
                                            const void *v_cache, const int *cache_seqlens,
                                            int B, int Lmax, int Hq, int Hkv, int d,
                                            const int64_t cache_strides[3], float scale,
                                            int num_splits, void *o, float *lse,
                                            cudaStream_t stream) {
  // Sizes, head dimension and pointers are validated by fa_fwd_kvcache; only the scratch
  // bound is checked here, before the array's address is looked up.
  if (B < 0 || Lmax < 0 || Hq <= 0 || Hkv <= 0 || num_splits < 0) return FA_ERR_INVALID_ARG;
  if (B == 0) return FA_OK;
  const size_t need = Lmax > 0 ? fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits) : 0;
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_WORKSPACE;
  void *scratch = nullptr;
  const fa_status st = scratch_for_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, B, Lmax, Hq, Hkv, d, cache_strides,
                        scale, num_splits, scratch, FA_NOALLOC_SCRATCH_BYTES, o, lse, FA_BF16, nullptr, nullptr,
                        stream);
}
