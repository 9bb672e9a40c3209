// decode_noalloc.cu -- single-token decode for callers that cannot allocate
// device memory.
//
// Some callers of this library have no way to obtain scratch memory: code
// that runs where cudaMalloc is forbidden or unavailable, such as a host
// runtime that hands out only the input and output buffers it already owns,
// or a caller whose allocator is locked while its work is being queued.
// gqa_attn_decode needs a caller-provided workspace for the split-KV
// partials; this entry point instead uses one fixed scratch array compiled
// into the library.
//
// The array lives in device memory of every GPU that loads the library and
// stays there until the process exits.  Host code cannot use the array's name
// as a device address (on the host it names a host-side stand-in), so the
// device address is obtained once per device with cudaGetSymbolAddress, with
// that device current, during the first call made on it.  That first call
// should therefore be made before any stream capture begins.
//
// All calls share the one array, and each call leaves its contents behind.
// No byte of it needs to start at zero: every partial a call reads was
// written earlier in the same call, and the status word at its start only
// accumulates flags, which this entry point does not report.  Two calls whose
// work may overlap on the GPU (different streams, or different host threads)
// race on the array and give wrong results; serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "gqa_attn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = GQA_ATTN_NOALLOC_SCRATCH_BYTES;  // 16 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device and kept for the life of the process).  The cached
// address belongs to the device's primary context, the one the CUDA runtime
// uses; after cudaDeviceReset, or with another driver-API context current,
// it no longer names the array.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GQA_OK;
}

}  // namespace

extern "C" GQA_ATTN_API int gqa_attn_decode_noalloc(const void* q, const void* k, const void* v,
                                                    void* o, const int32_t* kv_lens, int B, int Hq,
                                                    int Hkv, int D, int S_cap, int max_kv_len,
                                                    float scale, int dtype, void* stream) {
  // the checks of gqa_attn_decode first, so that an invalid call gets the
  // same error code from both entry points
  const int valid = gqa::validate_decode_args(q, k, v, o, kv_lens, B, Hq, Hkv, D, S_cap, max_kv_len, scale,
                                              dtype);
  if (valid != GQA_OK) return valid;
  const size_t need = gqa_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, dtype);
  if (need == 0) return GQA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return GQA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != GQA_OK) return rc;
  return gqa_attn_decode(q, k, v, o, kv_lens, B, Hq, Hkv, D, S_cap, max_kv_len, scale, dtype,
                         scratch, kScratchBytes, stream);
}
