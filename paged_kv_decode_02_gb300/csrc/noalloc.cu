// noalloc.cu -- bf16 paged decode for callers that cannot allocate device memory.
//
// pkv_decode_bf16 needs a caller-provided workspace for its split-KV partials and
// its per-sequence block prefix. Some callers have no allocator to give it: code
// running inside another runtime's memory pool, plugins that may not call
// cudaMalloc, or latency-critical paths where no allocation may happen. For
// them pkv_decode_bf16_noalloc uses a fixed scratch array that lives in this
// library's own device image instead, so the call allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv.h"

// The scratch itself: PKV_NOALLOC_SCRATCH_BYTES of device memory on every GPU that
// loads the library, held until the process exits. Host code must not use this name
// as a device address (on the host it is only a stand-in); the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
pkv_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_bf16_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale,
                                              const pkv_dims* dims, int32_t* status,
                                              pkv_stream_t stream) {
  if (!dims) return PKV_ERR_NULL;
  size_t need = 0;
  pkv_status st = pkv_decode_workspace_bytes(dims, PKV_KV_BF16, &need);
  if (st != PKV_OK) return st;
  if (need > size_t(PKV_NOALLOC_SCRATCH_BYTES)) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != PKV_OK) return st;
  // Nothing in the scratch has to start at zero: the decode writes the block prefix
  // and every partial before anything reads them.
  return pkv_decode_bf16(out, q, k_cache, v_cache, block_tables, context_lens, scale, dims,
                         scratch, size_t(PKV_NOALLOC_SCRATCH_BYTES), status, stream);
}
