// noalloc.cu -- bf16 paged decode for callers that cannot allocate device memory.
//
// pkv_decode_bf16 needs a caller-provided workspace for its split-KV partials and
// its per-sequence block prefix. Some callers have no allocator to give it: code
// running inside another runtime's memory pool, plugins that may not call
// cudaMalloc, or latency-critical paths where no allocation may happen. For
// them pkv_decode_bf16_noalloc uses a fixed scratch array that lives in this
// library's own device image instead, so the call allocates nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "pagedkv.h"

// The scratch itself: PKV_NOALLOC_SCRATCH_BYTES of device memory on every GPU that
// loads the library, held until the process exits. Host code must not use this name
// as a device address (on the host it is only a stand-in); the address comes from
// cudaGetSymbolAddress below.
//
// Layout: the first PKV_NOALLOC_MAX_SEQ_HEADS 8-byte words hold the counters of the
// in-kernel split-KV fold and nothing else, whatever the shapes of earlier calls, so a
// counter word never meets a stale partial of another call; the rest is the decode
// workspace. Device memory of a module starts zeroed, and every call leaves its
// counters at zero (or, after a timed-out call, tagged with a launch that is over,
// which no later launch mistakes for its own).
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kCounterBytes = size_t(PKV_NOALLOC_MAX_SEQ_HEADS) * 8;
static_assert(kCounterBytes % 256 == 0 && kCounterBytes < PKV_NOALLOC_SCRATCH_BYTES,
              "counter region");
constexpr size_t kWorkspaceBytes = size_t(PKV_NOALLOC_SCRATCH_BYTES) - kCounterBytes;

constexpr int kMaxDevices = 64;

// The scratch address belongs to the context the module was loaded into, so it is
// kept per device together with the unique id of that context: after a device reset
// (a new primary context) or under another context made current on the device, the
// id differs and the address is looked up again.
struct ScratchAddr {
  unsigned long long ctx_id;  // 0: none yet
  void* ptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Unique id of the context current on this thread (0 when none is current yet).
pkv_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return PKV_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return PKV_ERR_CUDA;
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return PKV_ERR_CUDA;
  return PKV_OK;
}

// Device address of the scratch in the current context of the current device, looked
// up with cudaGetSymbolAddress the first time that context is seen.
pkv_status scratch_on_current_device(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  pkv_status st = current_context_id(&id);
  if (st != PKV_OK) return st;
  if (id == 0 || g_scratch[dev].ctx_id != id || g_scratch[dev].ptr == nullptr) {
    void* p = nullptr;
    // (makes the device's primary context current when no context is)
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    st = current_context_id(&id);
    if (st != PKV_OK) return st;
    if (id == 0) return PKV_ERR_CUDA;
    g_scratch[dev].ctx_id = id;
    g_scratch[dev].ptr = p;
  }
  *out = static_cast<unsigned char*>(g_scratch[dev].ptr);
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
  if (need > kWorkspaceBytes ||
      (long long)dims->num_seqs * dims->num_kv_heads > PKV_NOALLOC_MAX_SEQ_HEADS)
    return PKV_ERR_WORKSPACE;
  unsigned char* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != PKV_OK) return st;
  // Nothing in the scratch has to be cleared: the decode writes the block prefix and
  // every partial before anything reads them, and the counters are kept as above.
  return pkv::decode_bf16_fixed_counters(
      out, q, k_cache, v_cache, block_tables, context_lens, scale, dims,
      scratch + kCounterBytes, kWorkspaceBytes,
      reinterpret_cast<unsigned long long*>(scratch), size_t(PKV_NOALLOC_MAX_SEQ_HEADS), status,
      reinterpret_cast<cudaStream_t>(stream));
}
