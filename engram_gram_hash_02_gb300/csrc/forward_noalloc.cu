// engram_forward_noalloc: the whole path with its scratch in a static device array.
//
// For callers that may not allocate device memory: for instance a host program whose memory
// pool already owns every byte of device memory it may use (an inference engine that reserved
// HBM for its caches at start-up and hands plugins only the tensors it owns), or a real-time
// loop that cannot afford cudaMalloc's implicit device-wide synchronisation. Such a caller
// passes its inputs and outputs; the hash ids, gathered rows and kv live in g_scratch below.
//
// g_scratch is a file-scope __device__ array: every GPU that loads this library holds it
// (ENGRAM_NOALLOC_SCRATCH_BYTES) until the process exits. In host code its name is only a
// host-side stand-in, so its device address is looked up with cudaGetSymbolAddress, once per
// device, with that device current, on the first call made on that device. The address is kept
// together with the context it belongs to: after cudaDeviceReset re-creates the device's
// context (and reloads the module, so the array may sit elsewhere), the next call looks it up
// again instead of passing a stale address.
//
// Nothing in the scratch has to start at zero: each call overwrites the ids, rows and kv it
// reads. All calls share the one array, so calls whose work overlaps on the GPU (on different
// streams, or from different threads) race on it and must be ordered by the caller.
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) uint8_t g_scratch[ENGRAM_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
void* g_scratch_ctx[kMaxDevices] = {nullptr};   // the context g_scratch_ptr[dev] belongs to

// Device address of g_scratch on the current device (looked up on first use).
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return engram::fail_cuda(e, "engram_forward_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    engram::set_error("engram_forward_noalloc: device %d beyond the %d devices supported", dev, kMaxDevices);
    return ENGRAM_EINVAL;
  }
  void* ctx = engram::PerContextOnce::current_context();
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return engram::fail_cuda(e, "engram_forward_noalloc: cudaGetSymbolAddress");
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = engram::PerContextOnce::current_context();   // current once the module is loaded
  }
  *out = g_scratch_ptr[dev];
  return ENGRAM_OK;
}

}  // namespace

extern "C" int engram_forward_noalloc(const EngramDims* dims, const EngramHashTables* tables,
                                      const EngramLayerWeights* layers, const EngramTokens* tokens,
                                      float* const* streams, int32_t* out_ids, int32_t* err_flag,
                                      engram_stream_t stream) {
  ENGRAM_CHECK_ARG(dims != nullptr && tokens != nullptr, "dims and tokens must be non-NULL");
  const size_t need = engram_forward_workspace_bytes(dims, tokens->T);
  ENGRAM_CHECK_ARG(need <= (size_t)ENGRAM_NOALLOC_SCRATCH_BYTES,
                   "engram_forward_noalloc: %lld tokens need %zu bytes of scratch, above the fixed %zu; "
                   "use engram_forward with a caller workspace, or fewer tokens per call",
                   (long long)tokens->T, need, (size_t)ENGRAM_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  return engram_forward(dims, tables, layers, tokens, streams, scratch, (size_t)ENGRAM_NOALLOC_SCRATCH_BYTES,
                        out_ids, err_flag, stream);
}
