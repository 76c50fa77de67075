// cai_mqa_decode_no_alloc: the decode entry point for callers that cannot give
// the library any device scratch memory.
//
// Some hosts cannot allocate on the device when they call us: a serving loop
// that freezes allocation after warm-up (cudaMalloc can synchronise the device
// and stall every other stream), a plugin interface that hands over only
// input and output buffers, or an embedding framework that owns all device
// memory through its own allocator and gives its plug-ins no way to borrow
// from it.  For them this variant keeps the decode workspace -- the work-queue
// counters and the split-KV partials -- in a fixed scratch array compiled into
// the library instead of a caller workspace.
//
// The array is a file-scope __device__ object of kStaticScratchBytes: every
// GPU that loads the library holds it until the process exits.  Host code may
// not use the array's name as a device address (on the host it names a
// stand-in object), so the device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made on
// that device (and again on the first call after the device's primary context
// was replaced, e.g. after cudaDeviceReset); make that first call before any
// stream capture.  All calls share the one array and it keeps the last call's
// contents: two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it.  The queue counters in its first
// kWorkspaceHeader bytes must be zero when the decode kernel starts; every call
// clears them with a stream-ordered memset before its launch, so a call that
// follows one that gave up (CAI_DEVERR_TIMEOUT) starts clean.  The partials
// need no clearing: every partial a call reads is written first by that call.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace cai {
namespace {

constexpr size_t kStaticScratchBytes = CAI_NO_ALLOC_SCRATCH_BYTES;  // 32 MiB per GPU
__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  CUcontext ctx;  // context the address was looked up in
  void* addr;
};
ScratchSlot g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// The driver's cuCtxGetCurrent, looked up through the runtime (no -lcuda).
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
  }
  return fn;
}

// Device address of g_decode_scratch on the current device and context.
cai_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return CAI_ERR_UNSUPPORTED;
  auto get_ctx = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return cuda_status(cudaErrorInitializationError);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchSlot& slot = g_scratch[dev];
  if (!slot.addr || !ctx || slot.ctx != ctx) {
    // No context current yet (the lookup makes the primary context current) or
    // another one than at the last lookup: look the address up in this one.
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return cuda_status(cudaErrorInitializationError);
    slot.ctx = ctx;
    slot.addr = ptr;
  }
  *out = slot.addr;
  return CAI_OK;
}

}  // namespace
}  // namespace cai

extern "C" {

cai_status cai_mqa_decode_no_alloc(const cai_kv_pool* pools, int32_t num_pools, const int32_t* layer_to_pool,
                                   int32_t num_layers, int32_t layer, const uint16_t* q, int32_t batch,
                                   int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                                   const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                                   float* out, float* lse_out, int32_t* err_flag, void* stream) {
  if (!pools || num_pools <= 0 || !layer_to_pool || num_layers <= 0 || layer < 0 || layer >= num_layers)
    return CAI_ERR_INVALID_ARG;
  const int32_t buf = layer_to_pool[layer];
  if (buf < 0 || buf >= num_pools) return CAI_ERR_INVALID_ARG;
  const size_t need = cai_mqa_decode_workspace_size(batch, num_q_heads, max_pages_per_seq, pools[buf].page_size,
                                                    window, num_splits);
  if (need > cai::kStaticScratchBytes) return CAI_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && batch > 0) {
    const cai_status st = cai::scratch_address(&scratch);
    if (st != CAI_OK) return st;
    // The work-queue counters start every call at zero (stream-ordered, no allocation).
    const cudaError_t e = cudaMemsetAsync(scratch, 0, cai::kWorkspaceHeader, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cai::cuda_status(e);
  }
  return cai_mqa_decode(pools, num_pools, layer_to_pool, num_layers, layer, q, batch, num_q_heads, block_table,
                        max_pages_per_seq, ctx_len, window, softmax_scale, num_splits, scratch,
                        scratch ? cai::kStaticScratchBytes : 0, out, lse_out, err_flag, stream);
}

}  // extern "C"
