// cai_mqa_decode_no_alloc: the decode entry point for callers that cannot give
// the library any device scratch memory.
//
// Some hosts cannot allocate on the device when they call us: a serving loop
// that freezes allocation after warm-up (cudaMalloc can synchronise the device
// and stall every other stream), a plugin interface that hands over only
// input and output buffers, or an embedding framework that owns all device
// memory through its own allocator and gives its plug-ins no way to borrow
// from it.  For them this variant keeps the split-KV partials in a fixed
// scratch array compiled into the library instead of a caller workspace.
//
// The array is a file-scope __device__ object of kStaticScratchBytes: every
// GPU that loads the library holds it until the process exits.  Host code may
// not use the array's name as a device address (on the host it names a
// stand-in object), so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device; make that first call before any stream capture.  All calls
// share the one array and it keeps the last call's contents: two calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on it.  Nothing in the array has to start at zero: every partial that
// is read is written first by the same call.
#include <mutex>

#include "common.cuh"

namespace cai {
namespace {

constexpr size_t kStaticScratchBytes = CAI_NO_ALLOC_SCRATCH_BYTES;  // 32 MiB per GPU
__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_decode_scratch on the current device (null on failure).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
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
  if (need > 0) {
    scratch = cai::scratch_address();
    if (!scratch) return CAI_ERR_CUDA;
  }
  return cai_mqa_decode(pools, num_pools, layer_to_pool, num_layers, layer, q, batch, num_q_heads, block_table,
                        max_pages_per_seq, ctx_len, window, softmax_scale, num_splits, scratch,
                        need > 0 ? cai::kStaticScratchBytes : 0, out, lse_out, err_flag, stream);
}

}  // extern "C"
