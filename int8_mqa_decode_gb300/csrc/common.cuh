// Shared definitions of the CUDA side of libcai: launch parameter blocks,
// constants and the split plan.
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "cai.h"

namespace cai {

constexpr int kHeadDim = 128;
constexpr int kMaxSplits = 64;
constexpr int kDecodeTile = 128;       // tokens per decode tile (MMA M of the scores, K of PV)
constexpr int kRawTokens = 64;         // tokens per raw page stage (half a tile)
constexpr int kDecodeMaxHeads = 64;    // query heads per decode call at most (MMA N of the scores)
constexpr int kWorkspaceHeader = 256;  // decode workspace: work-queue counters, kept zero between calls
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Bytes of one page for head_dim 128: P * (2*128 + 8).
__host__ __device__ constexpr int page_bytes(int P) { return P * (2 * kHeadDim + 8); }

struct AppendParams {
  uint8_t* pages;
  int32_t num_pages, page_size, max_pages;
  const float* k_new;
  const float* v_new;
  int32_t batch, n_new;
  const int32_t* table;
  const int32_t* start_pos;
  int32_t* err;
};

// Work split of one decode launch.  The attended span [lo, hi) of every
// sequence is cut into consecutive chunks of `chunk` tokens starting at lo:
// split j covers [lo + j*chunk, min(hi, lo + (j+1)*chunk)).
struct DecodePlan {
  int32_t chunk;       // tokens per split, a multiple of kDecodeTile
  int32_t max_splits;  // upper bound of splits per sequence
};

constexpr int kMaxKvHeads = 8;         // KV heads (pools) one decode call can read

constexpr int kMaxDecodeJobs = 8;  // layers decoded by one launch

// One layer of a decode launch: its query, output and block table, its window and
// split plan, and the pool slots its KV heads read (slot0 + j for KV head j).
struct DecodeJob {
  int32_t slot0;
  int32_t window;
  const int32_t* table;  // [B][max_pages]
  int32_t max_pages;
  const uint16_t* q;     // bf16 bits [B][Hq][128]
  float* out;            // [B][Hq][128]
  float* lse_out;        // [B][Hq] natural log, nullable
  float* ws_o;           // [B][max_splits][Hq][128] partial outputs (normalised), null without splits
  float* ws_lse;         // [B][max_splits][Hq] partial lse, log2 units
  DecodePlan plan;
  int32_t item0;         // first work item of the layer; items are (b * KV heads + KV head) * max_splits + split
  // Continuous batching: when q_off is set, sequence b is decoded only if it brings exactly
  // one new token, q and out rows [q_off[b], q_off[b+1]) (< total_rows) of a packed batch,
  // and ctx_len holds its prefix length (the token sits at position ctx_len[b]); other
  // sequences are left to the prefill kernel.  Such a job is never split.
  const int32_t* q_off;
  int32_t total_rows;
};

// Row of sequence b in a job's q / out / lse_out.
__host__ __device__ inline int64_t job_row(const DecodeJob& jb, int b) { return jb.q_off ? jb.q_off[b] : b; }

struct DecodeParams {
  const uint8_t* pages[kMaxKvHeads];  // pool slots, one per (layer's) KV head, same page size
  int32_t slot_pages[kMaxKvHeads];    // pages in each slot
  int32_t num_slots;
  int32_t num_kv_heads;               // query heads [j*G, (j+1)*G) read KV head j, G = num_heads / num_kv_heads
  const int32_t* ctx_len;             // [B], shared by the layers
  int32_t batch, num_heads;
  float scale_log2;                   // softmax_scale * log2(e)
  int32_t num_jobs, num_items;
  DecodeJob job[kMaxDecodeJobs];
  uint32_t* queue;                    // [2]: next work item, CTAs finished (both zero between calls)
  int32_t* err;
  uint64_t wait_ns;                   // limit of every bounded wait inside the kernel
  int32_t drop_stage;                 // fault injection: K/V stage each CTA skips (-1: none)
  // 1: the kernel before this launch in the stream touches none of its memory and was
  // itself started only after everything before it had completed, so the launch does
  // not wait for it (it starts on SMs as that kernel's CTAs leave them).
  int32_t overlap_prev;
};

// Attended range and split bookkeeping shared by the decode and combine kernels.
struct SeqSplits {
  int32_t lo, hi;      // attended positions [lo, hi)
  int32_t nsplit;      // number of non-empty splits (0 if nothing to attend)
  bool valid;          // length within the block table
};

__host__ __device__ inline SeqSplits seq_splits(int32_t L, int32_t window, int32_t max_tokens, int32_t chunk) {
  SeqSplits s;
  s.valid = (L >= 0 && L <= max_tokens);
  if (!s.valid) L = 0;
  s.hi = L;
  s.lo = (window > 0 && L > window) ? L - window : 0;
  s.nsplit = s.hi > s.lo ? (s.hi - s.lo + chunk - 1) / chunk : 0;
  return s;
}

struct PrefillLaunch {
  const uint8_t* pages;
  int32_t num_pages, page_size, max_pages;
  const int32_t* table;
  const int32_t* prefix_len;
  const uint16_t* q;
  const int32_t* q_off;  // [batch + 1] packed new-token offsets (device), or null for n_new per sequence
  int32_t batch, n_new, total_new, num_heads, window;  // n_new: the most new tokens of any sequence
  float scale_log2;
  void* workspace;
  float* out;
  float* lse_out;
  int32_t* err;
  bool skip_single;      // with q_off: sequences with one new token are decoded elsewhere
};

// Limit of the kernels' bounded waits (cai_set_wait_limit_ns), read at every launch.
uint64_t wait_limit_ns();
// The stage every CTA skips (cai_set_fault_injection; -1: none), read at every launch.
int32_t fault_drop_stage();

size_t prefill_workspace_bytes(int32_t batch, int32_t max_pages_per_seq, int32_t page_size);
void prefill_piece_region(void* workspace, int32_t batch, int32_t max_pages_per_seq, int32_t page_size,
                          void** region, size_t* bytes);
cudaError_t launch_prefill(const PrefillLaunch& p, cudaStream_t stream);

// Launch with programmatic stream serialization: the grid may start while the
// previous kernel in the stream finishes; every kernel launched this way calls
// grid_dependency_wait() before it touches memory another kernel writes or reads.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host side: the split plan for a launch (also used by the workspace query).
DecodePlan plan_decode(int32_t batch, int32_t max_pages_per_seq, int32_t page_size, int32_t window,
                       int32_t num_splits, int32_t num_sms, int32_t items_per_sm);
int num_sms();

// CAI_OK for cudaSuccess; otherwise CAI_ERR_CUDA, with the error kept for
// cai_last_cuda_error() on this thread.
cai_status cuda_status(cudaError_t e);

// Kernel launchers (return cudaGetLastError()).
cudaError_t launch_append(const AppendParams* ps, int n, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int page_size, cudaStream_t stream);

}  // namespace cai
