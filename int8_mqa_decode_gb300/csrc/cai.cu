// Host side of the C ABI: argument validation, split planning and launches.
// Everything here is plain bookkeeping; all arithmetic on the data runs in
// the kernels.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "common.cuh"

namespace cai {

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline bool page_size_ok(int32_t P) { return P == 16 || P == 32 || P == 64; }
constexpr int32_t kItemsPerSmAlone = 32;  // a global layer's split target when launched alone
constexpr int32_t kItemsPerSmMixed = 5;   // ... when launched together with local layers

// Split plan.  The attended span of a sequence is at most `span` tokens (the
// window, or the block-table capacity for a global layer).  Chunks are
// multiples of the 128-token tile.  Automatic choice: about `items_per_sm` work
// items per SM for the expected total work of a global layer (half the capacity
// per sequence), chunks of 512 to 16384 tokens, at most 64 splits -- short items
// let the dynamic queue even out the SMs whatever the length mix, long ones pay
// fewer item boundaries (each costs a few thousand cycles).  A global layer
// launched with local layers, whose whole-window items then even out the tail,
// takes few long items: the hybrid step measured 0.235 ms at 4 items per SM,
// 0.215 at 6, 0.217 at 8, 0.221 at 12, 0.225 at 16, 0.234 at 22, 0.251 at 32.
// Launched alone (the long-context workload) the target matters little (8 to 32
// within 0.3%); 32 keeps the tail short.  A
// local layer is not split when its batch alone gives every SM a sequence (each
// extra split costs its partial's write and read, about an eighth of a
// 1024-token window at 32 heads; 2 and 4 splits measured slower).
DecodePlan plan_decode(int32_t batch, int32_t max_pages_per_seq, int32_t page_size, int32_t window,
                       int32_t num_splits, int32_t sms, int32_t items_per_sm) {
  const int64_t cap = (int64_t)max_pages_per_seq * page_size;
  const int64_t span = window > 0 ? (window < cap ? window : cap) : cap;
  int64_t chunk;
  if (num_splits > 0) {
    chunk = round_up(ceil_div(span, num_splits), kDecodeTile);
  } else if (window > 0) {
    const int64_t want = batch >= sms ? 1 : ceil_div(sms, batch);
    chunk = round_up(ceil_div(span, want), kDecodeTile);
  } else {
    const int64_t expected = (int64_t)batch * ((span + 1) / 2);
    chunk = round_up(ceil_div(expected, (int64_t)items_per_sm * sms), kDecodeTile);
    if (chunk < 512) chunk = 512;
    if (chunk > 16384) chunk = 16384;
  }
  const int64_t min_chunk = round_up(ceil_div(span, kMaxSplits), kDecodeTile);
  if (chunk < min_chunk) chunk = min_chunk;
  if (chunk < kDecodeTile) chunk = kDecodeTile;
  int64_t splits = ceil_div(span, chunk);
  if (splits < 1) splits = 1;
  DecodePlan p;
  p.chunk = (int32_t)chunk;
  p.max_splits = (int32_t)splits;
  return p;
}

static size_t workspace_bytes_for(int32_t batch, int32_t num_q_heads, const DecodePlan& plan) {
  if (plan.max_splits <= 1) return kWorkspaceHeader;
  const size_t rows = (size_t)batch * plan.max_splits * num_q_heads;
  const size_t o_bytes = (size_t)round_up((int64_t)(rows * kHeadDim * sizeof(float)), 256);
  return kWorkspaceHeader + o_bytes + (size_t)round_up((int64_t)(rows * sizeof(float)), 256);
}

}  // namespace cai

namespace cai {
namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int32_t> g_drop_stage{-1};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int32_t fault_drop_stage() { return g_drop_stage.load(std::memory_order_relaxed); }

cai_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CAI_OK;
  g_last_cuda_error = e;
  return CAI_ERR_CUDA;
}
}  // namespace cai

using namespace cai;

extern "C" {

const char* cai_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

void cai_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 2000000000ull, std::memory_order_relaxed); }

void cai_set_fault_injection(int32_t stage) { g_drop_stage.store(stage < 0 ? -1 : stage, std::memory_order_relaxed); }

size_t cai_page_bytes(int32_t page_size, int32_t head_dim) {
  if (page_size <= 0 || head_dim <= 0) return 0;
  return (size_t)page_size * (2 * (size_t)head_dim + 8);
}

const char* cai_status_string(cai_status status) {
  switch (status) {
    case CAI_OK: return "ok";
    case CAI_ERR_INVALID_ARG: return "invalid argument";
    case CAI_ERR_UNSUPPORTED: return "unsupported configuration";
    case CAI_ERR_WORKSPACE: return "workspace missing or too small";
    case CAI_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

static cai_status check_pool(const cai_kv_pool* pool) {
  if (!pool || !pool->pages || pool->num_pages <= 0) return CAI_ERR_INVALID_ARG;
  if (!aligned16(pool->pages)) return CAI_ERR_INVALID_ARG;
  if (pool->head_dim != kHeadDim || !page_size_ok(pool->page_size)) return CAI_ERR_UNSUPPORTED;
  return CAI_OK;
}

namespace {

cai_status append_params(const cai_kv_pool* pool, const float* k_new, const float* v_new, int32_t batch,
                         int32_t n_new, const int32_t* block_table, int32_t max_pages_per_seq,
                         const int32_t* start_pos, int32_t* err_flag, AppendParams& p) {
  cai_status st = check_pool(pool);
  if (st != CAI_OK) return st;
  if (batch < 0 || n_new < 0 || max_pages_per_seq <= 0) return CAI_ERR_INVALID_ARG;
  if ((int64_t)max_pages_per_seq * pool->page_size > (1ll << 30)) return CAI_ERR_UNSUPPORTED;
  if (batch == 0 || n_new == 0) return CAI_OK;
  if ((int64_t)batch * n_new > (1ll << 30)) return CAI_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !block_table || !start_pos) return CAI_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return CAI_ERR_INVALID_ARG;
  p.pages = static_cast<uint8_t*>(pool->pages);
  p.num_pages = pool->num_pages;
  p.page_size = pool->page_size;
  p.max_pages = max_pages_per_seq;
  p.k_new = k_new;
  p.v_new = v_new;
  p.batch = batch;
  p.n_new = n_new;
  p.table = block_table;
  p.start_pos = start_pos;
  p.err = err_flag;
  return CAI_OK;
}

}  // namespace

cai_status cai_kv_append(const cai_kv_pool* pool, const float* k_new, const float* v_new, int32_t batch,
                         int32_t n_new, const int32_t* block_table, int32_t max_pages_per_seq,
                         const int32_t* start_pos, int32_t* err_flag, void* stream) {
  AppendParams p;
  cai_status st = append_params(pool, k_new, v_new, batch, n_new, block_table, max_pages_per_seq, start_pos,
                                err_flag, p);
  if (st != CAI_OK || batch == 0 || n_new == 0) return st;
  return cuda_status(launch_append(&p, 1, static_cast<cudaStream_t>(stream)));
}

cai_status cai_kv_append_pools(const cai_kv_pool* pools, int32_t num_pools, const float* const* k_new,
                               const float* const* v_new, int32_t batch, int32_t n_new,
                               const int32_t* const* block_tables, int32_t max_pages_per_seq,
                               const int32_t* const* start_pos, int32_t* err_flag, void* stream) {
  if (!pools || !k_new || !v_new || !block_tables || !start_pos) return CAI_ERR_INVALID_ARG;
  if (num_pools < 1 || num_pools > kMaxKvHeads) return CAI_ERR_UNSUPPORTED;
  AppendParams ps[kMaxKvHeads];
  for (int i = 0; i < num_pools; ++i) {
    cai_status st = append_params(&pools[i], k_new[i], v_new[i], batch, n_new, block_tables[i], max_pages_per_seq,
                                  start_pos[i], err_flag, ps[i]);
    if (st != CAI_OK) return st;
  }
  if (batch == 0 || n_new == 0) return CAI_OK;
  return cuda_status(launch_append(ps, num_pools, static_cast<cudaStream_t>(stream)));
}

size_t cai_mqa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_pages_per_seq,
                                     int32_t page_size, int32_t window, int32_t num_splits) {
  if (batch <= 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 || !page_size_ok(page_size) || window < 0 ||
      num_splits < 0 || num_splits > kMaxSplits)
    return 0;
  return workspace_bytes_for(batch, num_q_heads,
                             plan_decode(batch, max_pages_per_seq, page_size, window, num_splits, num_sms(),
                                         kItemsPerSmAlone));
}

namespace {

// One layer of a decode launch, as the caller describes it.
struct LayerArgs {
  const cai_kv_pool* pools;  // num_kv_heads pools (one for MQA)
  const uint16_t* q;
  const int32_t* table;
  int32_t window;
  float* out;
  float* lse_out;
};

// Workspace bytes of a launch over these windows: the queue header, then for every
// layer that is split its partial outputs and log-sum-exps.
// Global layers launched together with local ones take longer items.
int32_t items_per_sm_for(const int32_t* windows, int32_t n) {
  bool local = false;
  for (int l = 0; l < n; ++l) local = local || windows[l] > 0;
  return n > 1 && local ? kItemsPerSmMixed : kItemsPerSmAlone;
}

size_t layers_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t max_pages_per_seq,
                              int32_t page_size, const int32_t* windows, int32_t n, int32_t num_splits) {
  size_t total = kWorkspaceHeader;
  const int32_t ips = items_per_sm_for(windows, n);
  for (int l = 0; l < n; ++l) {
    const DecodePlan plan =
        plan_decode(batch * num_kv_heads, max_pages_per_seq, page_size, windows[l], num_splits, num_sms(), ips);
    total += workspace_bytes_for(batch, num_q_heads, plan) - kWorkspaceHeader;
  }
  return total;
}

// Decode of n layers in one persistent launch.  Layer l reads its num_kv_heads
// pools (query heads [j*G, (j+1)*G) read pool j, G = num_q_heads / num_kv_heads);
// the layers share batch, heads, ctx_len, softmax scale and page size.  Their
// work items go through one queue, global layers first (their items are the
// longest), so the SMs even out over the whole step.
cai_status decode_layers_common(const LayerArgs* layers, int32_t n, int32_t num_kv_heads, int32_t batch,
                                int32_t num_q_heads, int32_t max_pages_per_seq, const int32_t* ctx_len,
                                float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                int32_t* err_flag, void* stream) {
  if (n < 1 || n > kMaxDecodeJobs) return CAI_ERR_UNSUPPORTED;
  if (num_kv_heads < 1 || num_kv_heads > kMaxKvHeads) return CAI_ERR_UNSUPPORTED;
  for (int l = 0; l < n; ++l) {
    if (!layers[l].pools) return CAI_ERR_INVALID_ARG;
    for (int j = 0; j < num_kv_heads; ++j) {
      cai_status st = check_pool(&layers[l].pools[j]);
      if (st != CAI_OK) return st;
      if (layers[l].pools[j].page_size != layers[0].pools[0].page_size) return CAI_ERR_INVALID_ARG;
    }
  }
  const int32_t P = layers[0].pools[0].page_size;
  if (batch < 0 || max_pages_per_seq <= 0 || num_splits < 0 || num_splits > kMaxSplits ||
      !std::isfinite(softmax_scale))
    return CAI_ERR_INVALID_ARG;
  for (int l = 0; l < n; ++l)
    if (layers[l].window < 0) return CAI_ERR_INVALID_ARG;
  if (num_q_heads < 1 || num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > kDecodeMaxHeads)
    return CAI_ERR_UNSUPPORTED;
  if ((int64_t)max_pages_per_seq * P > (1ll << 30) || batch > 65535) return CAI_ERR_UNSUPPORTED;
  if (batch == 0) return CAI_OK;
  if (!ctx_len) return CAI_ERR_INVALID_ARG;
  for (int l = 0; l < n; ++l) {
    if (!layers[l].q || !layers[l].table || !layers[l].out) return CAI_ERR_INVALID_ARG;
    if (!aligned16(layers[l].q) || !aligned16(layers[l].out)) return CAI_ERR_INVALID_ARG;
  }
  int32_t windows[kMaxDecodeJobs];
  for (int l = 0; l < n; ++l) windows[l] = layers[l].window;
  const size_t need = layers_workspace_bytes(batch, num_q_heads, num_kv_heads, max_pages_per_seq, P, windows, n,
                                             num_splits);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return CAI_ERR_WORKSPACE;

  DecodeParams p;
  p.num_slots = 0;
  p.num_kv_heads = num_kv_heads;
  p.ctx_len = ctx_len;
  p.batch = batch;
  p.num_heads = num_q_heads;
  p.scale_log2 = softmax_scale * kLog2e;
  p.num_jobs = n;
  p.queue = static_cast<uint32_t*>(workspace);
  p.err = err_flag;
  p.wait_ns = wait_limit_ns();
  p.drop_stage = fault_drop_stage();
  p.overlap_prev = 0;
  // Job order: global layers first, then wider windows first (stable).
  int order[kMaxDecodeJobs];
  for (int l = 0; l < n; ++l) order[l] = l;
  for (int a = 1; a < n; ++a)
    for (int b = a; b > 0; --b) {
      const int wa = windows[order[b]], wb = windows[order[b - 1]];
      const bool before = (wa == 0 && wb != 0) || (wa != 0 && wb != 0 && wa > wb);
      if (!before) break;
      const int t = order[b];
      order[b] = order[b - 1];
      order[b - 1] = t;
    }
  uint8_t* ws = static_cast<uint8_t*>(workspace) + kWorkspaceHeader;
  int64_t items = 0;
  for (int k = 0; k < n; ++k) {
    const LayerArgs& la = layers[order[k]];
    DecodeJob& jb = p.job[k];
    // Pool slots: layers reading the same pools share them.
    int slot0 = -1;
    for (int s0 = 0; s0 + num_kv_heads <= p.num_slots && slot0 < 0; s0 += num_kv_heads) {
      bool same = true;
      for (int j = 0; j < num_kv_heads; ++j) same = same && p.pages[s0 + j] == la.pools[j].pages;
      if (same) slot0 = s0;
    }
    if (slot0 < 0) {
      if (p.num_slots + num_kv_heads > kMaxKvHeads) return CAI_ERR_UNSUPPORTED;
      slot0 = p.num_slots;
      for (int j = 0; j < num_kv_heads; ++j) {
        p.pages[slot0 + j] = static_cast<const uint8_t*>(la.pools[j].pages);
        p.slot_pages[slot0 + j] = la.pools[j].num_pages;
      }
      p.num_slots += num_kv_heads;
    }
    jb.slot0 = slot0;
    jb.window = la.window;
    jb.table = la.table;
    jb.max_pages = max_pages_per_seq;
    jb.q = la.q;
    jb.out = la.out;
    jb.lse_out = la.lse_out;
    jb.plan = plan_decode(batch * num_kv_heads, max_pages_per_seq, P, la.window, num_splits, num_sms(),
                          items_per_sm_for(windows, n));
    jb.ws_o = nullptr;
    jb.ws_lse = nullptr;
    if (jb.plan.max_splits > 1) {
      const size_t rows = (size_t)batch * jb.plan.max_splits * num_q_heads;
      const size_t o_bytes = (size_t)round_up((int64_t)(rows * kHeadDim * sizeof(float)), 256);
      jb.ws_o = reinterpret_cast<float*>(ws);
      jb.ws_lse = reinterpret_cast<float*>(ws + o_bytes);
      ws += workspace_bytes_for(batch, num_q_heads, jb.plan) - kWorkspaceHeader;
    }
    jb.q_off = nullptr;
    jb.total_rows = 0;
    jb.item0 = (int32_t)items;
    items += (int64_t)batch * num_kv_heads * jb.plan.max_splits;
  }
  if (items > 2147483647ll) return CAI_ERR_UNSUPPORTED;
  p.num_items = (int32_t)items;
  for (int k = n; k < kMaxDecodeJobs; ++k) p.job[k] = p.job[n - 1];
  for (int j = p.num_slots; j < kMaxKvHeads; ++j) {
    p.pages[j] = nullptr;
    p.slot_pages[j] = 0;
  }
  return cuda_status(launch_decode(p, P, static_cast<cudaStream_t>(stream)));
}

// Decode of one layer over num_kv_heads pools (one for MQA).
cai_status decode_common(const cai_kv_pool* kv_pools, int32_t num_kv_heads, const uint16_t* q, int32_t batch,
                         int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                         const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                         void* workspace, size_t workspace_bytes, float* out, float* lse_out, int32_t* err_flag,
                         void* stream) {
  const LayerArgs la = {kv_pools, q, block_table, window, out, lse_out};
  return decode_layers_common(&la, 1, num_kv_heads, batch, num_q_heads, max_pages_per_seq, ctx_len, softmax_scale,
                              num_splits, workspace, workspace_bytes, err_flag, stream);
}

}  // namespace

cai_status cai_mqa_decode(const cai_kv_pool* pools, int32_t num_pools, const int32_t* layer_to_pool,
                          int32_t num_layers, int32_t layer, const uint16_t* q, int32_t batch,
                          int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                          const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, float* out, float* lse_out,
                          int32_t* err_flag, void* stream) {
  if (!pools || num_pools <= 0 || !layer_to_pool || num_layers <= 0 || layer < 0 || layer >= num_layers)
    return CAI_ERR_INVALID_ARG;
  const int32_t buf = layer_to_pool[layer];
  if (buf < 0 || buf >= num_pools) return CAI_ERR_INVALID_ARG;
  return decode_common(&pools[buf], 1, q, batch, num_q_heads, block_table, max_pages_per_seq, ctx_len, window,
                       softmax_scale, num_splits, workspace, workspace_bytes, out, lse_out, err_flag, stream);
}

size_t cai_mqa_decode_layers_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_pages_per_seq,
                                            int32_t page_size, int32_t num_layers, const int32_t* windows,
                                            int32_t num_splits) {
  if (batch <= 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 || !page_size_ok(page_size) || num_layers < 1 ||
      num_layers > kMaxDecodeJobs || !windows || num_splits < 0 || num_splits > kMaxSplits)
    return 0;
  for (int l = 0; l < num_layers; ++l)
    if (windows[l] < 0) return 0;
  return layers_workspace_bytes(batch, num_q_heads, 1, max_pages_per_seq, page_size, windows, num_layers,
                                num_splits);
}

cai_status cai_mqa_decode_layers(const cai_kv_pool* pools, int32_t num_pools, const int32_t* layer_to_pool,
                                 int32_t num_layers, const int32_t* windows, const uint16_t* const* q,
                                 int32_t batch, int32_t num_q_heads, const int32_t* const* block_tables,
                                 int32_t max_pages_per_seq, const int32_t* ctx_len, float softmax_scale,
                                 int32_t num_splits, void* workspace, size_t workspace_bytes, float* const* out,
                                 float* const* lse_out, int32_t* err_flag, void* stream) {
  if (!pools || num_pools <= 0 || !layer_to_pool || !windows || !q || !block_tables || !out)
    return CAI_ERR_INVALID_ARG;
  if (num_layers < 1 || num_layers > kMaxDecodeJobs) return CAI_ERR_UNSUPPORTED;
  LayerArgs la[kMaxDecodeJobs];
  for (int l = 0; l < num_layers; ++l) {
    const int32_t buf = layer_to_pool[l];
    if (buf < 0 || buf >= num_pools) return CAI_ERR_INVALID_ARG;
    la[l] = LayerArgs{&pools[buf], q[l], block_tables[l], windows[l], out[l], lse_out ? lse_out[l] : nullptr};
  }
  return decode_layers_common(la, num_layers, 1, batch, num_q_heads, max_pages_per_seq, ctx_len, softmax_scale,
                              num_splits, workspace, workspace_bytes, err_flag, stream);
}

size_t cai_gqa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t max_pages_per_seq, int32_t page_size, int32_t window,
                                     int32_t num_splits) {
  if (num_kv_heads < 1 || num_kv_heads > kMaxKvHeads || num_q_heads < 1 || num_q_heads % num_kv_heads != 0 ||
      batch <= 0 || (int64_t)batch * num_kv_heads > 2147483647ll)
    return 0;
  if (max_pages_per_seq <= 0 || !page_size_ok(page_size) || window < 0 || num_splits < 0 || num_splits > kMaxSplits)
    return 0;
  return workspace_bytes_for(batch, num_q_heads, plan_decode(batch * num_kv_heads, max_pages_per_seq, page_size,
                                                             window, num_splits, num_sms(), kItemsPerSmAlone));
}

cai_status cai_gqa_decode(const cai_kv_pool* kv_pools, int32_t num_kv_heads, const uint16_t* q, int32_t batch,
                          int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                          const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, float* out, float* lse_out, int32_t* err_flag,
                          void* stream) {
  if (!kv_pools) return CAI_ERR_INVALID_ARG;
  if ((int64_t)batch * num_kv_heads > 65535) return CAI_ERR_UNSUPPORTED;
  return decode_common(kv_pools, num_kv_heads, q, batch, num_q_heads, block_table, max_pages_per_seq, ctx_len,
                       window, softmax_scale, num_splits, workspace, workspace_bytes, out, lse_out, err_flag, stream);
}

size_t cai_mqa_prefill_workspace_size(int32_t batch, int32_t max_pages_per_seq, int32_t page_size) {
  if (batch <= 0 || max_pages_per_seq <= 0 || !page_size_ok(page_size)) return 0;
  return prefill_workspace_bytes(batch, max_pages_per_seq, page_size);
}

namespace {

cai_status prefill_common(const cai_kv_pool* pool, const uint16_t* q, int32_t batch, const int32_t* q_off,
                          int32_t n_new, int32_t total_new, int32_t num_q_heads, const int32_t* block_table,
                          int32_t max_pages_per_seq, const int32_t* prefix_len, int32_t window, float softmax_scale,
                          void* workspace, size_t workspace_bytes, float* out, float* lse_out, int32_t* err_flag,
                          void* stream) {
  cai_status st = check_pool(pool);
  if (st != CAI_OK) return st;
  if (batch < 0 || n_new < 0 || total_new < 0 || max_pages_per_seq <= 0 || window < 0 ||
      !std::isfinite(softmax_scale))
    return CAI_ERR_INVALID_ARG;
  if (num_q_heads < 1 || num_q_heads > 128 || (num_q_heads & (num_q_heads - 1)) != 0) return CAI_ERR_UNSUPPORTED;
  if ((int64_t)max_pages_per_seq * pool->page_size > (1ll << 24) || batch > 65535) return CAI_ERR_UNSUPPORTED;
  if ((int64_t)n_new * num_q_heads > (1ll << 24) || (int64_t)total_new * num_q_heads > (1ll << 31) / kHeadDim)
    return CAI_ERR_UNSUPPORTED;
  if (batch == 0 || n_new == 0 || total_new == 0) return CAI_OK;
  if (!q || !block_table || !prefix_len || !out) return CAI_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return CAI_ERR_INVALID_ARG;
  const size_t need = prefill_workspace_bytes(batch, max_pages_per_seq, pool->page_size);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return CAI_ERR_WORKSPACE;
  PrefillLaunch L;
  L.pages = static_cast<const uint8_t*>(pool->pages);
  L.num_pages = pool->num_pages;
  L.page_size = pool->page_size;
  L.max_pages = max_pages_per_seq;
  L.table = block_table;
  L.prefix_len = prefix_len;
  L.q = q;
  L.q_off = q_off;
  L.batch = batch;
  L.n_new = n_new;
  L.total_new = total_new;
  L.num_heads = num_q_heads;
  L.window = window;
  L.scale_log2 = softmax_scale * kLog2e;
  L.workspace = workspace;
  L.out = out;
  L.lse_out = lse_out;
  L.err = err_flag;
  // Continuous batching: sequences bringing one new token are decode steps; the decode
  // kernel runs them (with this call's window and scale, split as a decode call would be) and the
  // prefill kernel skips them, so they pay neither the prefill's 256-row q-tiles nor its
  // dequantised copy of their keys.  Its queue counters sit at the end of the workspace.
  // The two kernels share no memory (the decode writes the one-token rows and its
  // partials, the prefill the other rows and its copy of the keys), so the decode is
  // launched after the prefill without waiting for it: its CTAs take the SMs that the
  // prefill's last, partial wave leaves idle, and its queue hands them the items.
  L.skip_single = q_off != nullptr && num_q_heads <= kDecodeMaxHeads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.skip_single) {
    void* hdr = static_cast<uint8_t*>(workspace) + (need - kWorkspaceHeader);
    cudaError_t e = cudaMemsetAsync(hdr, 0, kWorkspaceHeader, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  cudaError_t e = launch_prefill(L, s);
  if (e != cudaSuccess || !L.skip_single) return cuda_status(e);
  {
    void* hdr = static_cast<uint8_t*>(workspace) + (need - kWorkspaceHeader);
    DecodeParams d;
    d.pages[0] = static_cast<const uint8_t*>(pool->pages);
    d.slot_pages[0] = pool->num_pages;
    for (int j = 1; j < kMaxKvHeads; ++j) {
      d.pages[j] = nullptr;
      d.slot_pages[j] = 0;
    }
    d.num_slots = 1;
    d.num_kv_heads = 1;
    d.ctx_len = prefix_len;
    d.batch = batch;
    d.num_heads = num_q_heads;
    d.scale_log2 = softmax_scale * kLog2e;
    d.num_jobs = 1;
    d.queue = static_cast<uint32_t*>(hdr);
    d.err = err_flag;
    d.wait_ns = wait_limit_ns();
    d.drop_stage = fault_drop_stage();
    d.overlap_prev = 1;
    DecodeJob& jb = d.job[0];
    jb.slot0 = 0;
    jb.window = window;
    jb.table = block_table;
    jb.max_pages = max_pages_per_seq;
    jb.q = q;
    jb.out = out;
    jb.lse_out = lse_out;
    // The automatic split plan, its partials in the workspace's piece region (a varlen
    // call's prefill cuts no q-tile into pieces, so the region is the decode's); fewer
    // splits when they would not fit.
    void* region = nullptr;
    size_t region_bytes = 0;
    prefill_piece_region(workspace, batch, max_pages_per_seq, pool->page_size, &region, &region_bytes);
    DecodePlan plan =
        plan_decode(batch, max_pages_per_seq, pool->page_size, window, 0, num_sms(), kItemsPerSmAlone);
    while (plan.max_splits > 1 && workspace_bytes_for(batch, num_q_heads, plan) - kWorkspaceHeader > region_bytes)
      plan = plan_decode(batch, max_pages_per_seq, pool->page_size, window, plan.max_splits - 1, num_sms(),
                         kItemsPerSmAlone);
    jb.plan = plan;
    jb.ws_o = nullptr;
    jb.ws_lse = nullptr;
    if (plan.max_splits > 1) {
      const size_t rows = (size_t)batch * plan.max_splits * num_q_heads;
      const size_t o_bytes = (size_t)round_up((int64_t)(rows * kHeadDim * sizeof(float)), 256);
      jb.ws_o = static_cast<float*>(region);
      jb.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(region) + o_bytes);
    }
    jb.item0 = 0;
    jb.q_off = q_off;
    jb.total_rows = total_new;
    for (int k = 1; k < kMaxDecodeJobs; ++k) d.job[k] = jb;
    d.num_items = batch * plan.max_splits;
    e = launch_decode(d, pool->page_size, s);
  }
  return cuda_status(e);
}

}  // namespace

cai_status cai_mqa_prefill_chunk(const cai_kv_pool* pool, const uint16_t* q, int32_t batch, int32_t n_new,
                                 int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                                 const int32_t* prefix_len, int32_t window, float softmax_scale, void* workspace,
                                 size_t workspace_bytes, float* out, float* lse_out, int32_t* err_flag,
                                 void* stream) {
  if ((int64_t)batch * n_new > 2147483647ll) return CAI_ERR_UNSUPPORTED;
  return prefill_common(pool, q, batch, nullptr, n_new, batch * n_new, num_q_heads, block_table, max_pages_per_seq,
                        prefix_len, window, softmax_scale, workspace, workspace_bytes, out, lse_out, err_flag, stream);
}

cai_status cai_mqa_prefill_varlen(const cai_kv_pool* pool, const uint16_t* q, int32_t batch,
                                  const int32_t* q_offsets, int32_t total_new, int32_t max_new, int32_t num_q_heads,
                                  const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* prefix_len,
                                  int32_t window, float softmax_scale, void* workspace, size_t workspace_bytes,
                                  float* out, float* lse_out, int32_t* err_flag, void* stream) {
  if (batch > 0 && total_new > 0 && !q_offsets) return CAI_ERR_INVALID_ARG;
  return prefill_common(pool, q, batch, q_offsets, max_new, total_new, num_q_heads, block_table, max_pages_per_seq,
                        prefix_len, window, softmax_scale, workspace, workspace_bytes, out, lse_out, err_flag, stream);
}

}  // extern "C"
