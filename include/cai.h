/*
 * cai.h - C ABI of the int8 MQA paged decode library (libcai.so).
 *
 * What the library computes comes from the pages it was written from:
 *  - "Character.AI: inference optimization", 03 Model architecture, technique
 *    table: Multi-Query Attention in every attention layer (all query heads
 *    read one K/V head); hybrid attention where most layers are local with a
 *    horizon of 1024 and one layer in six is global; KV shared by
 *    neighbouring layers.
 *  - same page, 05 Quantization and cost: the attention KV cache is int8.
 *  - same page, 04 Cache between turns, and the Red Hat page "Como funciona a
 *    inferencia de IA", section "3. Cache de prefixo": the KV of a cached
 *    prefix is reused and only new tokens are processed.
 *  - Red Hat page, section "1. PagedAttention": the cache is cut into
 *    fixed-size blocks placed anywhere in memory, with a per-request table of
 *    block ids.
 *  - Red Hat page, "Por que o cache KV existe": K and V are computed once for
 *    each new token and stored; the new token's query is compared with the
 *    keys of all tokens so far and the values are summed with those weights.
 *
 * Conventions for every call:
 *  - All pointers to tensors are DEVICE pointers unless marked "host".  The
 *    caller owns all memory; the library allocates nothing.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Host-side validation failures return a status and
 *    launch nothing.  Problems only the device can see (a block-table entry
 *    outside the pool, a length beyond the table) set bits in `*err_flag`
 *    (atomic OR; nullable) and the affected work is skipped: outputs of
 *    affected rows are then unspecified, but no out-of-bounds access happens.
 *  - The library keeps no global state apart from a per-device attribute
 *    cache; calls on different streams are independent.
 *  - head_dim is 128.  Queries are bf16 and must be within the fp16 range
 *    (|q| <= 65504): the tensor-core path runs in fp16 with fp32 accumulation.
 *    K/V inputs must be finite.
 */
#ifndef CAI_H_
#define CAI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cai_status {
  CAI_OK = 0,
  CAI_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned pointer, index out of range */
  CAI_ERR_UNSUPPORTED = 2, /* head_dim, page_size or head count outside what the kernels implement */
  CAI_ERR_WORKSPACE = 3,   /* workspace missing or smaller than cai_mqa_decode_workspace_size() */
  CAI_ERR_CUDA = 4         /* a CUDA runtime call or a launch failed */
} cai_status;

/* Bits OR-ed into *err_flag by the kernels. */
#define CAI_DEVERR_PAGE 1   /* a needed block-table entry is outside [0, num_pages) */
#define CAI_DEVERR_LENGTH 2 /* a length or position is negative or beyond max_pages_per_seq * page_size */
#define CAI_DEVERR_TIMEOUT 4 /* a bounded wait inside a kernel gave up; that launch's outputs are unspecified */

/* One KV buffer: a pool of fixed-size pages (PagedAttention blocks).
 * Page layout (bytes), for P = page_size and d = head_dim:
 *   [0,        P*d)        K codes, int8 [P][d] (token-major: slot s at s*d)
 *   [P*d,      2*P*d)      V codes, int8 [d][P] (channel-major: channel c at c*P)
 *   [2*P*d,    2*P*d+4*P)  K scales, fp32 [P]
 *   [2*P*d+4P, 2*P*d+8*P)  V scales, fp32 [P]
 * Token at position p of a sequence lives in page block_table[p / P], slot p % P.
 * `pages` must be 16-byte aligned; it holds num_pages * cai_page_bytes(P, d) bytes. */
typedef struct cai_kv_pool {
  void* pages;
  int32_t num_pages;
  int32_t page_size; /* 16, 32 or 64 tokens */
  int32_t head_dim;  /* 128 */
} cai_kv_pool;

/* Bytes of one page: page_size * (2*head_dim + 8).  0 for non-positive arguments. */
size_t cai_page_bytes(int32_t page_size, int32_t head_dim);

/* Quantize new tokens to int8 and write them into their pages.
 * Int8 KV cache ("Character.AI: inference optimization", 05), written once per
 * new token (Red Hat page, "Por que o cache KV existe").  For each token and
 * separately for K and V: s = max_i |x_i| / 127 (fp32, IEEE division),
 * code_i = clamp(round_half_even(x_i / s), -127, 127); codes 0 when s is 0 (an
 * all-zero vector, or max |x_i| / 127 below the smallest fp32 subnormal).
 * Results are bit-exact.
 *   pool        host pointer to the pool description
 *   k_new,v_new fp32 [batch][n_new][head_dim], 16-byte aligned
 *   block_table int32 [batch][max_pages_per_seq]; entries for the written positions must be valid pages
 *   start_pos   int32 [batch]: token i of sequence b goes to position start_pos[b] + i
 *   err_flag    int32, nullable
 * Positions outside [0, max_pages_per_seq * page_size) set CAI_DEVERR_LENGTH; bad
 * page ids set CAI_DEVERR_PAGE; such tokens are not written.  No other byte of the
 * pool changes (K and V of past tokens never change). */
cai_status cai_kv_append(const cai_kv_pool* pool, const float* k_new, const float* v_new, int32_t batch,
                         int32_t n_new, const int32_t* block_table, int32_t max_pages_per_seq,
                         const int32_t* start_pos, int32_t* err_flag, void* stream);

/* The append of one step into several KV buffers in one launch: for every i the
 * same as cai_kv_append(&pools[i], k_new[i], v_new[i], batch, n_new,
 * block_tables[i], max_pages_per_seq, start_pos[i], ...) (neighbouring layers
 * that share a buffer append once; "Character.AI: inference optimization"
 * page, 03 Model architecture).
 *   pools, num_pools       host array of 1..8 KV buffers
 *   k_new, v_new           host arrays [num_pools] of device fp32 [batch][n_new][head_dim], 16-byte aligned
 *   block_tables           host array [num_pools] of device int32 [batch][max_pages_per_seq]
 *   start_pos              host array [num_pools] of device int32 [batch]
 * Errors as for cai_kv_append; nothing is launched when an argument is rejected. */
cai_status cai_kv_append_pools(const cai_kv_pool* pools, int32_t num_pools, const float* const* k_new,
                               const float* const* v_new, int32_t batch, int32_t n_new,
                               const int32_t* const* block_tables, int32_t max_pages_per_seq,
                               const int32_t* const* start_pos, int32_t* err_flag, void* stream);

/* Bytes of workspace cai_mqa_decode needs for these arguments: a 256-byte
 * header (the counters of the kernel's work queue) plus, when sequences are
 * split, the partial outputs.  Arguments as for cai_mqa_decode.  The automatic
 * split plan (num_splits = 0) depends on the SM count of the current device:
 * query with the device that will run the call. */
size_t cai_mqa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_pages_per_seq,
                                     int32_t page_size, int32_t window, int32_t num_splits);

/* One decode step of one layer: MQA attention of one query token per sequence
 * over its int8 paged KV.
 *   pools, num_pools       host array of KV buffers
 *   layer_to_pool          host int32 [num_layers]: buffer read by each layer (layers may share one)
 *   layer                  the layer to run
 *   q                      bf16 bits [batch][num_q_heads][head_dim], 16-byte aligned
 *   num_q_heads            1..64 query heads, all sharing the single K/V head
 *   block_table            int32 [batch][max_pages_per_seq]
 *   ctx_len                int32 [batch]: cached tokens INCLUDING the current one (append first)
 *   window                 0 = global; W > 0 = local: only the last W positions
 *                          [max(0, L-W), L) are attended, pages wholly before them are never read
 *   softmax_scale          logit = softmax_scale * <q, k>
 *   num_splits             0 = automatic; otherwise the attended span of each sequence is cut
 *                          into at most this many consecutive chunks (1..64), processed as
 *                          separate work items and merged with their log-sum-exp
 *   workspace              device scratch of at least cai_mqa_decode_workspace_size() bytes,
 *                          256-byte aligned.  Its first 256 bytes must be zero before the first
 *                          call that uses it; every call leaves them zero again (after a call
 *                          that reported CAI_DEVERR_TIMEOUT, zero them before reuse).  Calls that
 *                          share a workspace must not overlap on the GPU.
 *   out                    fp32 [batch][num_q_heads][head_dim], 16-byte aligned
 *   lse_out                fp32 [batch][num_q_heads] natural-log log-sum-exp of the logits, nullable;
 *                          any 4-byte alignment (at 16 bytes it is written by bulk copies)
 * A sequence with nothing to attend (L = 0) gets out = 0 and lse = -inf. */
cai_status cai_mqa_decode(const cai_kv_pool* pools, int32_t num_pools, const int32_t* layer_to_pool,
                          int32_t num_layers, int32_t layer, const uint16_t* q, int32_t batch,
                          int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                          const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, float* out, float* lse_out,
                          int32_t* err_flag, void* stream);

/* Workspace bytes for cai_mqa_decode_layers (windows: host int32 [num_layers]); 0 if the
 * arguments are invalid. */
size_t cai_mqa_decode_layers_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_pages_per_seq,
                                            int32_t page_size, int32_t num_layers, const int32_t* windows,
                                            int32_t num_splits);

/* One decode step of several layers in one launch: for every layer l the same
 * computation as cai_mqa_decode, on the same work split, with the work items of
 * all the layers taken from one queue (global layers first) so that the SMs even
 * out over the whole step instead of layer by layer.  One call covers a decode
 * step of the hybrid stack ("Character.AI: inference optimization" page,
 * 03 Model architecture: local layers with a 1024 horizon, one global layer in
 * six, neighbouring layers sharing one KV buffer; 02 The bottleneck: reading the
 * attention KV dominates the I/O of a step).
 *   pools, num_pools       host array of KV buffers
 *   layer_to_pool          host int32 [num_layers]: buffer read by each layer (layers may share one)
 *   num_layers             1..8
 *   windows                host int32 [num_layers]: 0 = global, W > 0 = local (as in cai_mqa_decode)
 *   q                      host array [num_layers] of device bf16 bits [batch][num_q_heads][head_dim],
 *                          each 16-byte aligned
 *   block_tables           host array [num_layers] of device int32 [batch][max_pages_per_seq]
 *   ctx_len                int32 [batch], shared by the layers (append first)
 *   workspace              device scratch of cai_mqa_decode_layers_workspace_size() bytes, 256-byte
 *                          aligned, first 256 bytes zero (as for cai_mqa_decode)
 *   out                    host array [num_layers] of device fp32 [batch][num_q_heads][head_dim],
 *                          each 16-byte aligned
 *   lse_out                host array [num_layers] of nullable device fp32 [batch][num_q_heads], or null
 * All buffers must use one page size; at most 8 distinct buffers.  Errors as for
 * cai_mqa_decode; nothing is launched when an argument is rejected. */
cai_status cai_mqa_decode_layers(const cai_kv_pool* pools, int32_t num_pools, const int32_t* layer_to_pool,
                                 int32_t num_layers, const int32_t* windows, const uint16_t* const* q,
                                 int32_t batch, int32_t num_q_heads, const int32_t* const* block_tables,
                                 int32_t max_pages_per_seq, const int32_t* ctx_len, float softmax_scale,
                                 int32_t num_splits, void* workspace, size_t workspace_bytes, float* const* out,
                                 float* const* lse_out, int32_t* err_flag, void* stream);

/* Decode without any caller scratch.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot allocate device memory at
 * the moment they decode -- a serving loop that forbids cudaMalloc after
 * warm-up (an allocation can synchronise the device and stall other
 * streams), a plug-in interface that passes only input and output buffers,
 * or a framework that owns all device memory and lends none to its plug-ins.
 * It computes exactly what cai_mqa_decode computes, with the same arguments
 * minus the workspace: the work-queue counters and the split partials live in
 * a scratch array built into the library, CAI_NO_ALLOC_SCRATCH_BYTES per GPU,
 * held by every GPU that loads the library until the process exits.  A call
 * whose plan needs more (cai_mqa_decode_workspace_size() above the limit)
 * returns CAI_ERR_WORKSPACE and launches nothing: lower num_splits (1 needs
 * only the 256-byte counter header).  The first call on a device looks up the
 * array's device address on that device (again after the device's primary
 * context was replaced, e.g. by cudaDeviceReset); make that first call before
 * any stream capture.  Each call clears the counter header with a
 * stream-ordered memset before its launch, so a call after one that reported
 * CAI_DEVERR_TIMEOUT starts clean.  All calls share the array and it keeps the
 * last call's contents: calls whose kernels overlap on the GPU (unordered
 * streams) race on it.  A device index of 64 or more returns
 * CAI_ERR_UNSUPPORTED; a failed address lookup returns CAI_ERR_CUDA with the
 * error in cai_last_cuda_error(). */
#define CAI_NO_ALLOC_SCRATCH_BYTES (32u << 20)
cai_status cai_mqa_decode_no_alloc(const cai_kv_pool* pools, int32_t num_pools, const int32_t* layer_to_pool,
                                   int32_t num_layers, int32_t layer, const uint16_t* q, int32_t batch,
                                   int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                                   const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                                   float* out, float* lse_out, int32_t* err_flag, void* stream);

/* Bytes of workspace cai_mqa_prefill_chunk needs: a contiguous 16-bit copy of
 * the K and V codes and the scales of up to max_pages_per_seq * page_size keys
 * per sequence (rounded up to 128).  Arguments as for cai_mqa_prefill_chunk. */
size_t cai_mqa_prefill_workspace_size(int32_t batch, int32_t max_pages_per_seq, int32_t page_size);

/* Attention for a chunk of new tokens appended on top of a reused prefix.
 * Prefix caching (Red Hat page, "3. Cache de prefixo") and the cross-turn
 * cache ("Character.AI: inference optimization", 04): the prefix K/V is read
 * from the int8 cache, not recomputed.  The chunk's own K/V must already be
 * appended (cai_kv_append with start_pos = prefix_len), so prefix and chunk
 * keys are read from the same int8 pages.  New token i of sequence b sits at
 * position p0 + i (p0 = prefix_len[b]) and attends keys [lo, p0 + i] with
 * lo = 0 (window 0) or max(0, p0 + i + 1 - window).
 *   q           bf16 bits [batch][n_new][num_q_heads][head_dim], 16-byte aligned
 *   num_q_heads a power of two from 1 to 128
 *   block_table int32 [batch][max_pages_per_seq]; prefix_len int32 [batch]
 *   workspace   device scratch of cai_mqa_prefill_workspace_size() bytes, 256-byte aligned
 *   out         fp32 [batch][n_new][num_q_heads][head_dim], 16-byte aligned
 *   lse_out     fp32 [batch][n_new][num_q_heads], natural log, nullable
 * A sequence whose prefix_len + n_new exceeds the table sets CAI_DEVERR_LENGTH and
 * gets out = 0, lse = -inf. */
cai_status cai_mqa_prefill_chunk(const cai_kv_pool* pool, const uint16_t* q, int32_t batch, int32_t n_new,
                                 int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                                 const int32_t* prefix_len, int32_t window, float softmax_scale, void* workspace,
                                 size_t workspace_bytes, float* out, float* lse_out, int32_t* err_flag,
                                 void* stream);

/* Grouped-query attention: num_kv_heads K/V heads, each shared by a group of
 * G = num_q_heads / num_kv_heads query heads (query heads [j*G, (j+1)*G) read KV head
 * j).  The pages compare Multi-Query Attention, one K/V head for all query heads,
 * against it: MQA keeps the KV cache 8X smaller than the grouped-query attention of
 * most open models ("Character.AI: inference optimization", section 03 and its
 * technique table).  Each KV head lives in its own pool (same page size and page
 * count, same block table and lengths) and is appended with cai_kv_append like an MQA
 * buffer; with num_kv_heads = 1 this is cai_mqa_decode.
 *   kv_pools    host array [num_kv_heads], 1 <= num_kv_heads <= 8
 *   num_q_heads a multiple of num_kv_heads with G <= 64
 *   q, out, lse_out, block_table, ctx_len, window, num_splits as cai_mqa_decode
 *   workspace   device scratch of cai_gqa_decode_workspace_size() bytes, 256-byte aligned,
 *               first 256 bytes zero before the first use (kept zero by every call) */
size_t cai_gqa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t max_pages_per_seq, int32_t page_size, int32_t window,
                                     int32_t num_splits);
cai_status cai_gqa_decode(const cai_kv_pool* kv_pools, int32_t num_kv_heads, const uint16_t* q, int32_t batch,
                          int32_t num_q_heads, const int32_t* block_table, int32_t max_pages_per_seq,
                          const int32_t* ctx_len, int32_t window, float softmax_scale, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, float* out, float* lse_out, int32_t* err_flag,
                          void* stream);

/* Continuous batching: the same attention for a batch whose sequences bring different
 * numbers of new tokens in one call -- decode steps (one token) next to prefill
 * chunks (Red Hat page, "2. Processamento contínuo em lotes" and its figure 7:
 * finished requests leave and new ones join as slots free up, instead of the whole
 * batch waiting for its slowest request).  Sequence b owns new-token rows [q_offsets[b], q_offsets[b+1])
 * of q, out and lse_out (packed), its token i sits at position prefix_len[b] + i and
 * attends as in cai_mqa_prefill_chunk.  Its K/V must already be appended.
 *   q           bf16 bits [total_new][num_q_heads][head_dim], 16-byte aligned
 *   q_offsets   int32 [batch + 1] (device), non-decreasing, q_offsets[batch] <= total_new
 *   max_new     host bound on q_offsets[b+1] - q_offsets[b] (sizes the launch)
 *   out         fp32 [total_new][num_q_heads][head_dim], 16-byte aligned;
 *               lse_out fp32 [total_new][num_q_heads], nullable
 * Other arguments, workspace and limits as cai_mqa_prefill_chunk.  A sequence whose
 * offsets are out of order, beyond total_new or longer than max_new, or whose
 * prefix_len + length exceeds the table, sets CAI_DEVERR_LENGTH; its rows (if its
 * offsets are valid) get out = 0, lse = -inf.  With num_q_heads <= 64 the sequences with
 * exactly one new token run through the decode kernel and the prefill kernel skips
 * them (the results are the same either way): on `stream`, the prefill's key copy and
 * attention launches, then the decode launch (and its split combine), which shares no
 * memory with the prefill and starts on the SMs that the prefill's CTAs leave; it ends
 * after the prefill, so work later in the stream finds both complete. */
cai_status cai_mqa_prefill_varlen(const cai_kv_pool* pool, const uint16_t* q, int32_t batch,
                                  const int32_t* q_offsets, int32_t total_new, int32_t max_new, int32_t num_q_heads,
                                  const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* prefix_len,
                                  int32_t window, float softmax_scale, void* workspace, size_t workspace_bytes,
                                  float* out, float* lse_out, int32_t* err_flag, void* stream);

/* ---- Cross-turn KV cache in host memory ----------------------------------
 * "Character.AI: inference optimization", 04 Cache between turns: the KV of
 * every processed prefix and generated message is kept in host memory in an
 * LRU cache with a tree structure, indexed by a rolling hash of the prefix
 * tokens; a query retrieves the longest matching prefix.  Here the tree's
 * edges are whole pages (page_size tokens, all KV buffers of a layer stack);
 * matches are confirmed token by token, so hash collisions cannot return the
 * wrong KV; eviction removes the least recently used leaf.  Restored pages are
 * byte-identical to the stored ones.  The cache owns a host arena of
 * capacity_pages * num_buffers * cai_page_bytes() bytes (pinned when a GPU is
 * present).  Calls on one cache are serialised by a mutex. */
typedef struct cai_host_cache cai_host_cache;

/* NULL on bad arguments or when the arena cannot be allocated. */
cai_host_cache* cai_host_cache_create(int32_t page_size, int32_t head_dim, int32_t num_buffers,
                                      int64_t capacity_pages);
void cai_host_cache_destroy(cai_host_cache* cache);

/* Tokens of the longest cached prefix of tokens[0, n_tokens): a multiple of page_size
 * (0 on a miss).  Marks the matched path as recently used. */
int32_t cai_host_cache_match(cai_host_cache* cache, const int32_t* tokens, int32_t n_tokens);

/* Copy the cached pages of tokens[0, n_tokens) (n_tokens a multiple of page_size, all
 * cached) into pages block_table_row[0 .. n_tokens/page_size) of each of the num_buffers
 * pools.  block_table_row and pools are host arrays; pools[i].pages may be device or
 * host memory.  Device copies are asynchronous on `stream`: a copy kernel reads the
 * pinned host arena directly (the arena must stay alive until they are done). */
cai_status cai_host_cache_restore(cai_host_cache* cache, const int32_t* tokens, int32_t n_tokens,
                                  const cai_kv_pool* pools, const int32_t* block_table_row, void* stream);

/* cai_host_cache_restore for several sequences at once (a scheduler resuming a batch of
 * dialogues): sequence i copies its cached pages of tokens[i][0, n_tokens[i]) into pages
 * block_table_rows[i][...] of each pool.  tokens, n_tokens and block_table_rows are host
 * arrays [num_seqs]; every path is checked before anything is copied (CAI_ERR_INVALID_ARG
 * when one is not fully cached).  The device copies of all the sequences are queued on
 * `stream` together (one copy kernel per 1024 pages). */
cai_status cai_host_cache_restore_batch(cai_host_cache* cache, int32_t num_seqs, const int32_t* const* tokens,
                                        const int32_t* n_tokens, const cai_kv_pool* pools,
                                        const int32_t* const* block_table_rows, void* stream);

/* Keep the full pages of tokens[0, n_tokens) (a trailing partial page is ignored), read
 * from pages block_table_row[...] of each pool; pages already cached are not copied
 * again.  Evicts least recently used leaves when the arena is full; returns
 * CAI_ERR_WORKSPACE if the path alone does not fit.  Returns after the copies are done. */
cai_status cai_host_cache_store(cai_host_cache* cache, const int32_t* tokens, int32_t n_tokens,
                                const cai_kv_pool* pools, const int32_t* block_table_row, void* stream);

/* Counters: matches with at least one page, matches with none, pages held, evictions. */
void cai_host_cache_stats(cai_host_cache* cache, int64_t* hits, int64_t* misses, int64_t* pages_cached,
                          int64_t* evictions);

/* ---- Local-window page recycling.
 * A local layer attends only the last `window` positions ("Character.AI: inference
 * optimization", section 03, hybrid attention with a 1024-token horizon), so a buffer
 * read only by local layers needs to keep just the pages of that window.  It can hold
 * each sequence in a ring of pages: logical page k of the sequence lives in ring slot
 * k % ring.  The kernels read no page outside the call's own range: decode reads the
 * pages of [ctx_len - window, ctx_len), prefill those of
 * [max(0, prefix + 1 - window), prefix + n_new), append those it writes.  (The pages
 * describe the horizon but not how freed memory is reused; this ring is that reuse.) */

/* Ring length (pages per sequence) for a local buffer read with `window` and written at
 * most `max_new_tokens` positions per call (1 for decode, the chunk length for prefill):
 * ceil((window + max_new_tokens - 1) / page_size) + 1.  0 for invalid arguments
 * (window < 1, max_new_tokens < 1, page_size < 1). */
int32_t cai_ring_pages(int32_t window, int32_t page_size, int32_t max_new_tokens);

/* Fill one host block-table row for a sequence whose positions [0, hi) are written
 * (hi includes the tokens of the coming call): the last `ring` pages before
 * ceil(hi / page_size) map to ring_ids[k % ring]; every other entry is -1, so that a
 * kernel reading a freed or unwritten page sets CAI_DEVERR_PAGE instead of reading
 * another position's data.  row: host int32 [max_pages_per_seq]; ring_ids: host int32
 * [ring], distinct page ids of the buffer's pool.  Returns CAI_ERR_INVALID_ARG for null
 * pointers, ring < 1, page_size < 1, hi < 0 or ceil(hi / page_size) > max_pages_per_seq. */
cai_status cai_ring_table_row(int32_t* row, int32_t max_pages_per_seq, const int32_t* ring_ids, int32_t ring,
                              int32_t hi, int32_t page_size);

/* Limit, in nanoseconds, of every bounded wait inside the decode and prefill kernels
 * (process-wide, read at each launch; 0 restores the default of 2 s; a wait checks its
 * clock after each suspension of up to 1 ms, so shorter limits act as about 1 ms).  A
 * CTA whose wait runs out sets CAI_DEVERR_TIMEOUT, stops its work, waits for its own
 * copies and tensor-core operations in flight, frees its tensor memory and returns;
 * that launch's outputs are unspecified.  A short limit is for failure-detection
 * tests; a serving process leaves the default. */
void cai_set_wait_limit_ns(uint64_t ns);

/* Fault injection for failure-detection tests (process-wide, read at each launch;
 * -1, the default, turns it off).  With stage = n >= 0, every CTA of the following
 * decode launches skips the load of its n-th K/V stage (64 tokens), and every CTA of
 * the following prefill launches skips the load of its n-th K tile (128 keys); the
 * waits for them run out after the wait limit and the launch reports
 * CAI_DEVERR_TIMEOUT.  Nothing faults: the load is simply never issued.  A CTA with
 * fewer stages than n + 1 is not affected. */
void cai_set_fault_injection(int32_t stage);

/* The CUDA runtime's description of the error behind the last CAI_ERR_CUDA returned on
 * this thread ("no error" if none). */
const char* cai_last_cuda_error(void);

/* Static description of a status code. */
const char* cai_status_string(cai_status status);

#ifdef __cplusplus
}
#endif

#endif /* CAI_H_ */
