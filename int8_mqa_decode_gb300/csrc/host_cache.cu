// Cross-turn KV cache in host memory.
//
// "Character.AI: inference optimization", 04 Cache between turns: for every
// processed prefix and every generated message the KV values stay in host
// memory and are retrieved by later queries; they are organised as an LRU
// cache with a tree structure, indexed by a rolling hash of the prefix
// tokens, and a query takes the longest matching prefix, which lets even
// partly identical messages reuse their common part.
//
// Here the tree's edges are whole KV pages: node k on a path holds page k of
// a token sequence (page_size tokens) for every KV buffer, and its key is a
// rolling hash chained over the pages before it, h_k = mix(h_{k-1}, page k's
// tokens).  Lookups walk the tree from the root by hash and confirm each step
// by comparing the page's tokens, so a hash collision can never return the
// wrong KV.  Eviction takes the least recently used leaf (a page whose longer
// continuations are all gone), so a cached path never has holes.  Pages live
// in one host arena, pinned when a GPU is present.  Copies between the arena
// and device pools are done by a copy kernel that reads (restore) or writes
// (store) the pinned arena directly through its device mapping, up to 1024
// pages per launch, the page list passed as kernel parameters (one small
// cudaMemcpyAsync per page had made a long prefix thousands of calls); plain
// memcpy when both sides are host memory.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <list>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "cai.h"

namespace {

uint64_t mix64(uint64_t z) {  // splitmix64 finaliser (Steele, Lea, Flood 2014)
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t chain_hash(uint64_t parent, const int32_t* tok, int n) {
  uint64_t h = parent ^ 0x9E3779B97F4A7C15ull;
  for (int i = 0; i < n; ++i) h = mix64(h + (uint64_t)(uint32_t)tok[i] + 0x9E3779B97F4A7C15ull * (i + 1));
  return h;
}

bool is_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool copy_bytes(void* dst, const void* src, size_t n, cudaStream_t stream) {
  if (!is_device(dst) && !is_device(src)) {
    std::memcpy(dst, src, n);
    return true;
  }
  return cudaMemcpyAsync(dst, src, n, cudaMemcpyDefault, stream) == cudaSuccess;
}

// Page copies of one launch: every byte of each source page to its destination page
// (pinned host <-> device, both addresses 16-byte aligned, page_bytes a multiple of 16).
constexpr int kCopyBatch = 1024;
struct PageCopies {
  const uint8_t* src[kCopyBatch];
  uint8_t* dst[kCopyBatch];
  int32_t n;
  int32_t page_bytes;
};

__global__ void __launch_bounds__(256) page_copy_kernel(const __grid_constant__ PageCopies c) {
  const int units = c.page_bytes / 16;
  for (int i = blockIdx.x; i < c.n; i += gridDim.x) {
    const uint4* s = reinterpret_cast<const uint4*>(c.src[i]);
    uint4* d = reinterpret_cast<uint4*>(c.dst[i]);
    for (int k = threadIdx.x; k < units; k += blockDim.x) d[k] = s[k];
  }
}

// Copies the listed pages on `stream`, kCopyBatch per launch.
class PageCopier {
 public:
  PageCopier(int32_t page_bytes, cudaStream_t stream) : stream_(stream) {
    batch_.n = 0;
    batch_.page_bytes = page_bytes;
  }
  bool add(const uint8_t* src, uint8_t* dst) {
    batch_.src[batch_.n] = src;
    batch_.dst[batch_.n] = dst;
    return ++batch_.n < kCopyBatch || flush();
  }
  bool flush() {
    if (batch_.n == 0) return true;
    const int blocks = batch_.n < 1024 ? batch_.n : 1024;
    page_copy_kernel<<<blocks, 256, 0, stream_>>>(batch_);
    batch_.n = 0;
    return cudaGetLastError() == cudaSuccess;
  }

 private:
  PageCopies batch_;
  cudaStream_t stream_;
};

struct Node {
  int parent = -1;
  uint64_t hash = 0;
  std::vector<int32_t> tokens;              // the page's tokens (page_size of them)
  std::unordered_map<uint64_t, int> kids;  // child hash -> node id
  int64_t slot = -1;                        // page slot in the arena
  std::list<int>::iterator lru;             // position in the LRU list (leaves and inner nodes)
};

}  // namespace

struct cai_host_cache {
  int32_t page_size, head_dim, num_buffers;
  size_t page_bytes, capacity;
  uint8_t* arena = nullptr;
  bool pinned = false;
  std::vector<int64_t> free_slots;
  std::vector<Node> nodes;  // node 0 is the root (no page)
  std::vector<int> free_nodes;
  std::list<int> lru;       // front = most recently used
  int64_t hits = 0, misses = 0, evictions = 0;
  std::mutex mu;

  uint8_t* slot_ptr(int64_t slot, int buf) { return arena + ((size_t)slot * num_buffers + buf) * page_bytes; }

  // Child of `parent` holding exactly these page tokens, or -1.
  int find_child(int parent, const int32_t* tok) {
    const uint64_t h = chain_hash(nodes[parent].hash, tok, page_size);
    auto it = nodes[parent].kids.find(h);
    if (it == nodes[parent].kids.end()) return -1;
    const Node& c = nodes[it->second];
    if (std::memcmp(c.tokens.data(), tok, sizeof(int32_t) * page_size) != 0) return -1;
    return it->second;
  }

  void touch(int id) {
    lru.erase(nodes[id].lru);
    lru.push_front(id);
    nodes[id].lru = lru.begin();
  }

  // Free the least recently used leaf other than `keep`; false if there is none.
  bool evict_one(int keep) {
    for (auto it = lru.rbegin(); it != lru.rend(); ++it) {
      const int id = *it;
      if (id == keep || !nodes[id].kids.empty()) continue;
      Node& n = nodes[id];
      nodes[n.parent].kids.erase(n.hash);
      free_slots.push_back(n.slot);
      lru.erase(n.lru);
      n = Node();
      free_nodes.push_back(id);
      ++evictions;
      return true;
    }
    return false;
  }
};

extern "C" {

cai_host_cache* cai_host_cache_create(int32_t page_size, int32_t head_dim, int32_t num_buffers,
                                      int64_t capacity_pages) {
  if (page_size <= 0 || head_dim <= 0 || num_buffers <= 0 || capacity_pages <= 0) return nullptr;
  cai_host_cache* c = new cai_host_cache();
  c->page_size = page_size;
  c->head_dim = head_dim;
  c->num_buffers = num_buffers;
  c->page_bytes = cai_page_bytes(page_size, head_dim);
  c->capacity = (size_t)capacity_pages;
  const size_t bytes = c->capacity * num_buffers * c->page_bytes;
  void* p = nullptr;
  if (cudaMallocHost(&p, bytes) == cudaSuccess) {
    c->pinned = true;
  } else {
    cudaGetLastError();
    p = std::malloc(bytes);
  }
  if (!p) {
    delete c;
    return nullptr;
  }
  c->arena = static_cast<uint8_t*>(p);
  for (int64_t s = (int64_t)c->capacity - 1; s >= 0; --s) c->free_slots.push_back(s);
  c->nodes.emplace_back();  // root
  c->nodes[0].hash = 0x243F6A8885A308D3ull;
  return c;
}

void cai_host_cache_destroy(cai_host_cache* c) {
  if (!c) return;
  if (c->pinned)
    cudaFreeHost(c->arena);
  else
    std::free(c->arena);
  delete c;
}

int32_t cai_host_cache_match(cai_host_cache* c, const int32_t* tokens, int32_t n_tokens) {
  if (!c || !tokens || n_tokens < 0) return 0;
  std::lock_guard<std::mutex> lock(c->mu);
  int node = 0, pages = 0;
  for (int32_t off = 0; off + c->page_size <= n_tokens; off += c->page_size) {
    const int child = c->find_child(node, tokens + off);
    if (child < 0) break;
    node = child;
    ++pages;
  }
  for (int id = node; id > 0; id = c->nodes[id].parent) c->touch(id);
  if (pages > 0)
    ++c->hits;
  else
    ++c->misses;
  return pages * c->page_size;
}

namespace {

// The cached path of tokens[0, n_tokens) checked against the pools and the table row;
// CAI_OK with the path's nodes, or the status to return (nothing copied).
cai_status restore_path(cai_host_cache* c, const int32_t* tokens, int32_t n_tokens, const cai_kv_pool* pools,
                        const int32_t* block_table_row, std::vector<int>& path) {
  if (!tokens || !block_table_row || n_tokens < 0 || n_tokens % c->page_size != 0) return CAI_ERR_INVALID_ARG;
  path.clear();
  int node = 0;
  for (int32_t k = 0; k * c->page_size < n_tokens; ++k) {
    node = c->find_child(node, tokens + (size_t)k * c->page_size);
    if (node < 0) return CAI_ERR_INVALID_ARG;  // not cached (evicted since the match?)
    path.push_back(node);
  }
  for (int b = 0; b < c->num_buffers; ++b) {
    const cai_kv_pool& p = pools[b];
    if (!p.pages || p.page_size != c->page_size || p.head_dim != c->head_dim) return CAI_ERR_INVALID_ARG;
    for (size_t k = 0; k < path.size(); ++k)
      if (block_table_row[k] < 0 || block_table_row[k] >= p.num_pages) return CAI_ERR_INVALID_ARG;
  }
  return CAI_OK;
}

// Queue (or do) the copies of one checked path.
bool restore_copies(cai_host_cache* c, const std::vector<int>& path, const cai_kv_pool* pools,
                    const int32_t* block_table_row, PageCopier& copier, cudaStream_t stream) {
  const bool kernel = c->pinned && (c->page_bytes % 16) == 0;
  for (int b = 0; b < c->num_buffers; ++b) {
    const bool dev = is_device(pools[b].pages);
    for (size_t k = 0; k < path.size(); ++k) {
      uint8_t* dst = static_cast<uint8_t*>(pools[b].pages) + (size_t)block_table_row[k] * c->page_bytes;
      const uint8_t* src = c->slot_ptr(c->nodes[path[k]].slot, b);
      const bool ok = (kernel && dev) ? copier.add(src, dst) : copy_bytes(dst, src, c->page_bytes, stream);
      if (!ok) return false;
    }
  }
  return true;
}

}  // namespace

cai_status cai_host_cache_restore(cai_host_cache* c, const int32_t* tokens, int32_t n_tokens,
                                  const cai_kv_pool* pools, const int32_t* block_table_row, void* stream) {
  if (!c || !pools) return CAI_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  // The whole path must be cached before anything is copied.
  std::vector<int> path;
  const cai_status st = restore_path(c, tokens, n_tokens, pools, block_table_row, path);
  if (st != CAI_OK) return st;
  PageCopier copier((int32_t)c->page_bytes, static_cast<cudaStream_t>(stream));
  if (!restore_copies(c, path, pools, block_table_row, copier, static_cast<cudaStream_t>(stream)))
    return CAI_ERR_CUDA;
  return copier.flush() ? CAI_OK : CAI_ERR_CUDA;
}

cai_status cai_host_cache_restore_batch(cai_host_cache* c, int32_t num_seqs, const int32_t* const* tokens,
                                        const int32_t* n_tokens, const cai_kv_pool* pools,
                                        const int32_t* const* block_table_rows, void* stream) {
  if (!c || !pools || num_seqs < 0 || (num_seqs > 0 && (!tokens || !n_tokens || !block_table_rows)))
    return CAI_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  // Every sequence's path is checked before anything is copied.
  std::vector<std::vector<int>> paths(num_seqs);
  for (int32_t i = 0; i < num_seqs; ++i) {
    const cai_status st = restore_path(c, tokens[i], n_tokens[i], pools, block_table_rows[i], paths[i]);
    if (st != CAI_OK) return st;
  }
  PageCopier copier((int32_t)c->page_bytes, static_cast<cudaStream_t>(stream));
  for (int32_t i = 0; i < num_seqs; ++i)
    if (!restore_copies(c, paths[i], pools, block_table_rows[i], copier, static_cast<cudaStream_t>(stream)))
      return CAI_ERR_CUDA;
  return copier.flush() ? CAI_OK : CAI_ERR_CUDA;
}

cai_status cai_host_cache_store(cai_host_cache* c, const int32_t* tokens, int32_t n_tokens, const cai_kv_pool* pools,
                                const int32_t* block_table_row, void* stream) {
  if (!c || !tokens || !pools || !block_table_row || n_tokens < 0) return CAI_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  int node = 0;
  bool copied = false;
  const bool kernel = c->pinned && (c->page_bytes % 16) == 0;
  PageCopier copier((int32_t)c->page_bytes, static_cast<cudaStream_t>(stream));
  for (int32_t k = 0; (k + 1) * c->page_size <= n_tokens; ++k) {
    const int32_t* tok = tokens + (size_t)k * c->page_size;
    int child = c->find_child(node, tok);
    if (child < 0) {
      // The path so far is never evicted: its inner nodes have children and its end is kept.
      if (c->free_slots.empty() && !c->evict_one(node)) return CAI_ERR_WORKSPACE;
      const int64_t slot = c->free_slots.back();
      c->free_slots.pop_back();
      if (!c->free_nodes.empty()) {
        child = c->free_nodes.back();
        c->free_nodes.pop_back();
      } else {
        child = (int)c->nodes.size();
        c->nodes.emplace_back();
      }
      Node& n = c->nodes[child];
      n.parent = node;
      n.hash = chain_hash(c->nodes[node].hash, tok, c->page_size);
      n.tokens.assign(tok, tok + c->page_size);
      n.slot = slot;
      c->lru.push_front(child);
      n.lru = c->lru.begin();
      c->nodes[node].kids[n.hash] = child;
      for (int b = 0; b < c->num_buffers; ++b) {
        const cai_kv_pool& p = pools[b];
        if (!p.pages || p.page_size != c->page_size || p.head_dim != c->head_dim) return CAI_ERR_INVALID_ARG;
        const int32_t pid = block_table_row[k];
        if (pid < 0 || pid >= p.num_pages) return CAI_ERR_INVALID_ARG;
        const uint8_t* src = static_cast<const uint8_t*>(p.pages) + (size_t)pid * c->page_bytes;
        const bool ok = (kernel && is_device(p.pages))
                            ? copier.add(src, c->slot_ptr(slot, b))
                            : copy_bytes(c->slot_ptr(slot, b), src, c->page_bytes, static_cast<cudaStream_t>(stream));
        if (!ok) return CAI_ERR_CUDA;
        copied = true;
      }
    }
    node = child;
  }
  for (int id = node; id > 0; id = c->nodes[id].parent) c->touch(id);
  if (!copier.flush()) return CAI_ERR_CUDA;
  if (copied && is_device(pools[0].pages) &&
      cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CAI_ERR_CUDA;
  return CAI_OK;
}

void cai_host_cache_stats(cai_host_cache* c, int64_t* hits, int64_t* misses, int64_t* pages_cached,
                          int64_t* evictions) {
  if (!c) return;
  std::lock_guard<std::mutex> lock(c->mu);
  if (hits) *hits = c->hits;
  if (misses) *misses = c->misses;
  if (pages_cached) *pages_cached = (int64_t)(c->capacity - c->free_slots.size());
  if (evictions) *evictions = c->evictions;
}

}  // extern "C"
