// Chunked append-prefill attention on a reused prefix.
//
// What it computes (definition): new token i of sequence b sits at absolute
// position p0 + i (p0 = prefix length) and, for each query head h, attends
// the keys [lo, p0 + i] of its own sequence, where lo = 0 for a global layer
// or max(0, p0 + i + 1 - window) for a local one: softmax of
// softmax_scale * <q, s_k[t] * k_code[t]> and the weighted sum of
// s_v[t] * v_code[t].  The prefix keys are read back from the int8 cache, not
// recomputed (prefix caching, Red Hat page "3. Cache de prefixo"; cross-turn
// cache, "Character.AI: inference optimization" section 04), and the chunk's
// own keys were appended to the same pages before this call.
//
// How:
//  1. dequant pass: the sequence's int8 pages are copied, exactly, into a
//     contiguous scratch copy: K as bf16 [B][KT][128], V as fp16 [B][KT][128]
//     and both scale rows as fp32 [B][KT].  The scales stay separate so every
//     logit and weight is formed in fp32 exactly as in the definition.
//  2. attention: one CTA per 128 query rows of a sequence, a row being one
//     (new token, head) pair.  128-key tiles of K and V arrive by TMA tensor
//     loads (cp.async.bulk.tensor) straight into the canonical no-swizzle
//     tcgen05 operand layout; S = Q K^T runs as tcgen05.mma kind::f16 (bf16,
//     M = N = 128, K = 128) into tensor memory; the online softmax (one thread
//     per row) applies the per-key scale, the causal/window mask and the
//     per-key V scale, and writes P (fp16) back into tensor memory, where it is
//     the A operand of O += P V (fp16, V from shared memory, MN-major).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace cai {
namespace {

constexpr int kRows = 128;                 // query rows per CTA (MMA M)
constexpr int kKeys = 128;                 // keys per tile (MMA N of S, K of PV)
constexpr int kTileBytes = kKeys * kHeadDim * 2;  // 32 KB of 16-bit values
constexpr int kStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kRows * kHeadDim * 2;
constexpr int kStageBytes = 2 * kTileBytes + 2 * kKeys * 4;  // K, V, K scales, V scales
constexpr int kOffBars = kOffStage + kStages * kStageBytes;  // full[2], s_bar, pv_bar
constexpr int kOffMisc = kOffBars + 8 * (kStages + 2);
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;

struct PrefillParams {
  const uint8_t* pages;
  int32_t num_pages, page_size, max_pages;
  const int32_t* table;
  const int32_t* prefix_len;
  const uint16_t* q;  // bf16 [B][n_new][Hq][128]
  int32_t batch, n_new, num_heads, log2_heads, window, kt_rows;
  float scale_log2;
  uint16_t* kb;  // scratch bf16 [B][KT][128]
  uint16_t* vh;  // scratch fp16 [B][KT][128]
  float* ks;     // scratch [B][KT]
  float* vs;     // scratch [B][KT]
  float* out;
  float* lse_out;
  int32_t* err;
};

__device__ __forceinline__ bool seq_ok(const PrefillParams& p, int32_t p0) {
  return p0 >= 0 && (int64_t)p0 + p.n_new <= (int64_t)p.max_pages * p.page_size;
}

// One warp per scratch row (sequence b, key t).
__global__ void __launch_bounds__(256) dequant_kernel(const PrefillParams p) {
  const int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (int64_t)p.batch * p.kt_rows) return;
  const int b = (int)(row / p.kt_rows);
  const int t = (int)(row - (int64_t)b * p.kt_rows);
  const int32_t p0 = p.prefix_len[b];
  const bool ok = seq_ok(p, p0);
  if (!ok) {
    if (t == 0 && lane == 0 && p.err) atomicOr(p.err, CAI_DEVERR_LENGTH);
    return;
  }
  const int len = p0 + p.n_new;
  if (t >= ((len + kKeys - 1) / kKeys) * kKeys) return;  // never read
  if (p.window > 0) {
    const int lo_min = max(0, p0 + 1 - p.window);
    if (t < (lo_min / kKeys) * kKeys) return;  // before every window
  }
  uint32_t kw = 0, vw = 0;
  float ksc = 0.0f, vsc = 0.0f;
  if (t < len) {
    const int P = p.page_size;
    const int32_t page = p.table[(int64_t)b * p.max_pages + t / P];
    if (page >= 0 && page < p.num_pages) {
      const int slot = t % P;
      const uint8_t* pg = p.pages + (int64_t)page * page_bytes(P);
      kw = reinterpret_cast<const uint32_t*>(pg + slot * kHeadDim)[lane];
      vw = reinterpret_cast<const uint32_t*>(pg + P * kHeadDim + slot * kHeadDim)[lane];
      const float* sc = reinterpret_cast<const float*>(pg + 2 * P * kHeadDim);
      ksc = sc[slot];
      vsc = sc[P + slot];
    } else if (lane == 0 && p.err) {
      atomicOr(p.err, CAI_DEVERR_PAGE);
    }
  }
  // int8 -> bf16 (K) and int8 -> fp16 (V): exact for |code| <= 127.
  uint16_t kb[4], vh[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float kf = (float)(int8_t)(kw >> (8 * e));
    const float vf = (float)(int8_t)(vw >> (8 * e));
    kb[e] = (uint16_t)(__float_as_uint(kf) >> 16);  // small integers: the top half is exact
    const __half hv = __float2half_rn(vf);
    vh[e] = *reinterpret_cast<const uint16_t*>(&hv);
  }
  const int64_t off = row * kHeadDim + lane * 4;
  *reinterpret_cast<uint2*>(p.kb + off) = make_uint2(kb[0] | ((uint32_t)kb[1] << 16), kb[2] | ((uint32_t)kb[3] << 16));
  *reinterpret_cast<uint2*>(p.vh + off) = make_uint2(vh[0] | ((uint32_t)vh[1] << 16), vh[2] | ((uint32_t)vh[3] << 16));
  if (lane == 0) {
    p.ks[row] = ksc;
    p.vs[row] = vsc;
  }
}

__device__ __forceinline__ void tma_load_rows128(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(0), "r"(smem_addr(bar))
      : "memory");
}

// Operand tiles in shared memory: element (r, k) of a 128x128 16-bit tile at
// (k/8)*2048 + r*16 + (k%8)*2 -- the order a [16 chunks][128 rows][8] TMA box
// writes.  As a K-major operand: LBO = 2048 (next 8 k), SBO = 128 (next 8 rows).
// As an MN-major operand (rows = K, k = N): LBO = 128, SBO = 2048.
__global__ void __launch_bounds__(128, 1) prefill_kernel(const PrefillParams p,
                                                         const __grid_constant__ CUtensorMap kmap,
                                                         const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem + kOffQ;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* s_bar = full + kStages;
  uint64_t* pv_bar = full + kStages + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int32_t* timeout = reinterpret_cast<int32_t*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int b = blockIdx.y;
  const int Hq = p.num_heads;
  const int row0 = blockIdx.x * kRows;  // first (token, head) row of this CTA within the sequence
  const int i0 = row0 >> p.log2_heads;
  const int32_t p0 = p.prefix_len[b];
  const int my_i = (row0 + tid) >> p.log2_heads;
  const int my_h = (row0 + tid) & (Hq - 1);
  const bool my_row = my_i < p.n_new;
  float* out_row = p.out + (((int64_t)b * p.n_new + my_i) * Hq + my_h) * kHeadDim;

  if (!seq_ok(p, p0)) {  // flagged by the dequant pass; outputs defined as 0 / -inf
    if (my_row) {
      for (int d = 0; d < kHeadDim; d += 4) *reinterpret_cast<float4*>(out_row + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.lse_out) p.lse_out[((int64_t)b * p.n_new + my_i) * Hq + my_h] = -INFINITY;
    }
    return;
  }
  const int i_last = min(i0 + (kRows >> p.log2_heads), p.n_new) - 1;
  const int kv_hi = p0 + i_last + 1;
  const int kv_lo = p.window > 0 ? max(0, p0 + i0 + 1 - p.window) : 0;
  const int kt0 = kv_lo / kKeys;
  const int nkt = (kv_hi - 1) / kKeys - kt0 + 1;
  const int64_t seq_row0 = (int64_t)b * p.kt_rows;

  const int q_pos = p0 + my_i;
  const int k_lo = p.window > 0 ? max(0, q_pos + 1 - p.window) : 0;

  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    mbar_init(s_bar, 1);
    mbar_init(pv_bar, 1);
    *timeout = 0;
    fence_barrier_init();
  }
  // Q tile (bf16), rows beyond the chunk zero.
  {
    const uint16_t* qb = p.q + ((int64_t)b * p.n_new * Hq + row0) * kHeadDim;
    const int rows_here = min(kRows, p.n_new * Hq - row0);
    for (int u = tid; u < kRows * 16; u += blockDim.x) {
      const int r = u >> 4, c = u & 15;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (r < rows_here) w = *reinterpret_cast<const uint4*>(qb + (int64_t)r * kHeadDim + c * 8);
      *reinterpret_cast<uint4*>(qs + c * 2048 + r * 16) = w;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = (uint32_t)(warp * 32) << 16;

  auto issue = [&](int j) {
    const int stage = j % kStages;
    uint8_t* st = smem + kOffStage + stage * kStageBytes;
    const int kt = kt0 + j;
    mbar_arrive_expect_tx(&full[stage], kStageBytes);
    tma_load_rows128(st, &kmap, (int)(seq_row0 + (int64_t)kt * kKeys), &full[stage]);
    tma_load_rows128(st + kTileBytes, &vmap, (int)(seq_row0 + (int64_t)kt * kKeys), &full[stage]);
    bulk_g2s(st + 2 * kTileBytes, p.ks + seq_row0 + (int64_t)kt * kKeys, kKeys * 4, &full[stage]);
    bulk_g2s(st + 2 * kTileBytes + kKeys * 4, p.vs + seq_row0 + (int64_t)kt * kKeys, kKeys * 4, &full[stage]);
  };
  if (tid == 0) {
    issue(0);
    if (nkt > 1) issue(1);
  }

  float m_ref = -INFINITY, l_sum = 0.0f;
  bool ok_all = true;
  for (int j = 0; j < nkt; ++j) {
    const int stage = j % kStages;
    uint8_t* st = smem + kOffStage + stage * kStageBytes;
    const float* kscale = reinterpret_cast<const float*>(st + 2 * kTileBytes);
    const float* vscale = kscale + kKeys;
    if (!mbar_wait(&full[stage], (j / kStages) & 1)) ok_all = false;
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(kRows, kKeys, 0, 0);
      const uint32_t qa = smem_addr(qs), ka = smem_addr(st);
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks)
        mma_f16_ss(tmem + kColS, smem_desc(qa + ks * 4096, 2048, 128), smem_desc(ka + ks * 4096, 2048, 128), idesc,
                   ks > 0);
      mma_commit(s_bar);
    }
    if (!mbar_wait(s_bar, j & 1)) ok_all = false;
    if (j > 0 && !mbar_wait(pv_bar, (j - 1) & 1)) ok_all = false;
    tc_fence_after();
    if (tid == 0 && j > 0 && j + 1 < nkt) issue(j + 1);  // into the stage tile j-1 used

    // ---- softmax of this thread's row over the 128 keys of the tile
    const int key0 = (kt0 + j) * kKeys;
    float z[kKeys];
#pragma unroll
    for (int c = 0; c < kKeys; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + t_lane + kColS + c, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) z[c + e] = __uint_as_float(r[e]) * (kscale[c + e] * p.scale_log2);
    }
    const bool full_tile = key0 >= k_lo && key0 + kKeys - 1 <= q_pos;
    if (!full_tile) {
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        const int key = key0 + c;
        if (key < k_lo || key > q_pos) z[c] = -INFINITY;
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kKeys; ++c) mx = fmaxf(mx, z[c]);
    const bool raise = mx > m_ref + kRescaleThreshold;
    const float alpha = raise ? ex2_approx(m_ref - mx) : 1.0f;
    if (j > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
      for (int c = 0; c < kHeadDim; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + t_lane + kColO + c, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st_32x32b_x32(tmem + t_lane + kColO + c, o);
      }
      tmem_wait_st();
    }
    if (raise) {
      l_sum *= alpha;
      m_ref = mx;
    }
    const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
#pragma unroll
    for (int c = 0; c < kKeys; c += 64) {
      uint32_t pw[32];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        const float a = ex2_approx(z[c + e] - m_use), bb = ex2_approx(z[c + e + 1] - m_use);
        l_sum += a + bb;
        pw[e / 2] = pack_f16x2(a * vscale[c + e], bb * vscale[c + e + 1]);
      }
      tmem_st_32x32b_x32(tmem + t_lane + kColP + c / 2, pw);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_f16_f32(kRows, kHeadDim, 0, 1);
      const uint32_t va = smem_addr(st + kTileBytes);
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks)
        mma_f16_ts(tmem + kColO, tmem + kColP + ks * 8, smem_desc(va + ks * 256, 128, 2048), idesc,
                   (j > 0 || ks > 0) ? 1u : 0u);
      mma_commit(pv_bar);
    }
  }
  if (!mbar_wait(pv_bar, (nkt - 1) & 1)) ok_all = false;
  tc_fence_after();
  if (!ok_all) atomicOr(timeout, 1);

  const float inv = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
#pragma unroll
  for (int c = 0; c < kHeadDim; c += 32) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tmem + t_lane + kColO + c, o);
    tmem_wait_ld();
    if (my_row) {
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(out_row + c + e) =
            make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                        __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
    }
  }
  if (my_row && p.lse_out)
    p.lse_out[((int64_t)b * p.n_new + my_i) * Hq + my_h] = l_sum > 0.0f ? (m_ref + __log2f(l_sum)) * kLn2 : -INFINITY;
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *timeout && p.err) atomicOr(p.err, CAI_DEVERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// A [rows][128] 16-bit row-major matrix seen as (8 elements, rows, 16 chunks)
// so that a (8, 128, 16) box lands in shared memory as [chunk][row][8].
bool encode_rows128(CUtensorMap* map, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {8, rows, 16};
  cuuint64_t strides[2] = {kHeadDim * 2, 16};
  cuuint32_t box[3] = {8, (cuuint32_t)kRows, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_workspace_bytes(int32_t batch, int32_t max_pages_per_seq, int32_t page_size) {
  const int64_t kt = ((int64_t)max_pages_per_seq * page_size + kKeys - 1) / kKeys * kKeys;
  const int64_t rows = (int64_t)batch * kt;
  const int64_t a = ((rows * kHeadDim * 2 + 255) / 256) * 256;
  const int64_t s = ((rows * 4 + 255) / 256) * 256;
  return (size_t)(2 * a + 2 * s);
}

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t stream) {
  PrefillParams p;
  p.pages = L.pages;
  p.num_pages = L.num_pages;
  p.page_size = L.page_size;
  p.max_pages = L.max_pages;
  p.table = L.table;
  p.prefix_len = L.prefix_len;
  p.q = L.q;
  p.batch = L.batch;
  p.n_new = L.n_new;
  p.num_heads = L.num_heads;
  p.log2_heads = 31 - __builtin_clz((unsigned)L.num_heads);
  p.window = L.window;
  p.kt_rows = (int32_t)(((int64_t)L.max_pages * L.page_size + kKeys - 1) / kKeys * kKeys);
  p.scale_log2 = L.scale_log2;
  const int64_t rows = (int64_t)L.batch * p.kt_rows;
  const int64_t a = ((rows * kHeadDim * 2 + 255) / 256) * 256;
  const int64_t s = ((rows * 4 + 255) / 256) * 256;
  uint8_t* ws = static_cast<uint8_t*>(L.workspace);
  p.kb = reinterpret_cast<uint16_t*>(ws);
  p.vh = reinterpret_cast<uint16_t*>(ws + a);
  p.ks = reinterpret_cast<float*>(ws + 2 * a);
  p.vs = reinterpret_cast<float*>(ws + 2 * a + s);
  p.out = L.out;
  p.lse_out = L.lse_out;
  p.err = L.err;

  CUtensorMap kmap, vmap;
  if (!encode_rows128(&kmap, p.kb, (uint64_t)rows) || !encode_rows128(&vmap, p.vh, (uint64_t)rows))
    return cudaErrorInvalidValue;

  const int64_t warps = rows;
  dequant_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int qtiles = (L.n_new * L.num_heads + kRows - 1) / kRows;
  prefill_kernel<<<dim3(qtiles, L.batch), 128, kSmemBytes, stream>>>(p, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace cai
