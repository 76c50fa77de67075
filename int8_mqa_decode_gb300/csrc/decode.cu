// Split-KV MQA decode over the int8 paged KV cache, and the log-sum-exp
// combine of the splits.
//
// What it computes (definition): for one query token per sequence and each
// query head h, softmax over the attended positions of
//   z_t = softmax_scale * <q_h, s_k[t] * k_code[t]>
// and out_h = sum_t p_t * s_v[t] * v_code[t]  (Red Hat page, "Por que o cache
// KV existe"), where every head reads the same single K/V head (Multi-Query
// Attention) and a local layer attends only the last `window` positions
// (hybrid attention, technique table of "Character.AI: inference
// optimization", section 03).
//
// How (one CTA per (sequence, split); 4 warps; 2 CTAs per SM):
//  * pages of a 64-token tile arrive by 1-D bulk copies (TMA engine) into a
//    3-stage ring; one copy per page brings K codes, V codes and both scale
//    rows, and serves all query heads;
//  * all warps convert the int8 codes to fp16 (exact) into the canonical
//    no-swizzle tcgen05 operand layouts (K: K-major; V: MN-major);
//  * S = Q K^T runs on the tensor cores (tcgen05.mma kind::f16, M = 64 padded
//    heads, N = 64 tokens, K = 128) into tensor memory; the per-token K scale
//    and the softmax scale are applied in fp32 afterwards;
//  * online softmax on S (two threads per head, one shuffle for the row max),
//    with the reference max raised only when a logit exceeds it by 2^8 so that
//    the output accumulator is rarely rescaled; P is scaled by the per-token V
//    scale, rounded to fp16 and stored as the A operand of O += P V;
//  * the split's partial output and log-sum-exp go to the workspace, or
//    straight to `out` when the sequence has a single split.
#include "common.cuh"
#include "ptx.cuh"

namespace cai {
namespace {

constexpr int T = kDecodeTile;                 // tokens per tile
constexpr int NST = kDecodeStages;             // raw stages
constexpr int kRawStageBytes = T * 264;        // 64 tokens of K, V and scales
constexpr int kK16Bytes = T * kHeadDim * 2;    // fp16 K tile
constexpr int kV16Bytes = T * kHeadDim * 2;    // fp16 V tile
constexpr int kQ16Bytes = kDecodeRows * kHeadDim * 2;
constexpr int kP16Bytes = kDecodeRows * T * 2;
constexpr int kOffRaw = 0;
constexpr int kOffK16 = kOffRaw + NST * kRawStageBytes;
constexpr int kOffV16 = kOffK16 + kK16Bytes;
constexpr int kOffQ16 = kOffV16 + kV16Bytes;
constexpr int kOffP16 = kOffQ16 + kQ16Bytes;
constexpr int kOffKsc = kOffP16 + kP16Bytes;
constexpr int kOffVsc = kOffKsc + T * 4;
constexpr int kOffKbias = kOffVsc + T * 4;
constexpr int kOffBars = kOffKbias + T * 4;     // full[NST], s_bar, pv_bar
constexpr int kOffMisc = kOffBars + 8 * (NST + 2);
constexpr int kSmemBytes = kOffMisc + 16 + 1024; // + alignment slack
constexpr uint32_t kTmemCols = 256;             // S: cols [0, 64); O: cols [128, 256)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: p <= 2^8 between rescales

// K-major no-swizzle operand tile with 128 columns (fp16): element (r, k) at
// (r/8)*2048 + (k/8)*128 + (r%8)*16 + (k%8)*2.
__device__ __forceinline__ uint32_t kmajor128_off(int r, int k8) { return (r >> 3) * 2048 + k8 * 128 + (r & 7) * 16; }
// MN-major no-swizzle tile, T tokens along K, 128 channels along N: element (t, n)
// at (n/8)*(T*16) + (t/8)*128 + (t%8)*16 + (n%8)*2.
__device__ __forceinline__ uint32_t mnmajor_off(int t, int n8) { return n8 * (T * 16) + (t >> 3) * 128 + (t & 7) * 16; }

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

template <int P>
__global__ void __launch_bounds__(128, 2) decode_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem + kOffRaw;
  uint8_t* k16 = smem + kOffK16;
  uint8_t* v16 = smem + kOffV16;
  uint8_t* q16 = smem + kOffQ16;
  uint8_t* p16 = smem + kOffP16;
  float* ksc = reinterpret_cast<float*>(smem + kOffKsc);
  float* vsc = reinterpret_cast<float*>(smem + kOffVsc);
  float* kbias = reinterpret_cast<float*>(smem + kOffKbias);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* s_bar = full + NST;
  uint64_t* pv_bar = full + NST + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  uint32_t* page_ok = tmem_slot + 1;  // [NST] bit per page slot of the stage
  int32_t* timeout = reinterpret_cast<int32_t*>(tmem_slot + 1 + NST);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y, split = blockIdx.x;
  const int Hq = p.num_heads;
  const int max_tokens = p.max_pages * P;
  const SeqSplits sp = seq_splits(p.ctx_len[b], p.window, max_tokens, p.plan.chunk);

  if (!sp.valid || sp.nsplit == 0) {
    // Nothing to attend (or an invalid length): out = 0, lse = -inf, written by split 0.
    if (split == 0) {
      if (!sp.valid && tid == 0) set_err(p.err, CAI_DEVERR_LENGTH);
      for (int e = tid; e < Hq * kHeadDim; e += blockDim.x) p.out[(int64_t)b * Hq * kHeadDim + e] = 0.0f;
      if (p.lse_out)
        for (int h = tid; h < Hq; h += blockDim.x) p.lse_out[(int64_t)b * Hq + h] = -INFINITY;
    }
    return;
  }
  if (split >= sp.nsplit) return;
  const int chunk_idx = sp.first_chunk + split;
  const int start = max(sp.lo, chunk_idx * p.plan.chunk);
  const int end = min(sp.hi, (chunk_idx + 1) * p.plan.chunk);
  const int tile0 = start / T;
  const int ntiles = (end - 1) / T - tile0 + 1;
  const bool direct = sp.nsplit == 1;
  const int32_t* table = p.table + (int64_t)b * p.max_pages;

  // ---- set-up: barriers, tensor memory, Q (bf16 -> fp16, padded rows = 0)
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1);
    mbar_init(s_bar, 1);
    mbar_init(pv_bar, 1);
    *timeout = 0;
    fence_barrier_init();
  }
  {
    const uint16_t* qb = p.q + (int64_t)b * Hq * kHeadDim;
    for (int u = tid; u < kDecodeRows * 16; u += blockDim.x) {  // (row, 8-channel group)
      const int r = u >> 4, k8 = u & 15;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (r < Hq) {
        const uint4 src = *reinterpret_cast<const uint4*>(qb + r * kHeadDim + k8 * 8);
        const uint32_t s4[4] = {src.x, src.y, src.z, src.w};
        uint32_t d4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(s4[e] << 16), hi = __uint_as_float(s4[e] & 0xFFFF0000u);
          d4[e] = pack_f16x2(lo, hi);
        }
        w = make_uint4(d4[0], d4[1], d4[2], d4[3]);
      }
      *reinterpret_cast<uint4*>(q16 + kmajor128_off(r, k8)) = w;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Issue the bulk copies of tile i into its stage (thread 0 only).
  auto issue_tile = [&](int i) {
    const int stage = i % NST;
    const int tb = (tile0 + i) * T;
    uint32_t bytes = 0, ok = 0;
#pragma unroll
    for (int ps = 0; ps < T / P; ++ps) {
      const int t0 = tb + ps * P;
      if (t0 + P <= start || t0 >= end) continue;  // page wholly outside the split
      const int32_t pid = table[t0 / P];
      if (pid < 0 || pid >= p.num_pages) {
        set_err(p.err, CAI_DEVERR_PAGE);
        continue;
      }
      ok |= 1u << ps;
      bytes += page_bytes(P);
    }
    page_ok[stage] = ok;
    mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
    for (int ps = 0; ps < T / P; ++ps) {
      if (!(ok & (1u << ps))) continue;
      const int32_t pid = table[(tb + ps * P) / P];
      bulk_g2s(raw + stage * kRawStageBytes + ps * page_bytes(P), p.pages + (int64_t)pid * page_bytes(P),
               page_bytes(P), &full[stage]);
    }
  };

  if (tid == 0)
    for (int i = 0; i < NST && i < ntiles; ++i) issue_tile(i);

  // Softmax state: this thread owns head row h, token half th of each tile.
  const int h = warp * 16 + (lane & 15);
  const int th = lane >> 4;
  float m_ref = -INFINITY, l_sum = 0.0f;
  const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
  bool ok_all = true;

  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % NST;
    const uint8_t* rs = raw + stage * kRawStageBytes;
    if (!mbar_wait(&full[stage], (i / NST) & 1)) ok_all = false;
    if (i > 0 && !mbar_wait(pv_bar, (i - 1) & 1)) ok_all = false;

    // ---- int8 -> fp16 conversion of K and V (rotated lane mapping: conflict-free)
#pragma unroll
    for (int it = 0; it < (T * 8) / 128; ++it) {
      const int unit = it * 16 + (tid >> 3);  // 0 .. T-1 groups of 8 units
      const int t = (unit >> 3) * 8 + (tid & 7);
      const int c = ((unit & 7) + (tid & 7)) & 7;  // 16-byte chunk of the 128-byte row
      const int ps = t / P, slot = t % P;
      const uint8_t* pg = rs + ps * page_bytes(P);
      const uint4 kw = *reinterpret_cast<const uint4*>(pg + slot * kHeadDim + c * 16);
      const uint4 vw = *reinterpret_cast<const uint4*>(pg + P * kHeadDim + slot * kHeadDim + c * 16);
      uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
      i8x4_to_f16x4(kw.x, a0, a1);
      i8x4_to_f16x4(kw.y, a2, a3);
      i8x4_to_f16x4(kw.z, a4, a5);
      i8x4_to_f16x4(kw.w, a6, a7);
      *reinterpret_cast<uint4*>(k16 + kmajor128_off(t, 2 * c)) = make_uint4(a0, a1, a2, a3);
      *reinterpret_cast<uint4*>(k16 + kmajor128_off(t, 2 * c + 1)) = make_uint4(a4, a5, a6, a7);
      i8x4_to_f16x4(vw.x, a0, a1);
      i8x4_to_f16x4(vw.y, a2, a3);
      i8x4_to_f16x4(vw.z, a4, a5);
      i8x4_to_f16x4(vw.w, a6, a7);
      *reinterpret_cast<uint4*>(v16 + mnmajor_off(t, 2 * c)) = make_uint4(a0, a1, a2, a3);
      *reinterpret_cast<uint4*>(v16 + mnmajor_off(t, 2 * c + 1)) = make_uint4(a4, a5, a6, a7);
    }
    if (tid < T) {
      const int t = tid;
      const int ps = t / P, slot = t % P;
      const int abs_t = (tile0 + i) * T + t;
      const bool valid = abs_t >= start && abs_t < end && ((page_ok[stage] >> ps) & 1u);
      const float* sc = reinterpret_cast<const float*>(rs + ps * page_bytes(P) + 2 * P * kHeadDim);
      ksc[t] = valid ? sc[slot] * p.scale_log2 : 0.0f;
      kbias[t] = valid ? 0.0f : -INFINITY;
      vsc[t] = valid ? sc[P + slot] : 0.0f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
      if (i + NST < ntiles) issue_tile(i + NST);
      constexpr uint32_t idesc = idesc_f16_f32(64, T, 0, 0);
      const uint32_t qa = smem_addr(q16), ka = smem_addr(k16);
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks)
        mma_f16_ss(tmem + kColS, smem_desc(qa + ks * 256, 128, 2048), smem_desc(ka + ks * 256, 128, 2048), idesc,
                   ks > 0);
      mma_commit(s_bar);
    }
    if (!mbar_wait(s_bar, i & 1)) ok_all = false;
    tc_fence_after();

    // ---- softmax on this thread's 32 logits
    uint32_t sr[32];
    tmem_ld_16x32bx2_x32<32>(tmem + t_lane + kColS, sr);
    tmem_wait_ld();
    float z[32];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int t = th * 32 + j;
      z[j] = fmaf(__uint_as_float(sr[j]), ksc[t], kbias[t]);
      mx = fmaxf(mx, z[j]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const bool raise = mx > m_ref + kRescaleThreshold;
    const float alpha = raise ? ex2_approx(m_ref - mx) : 1.0f;  // m_ref = -inf -> 0
    if (i > 0 && __any_sync(0xffffffffu, raise)) {
      // Rescale this warp's rows of O (columns th*64 .. th*64+63).
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        const uint32_t ta = tmem + t_lane + kColO + half * 32;
        tmem_ld_16x32bx2_x32<64>(ta, o);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
        tmem_st_16x32bx2_x32<64>(ta, o);
      }
      tmem_wait_st();
    }
    if (raise) {
      l_sum *= alpha;
      m_ref = mx;
    }
    const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
    uint32_t pw[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const int t = th * 32 + j;
      const float p0 = ex2_approx(z[j] - m_use), p1 = ex2_approx(z[j + 1] - m_use);
      l_sum += p0 + p1;
      pw[j / 2] = pack_f16x2(p0 * vsc[t], p1 * vsc[t + 1]);
    }
    // P (fp16) as the K-major A operand: row h, tokens th*32 .. th*32+31.
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(p16 + (h >> 3) * (T * 16) + (th * 4 + c) * 128 + (h & 7) * 16) =
          make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(64, kHeadDim, 0, 1);
      const uint32_t pa = smem_addr(p16), va = smem_addr(v16);
#pragma unroll
      for (int ks = 0; ks < T / 16; ++ks)
        mma_f16_ss(tmem + kColO, smem_desc(pa + ks * 256, 128, T * 16), smem_desc(va + ks * 256, 128, T * 16), idesc,
                   (i > 0 || ks > 0) ? 1u : 0u);
      mma_commit(pv_bar);
    }
  }
  if (!mbar_wait(pv_bar, (ntiles - 1) & 1)) ok_all = false;
  tc_fence_after();
  if (!ok_all) atomicOr(timeout, 1);

  // ---- epilogue: normalise this thread's half row of O and write it.
  const float l_row = l_sum + __shfl_xor_sync(0xffffffffu, l_sum, 16);
  const float inv = l_row > 0.0f ? 1.0f / l_row : 0.0f;
  const float lse2 = l_row > 0.0f ? m_ref + __log2f(l_row) : -INFINITY;
  float* dst;
  if (direct) {
    dst = p.out + ((int64_t)b * Hq + h) * kHeadDim + th * 64;
  } else {
    dst = p.ws_o + (((int64_t)b * p.plan.max_splits + split) * Hq + h) * kHeadDim + th * 64;
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t o[32];
    tmem_ld_16x32bx2_x32<64>(tmem + t_lane + kColO + half * 32, o);
    tmem_wait_ld();
    if (h < Hq) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(dst + half * 32 + j) =
            make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv, __uint_as_float(o[j + 2]) * inv,
                        __uint_as_float(o[j + 3]) * inv);
    }
  }
  if (h < Hq && th == 0) {
    if (direct) {
      if (p.lse_out) p.lse_out[(int64_t)b * Hq + h] = lse2 * kLn2;
    } else {
      p.ws_lse[((int64_t)b * p.plan.max_splits + split) * Hq + h] = lse2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *timeout) set_err(p.err, CAI_DEVERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// One warp per (sequence, head): merge the partial outputs of the splits by
// their log-sum-exp: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M).
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p, int page_size) {
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int Hq = p.num_heads;
  if (gw >= p.batch * Hq) return;
  const int b = gw / Hq, h = gw - b * Hq;
  const SeqSplits sp = seq_splits(p.ctx_len[b], p.window, p.max_pages * page_size, p.plan.chunk);
  if (!sp.valid || sp.nsplit <= 1) return;  // written by the decode kernel itself
  const int S = p.plan.max_splits;
  const float* lse = p.ws_lse + (int64_t)b * S * Hq + h;
  float M = -INFINITY;
  for (int j = 0; j < sp.nsplit; ++j) M = fmaxf(M, lse[(int64_t)j * Hq]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.0f;
  if (M != -INFINITY) {
    for (int j = 0; j < sp.nsplit; ++j) {
      const float w = ex2_approx(lse[(int64_t)j * Hq] - M);
      const float4 o = reinterpret_cast<const float4*>(p.ws_o + (((int64_t)b * S + j) * Hq + h) * kHeadDim)[lane];
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
      wsum += w;
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  reinterpret_cast<float4*>(p.out + ((int64_t)b * Hq + h) * kHeadDim)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (p.lse_out && lane == 0) p.lse_out[(int64_t)b * Hq + h] = wsum > 0.0f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
}

template <int P>
cudaError_t launch_decode_p(const DecodeParams& p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(p.plan.max_splits, p.batch);
  decode_kernel<P><<<grid, 128, kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.plan.max_splits <= 1) return e;
  const int64_t warps = (int64_t)p.batch * p.num_heads;
  combine_kernel<<<(unsigned)((warps + 3) / 4), 128, 0, stream>>>(p, P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int page_size, cudaStream_t stream) {
  switch (page_size) {
    case 16: return launch_decode_p<16>(p, stream);
    case 32: return launch_decode_p<32>(p, stream);
    case 64: return launch_decode_p<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cai
