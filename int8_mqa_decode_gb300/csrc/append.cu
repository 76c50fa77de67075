// Fused quantize-and-append (int8 KV cache, "Character.AI: inference
// optimization", 05; K and V computed once per new token and stored, Red Hat
// page "Por que o cache KV existe").
//
// One warp per (sequence, new token, K|V): 32 lanes x float4 = one 128-wide
// row read with 512-byte coalesced loads; warp-shuffle absmax; IEEE fp32
// division for the scale and for every quotient, round-half-even, clamp to
// [-127, 127]; the codes go to the token's K row (one 32-bit store per lane)
// or to its column of the channel-major V block (four byte stores per lane),
// and one fp32 scale.
// Bit-exact by construction: no fused multiply-add touches the quotient path
// and the build uses neither fast-math nor flush-to-zero.
#include "common.cuh"
#include "ptx.cuh"

namespace cai {
namespace {

// Up to kMaxKvHeads pools in one launch: blockIdx.y selects the pool.
struct AppendArgs {
  AppendParams pool[kMaxKvHeads];
};

__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendArgs args) {
  grid_dependency_wait();
  grid_launch_dependents();
  const AppendParams& p = args.pool[blockIdx.y];
  const int warp_global = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int rows = p.batch * p.n_new;
  if (warp_global >= 2 * rows) return;
  const int is_v = warp_global >= rows;
  const int row = is_v ? warp_global - rows : warp_global;
  const int b = row / p.n_new;
  const int i = row - b * p.n_new;

  const float* src = (is_v ? p.v_new : p.k_new) + (int64_t)row * kHeadDim;
  const float4 x = reinterpret_cast<const float4*>(src)[lane];

  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

  const int32_t pos = p.start_pos[b] + i;
  const int32_t P = p.page_size;
  if (pos < 0 || pos >= p.max_pages * P) {
    if (lane == 0 && p.err) atomicOr(p.err, CAI_DEVERR_LENGTH);
    return;
  }
  const int32_t page = p.table[(int64_t)b * p.max_pages + pos / P];
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0 && p.err) atomicOr(p.err, CAI_DEVERR_PAGE);
    return;
  }
  const int32_t slot = pos - (pos / P) * P;

  // A zero scale (an all-zero vector, or amax / 127 underflowing to 0) gives zero codes.
  const float s = __fdiv_rn(amax, 127.0f);
  uint32_t packed = 0;
  if (s != 0.0f) {
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int c = __float2int_rn(__fdiv_rn(xs[e], s));
      c = c > 127 ? 127 : (c < -127 ? -127 : c);
      packed |= (uint32_t)(c & 0xFF) << (8 * e);
    }
  }
  uint8_t* pg = p.pages + (int64_t)page * page_bytes(P);
  if (!is_v) {
    // K codes are token-major: one 128-byte row per slot.
    reinterpret_cast<uint32_t*>(pg + slot * kHeadDim)[lane] = packed;
  } else {
    // V codes are channel-major: channel c's P codes are contiguous, so this token's
    // code of channel c is byte c * P + slot of the V block.
    uint8_t* v = pg + P * kHeadDim + slot;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[(lane * 4 + e) * P] = (uint8_t)(packed >> (8 * e));
  }
  if (lane == 0) {
    float* scales = reinterpret_cast<float*>(pg + 2 * P * kHeadDim) + (is_v ? P : 0);
    scales[slot] = s;
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams* ps, int n, cudaStream_t stream) {
  if (n < 1 || n > kMaxKvHeads) return cudaErrorInvalidValue;
  AppendArgs a;
  for (int i = 0; i < kMaxKvHeads; ++i) a.pool[i] = ps[i < n ? i : n - 1];
  const int64_t warps = 2ll * ps[0].batch * ps[0].n_new;  // the same rows in every pool
  const int64_t blocks = (warps + 7) / 8;
  return launch_pdl(append_kernel, dim3((unsigned)blocks, (unsigned)n), dim3(256), 0, stream, a);
}

}  // namespace cai
