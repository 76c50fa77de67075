// GPU twin of the seeded input generators in synth/__init__.py.
//
// Input generation only: splitmix64 (Steele, Lea and Flood, OOPSLA 2014) at
// counter ((stream << 40) | (b << 27) | (p << 7) | d) * 4 + r, summed as an
// Irwin-Hall(12) normal, optionally rounded to bf16.  Every step is integer
// or exact fp32, so these bits equal the numpy ones.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t n) {
  uint64_t z = seed + (n + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float irwin_hall12(uint64_t seed, uint64_t idx) {
  int64_t acc = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint64_t h = splitmix64(seed, idx * 4ull + r);
    acc += (int64_t)(h & 0xFFFFFull) + (int64_t)((h >> 20) & 0xFFFFFull) + (int64_t)((h >> 40) & 0xFFFFFull);
  }
  acc -= (int64_t)6 << 20;
  return (float)acc / 1048576.0f;  // exact: |acc| < 2^24 and the divisor is a power of two
}

__device__ __forceinline__ uint64_t index_of(uint32_t stream, uint32_t b, uint32_t p, uint32_t d) {
  return ((uint64_t)stream << 40) | ((uint64_t)b << 27) | ((uint64_t)p << 7) | (uint64_t)d;
}

// out[i][n][d] = normal(stream, b = b0 + i, p = pos[i] + n, d)
__global__ void normal_rows_kernel(float* out, uint64_t seed, uint32_t stream, int32_t b0,
                                   const int32_t* pos, int32_t p_const, int32_t batch, int32_t n,
                                   int32_t dim) {
  int64_t total = (int64_t)batch * n * dim;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    int32_t d = (int32_t)(e % dim);
    int64_t row = e / dim;
    int32_t j = (int32_t)(row % n);
    int32_t i = (int32_t)(row / n);
    int32_t p = (pos ? pos[i] : p_const) + j;
    out[e] = irwin_hall12(seed, index_of(stream, (uint32_t)(b0 + i), (uint32_t)p, (uint32_t)d));
  }
}

__global__ void q_rows_kernel(uint16_t* out, uint64_t seed, uint32_t stream, int32_t b0, int32_t batch,
                              int32_t rows, int32_t dim) {
  int64_t total = (int64_t)batch * rows * dim;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    int32_t d = (int32_t)(e % dim);
    int64_t row = e / dim;
    int32_t r = (int32_t)(row % rows);
    int32_t i = (int32_t)(row / rows);
    float x = irwin_hall12(seed, index_of(stream, (uint32_t)(b0 + i), (uint32_t)r, (uint32_t)d));
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    out[e] = *reinterpret_cast<uint16_t*>(&h);
  }
}

int grid_for(int64_t total) {
  int64_t g = (total + 255) / 256;
  if (g > 152 * 64) g = 152 * 64;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" {

// fp32 rows for sequences b0 .. b0+batch-1: out[i][j][d] at position (pos ? pos[i] : p_const) + j.
// pos is a device array or null.  Returns a cudaError_t value.
int synth_normal_rows(float* out, uint64_t seed, uint32_t stream, int32_t b0, const int32_t* pos,
                      int32_t p_const, int32_t batch, int32_t n, int32_t dim, void* cuda_stream) {
  int64_t total = (int64_t)batch * n * dim;
  if (total == 0) return 0;
  normal_rows_kernel<<<grid_for(total), 256, 0, (cudaStream_t)cuda_stream>>>(out, seed, stream, b0, pos, p_const,
                                                                             batch, n, dim);
  return (int)cudaGetLastError();
}

// bf16 bits out[i][r][d] for sequences b0 .. b0+batch-1, row coordinate r.
int synth_q_rows(uint16_t* out, uint64_t seed, uint32_t stream, int32_t b0, int32_t batch, int32_t rows,
                 int32_t dim, void* cuda_stream) {
  int64_t total = (int64_t)batch * rows * dim;
  if (total == 0) return 0;
  q_rows_kernel<<<grid_for(total), 256, 0, (cudaStream_t)cuda_stream>>>(out, seed, stream, b0, batch, rows, dim);
  return (int)cudaGetLastError();
}

}  // extern "C"
