// Device twin of the seeded input generator in synth/__init__.py.
//
// value(i) = table[mix64(key + i) >> 48] * chan_mult[i % period]   (normal)
// value(i) = ((mix64(key + i) >> 40) & 0xFFFFFF) * 2^-24            (uniform)
// with mix64 the SplitMix64 finaliser.  Only integer operations, a table
// lookup and an exact power-of-two multiply are involved, so the host and the
// device produce identical bits.  Holds no arithmetic of the CSA2 method.
#include <cuda_runtime.h>
#include <stdint.h>

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_normal_kernel(float* out, int64_t n, uint64_t key, int64_t start,
                                   const float* table, const float* mult, int32_t period) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t g = start + i;
    float v = table[mix64(key + (uint64_t)g) >> 48];
    if (mult) v *= mult[g % period];
    out[i] = v;
  }
}

__global__ void fill_uniform_kernel(float* out, int64_t n, uint64_t key, int64_t start) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t h = mix64(key + (uint64_t)(start + i));
    out[i] = (float)((h >> 40) & 0xFFFFFFull) * 5.9604644775390625e-08f;
  }
}

extern "C" int synth_fill_normal(float* out, int64_t n, uint64_t key, int64_t start,
                                 const float* table, const float* mult, int32_t period,
                                 void* stream) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_normal_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, n, key, start, table,
                                                                        mult, period);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_uniform(float* out, int64_t n, uint64_t key, int64_t start,
                                  void* stream) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_uniform_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, n, key, start);
  return (int)cudaGetLastError();
}
