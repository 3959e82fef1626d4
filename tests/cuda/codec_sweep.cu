// Test kernel: the CUDA path's fp32 -> E2M1 and fp32 -> E4M3 conversion
// helpers (csrc/codec.cuh, the hardware conversions the append kernels use)
// applied to a range of fp32 bit patterns, both lanes of each packed result:
// lane 0 takes x, lane 1 takes -x.  tests/test_gpu_codec_sweep.py compares the
// codes with the oracle's codecs on every fp32 bit pattern.
#include <stdint.h>

#include "../../fp4_kv_cache_rope_gb300/csrc/codec.cuh"

__global__ void codec_sweep_kernel(uint64_t first, int64_t n, uint8_t* e2m1, uint16_t* e4m3) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float x = __uint_as_float((uint32_t)(first + (uint64_t)i));
    e2m1[i] = (uint8_t)csa2::e2m1x2_from_f32(x, -x);
    e4m3[i] = (uint16_t)csa2::e4m3x2_from_f32(x, -x);
  }
}

extern "C" int codec_sweep(uint64_t first, int64_t n, uint8_t* e2m1, uint16_t* e4m3) {
  codec_sweep_kernel<<<4096, 256>>>(first, n, e2m1, e4m3);
  return (int)cudaGetLastError();
}
