// Device side of the seeded input generator (see synth_inputs/__init__.py for
// the definition).  Integer-only up to one correctly rounded fp32 multiply, so
// it reproduces the host generator bit for bit.  It fills buffers; it knows
// nothing about the step.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint64_t key, uint64_t idx, uint64_t j) {
  return mix64(key + kGamma * (idx * 3ull + j + 1ull));
}

__device__ __forceinline__ float normal_at(uint64_t key, uint64_t idx, float sigma) {
  int64_t s = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t w = word(key, idx, j);
    s += int64_t(w & 0xFFFF) + int64_t((w >> 16) & 0xFFFF) + int64_t((w >> 32) & 0xFFFF) + int64_t(w >> 48);
  }
  const int64_t n = 2 * s - 12 * 65535;
  const float unit = __fmul_rn(float(n), 0x1p-17f);  // exact
  return __fmul_rn(unit, sigma);
}

__global__ void fill_normal_f32(float* dst, int64_t n, uint64_t key, int64_t start, float sigma) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    dst[i] = normal_at(key, uint64_t(start + i), sigma);
}

__global__ void fill_normal_bf16trunc(uint16_t* dst, int64_t n, uint64_t key, int64_t start, float sigma) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    dst[i] = uint16_t(__float_as_uint(normal_at(key, uint64_t(start + i), sigma)) >> 16);
}

__global__ void fill_uniform_f32(float* dst, int64_t n, uint64_t key, int64_t start, float hi) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const uint64_t w = word(key, uint64_t(start + i), 0);
    const float u = __fmul_rn(float(uint32_t(w >> 40)), 0x1p-24f);  // exact
    dst[i] = __fmul_rn(u, hi);
  }
}

int grid_for(int64_t n) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + 255) / 256;
  const int64_t cap = int64_t(sms) * 8;
  return int(want < cap ? (want > 0 ? want : 1) : cap);
}

int finish() { return cudaGetLastError() == cudaSuccess ? 0 : 1; }

}  // namespace

// Each returns 0 on success, 1 on a CUDA error; n == 0 launches nothing.
// dst: device buffer of n elements; element i gets the value of logical index
// start + i of the stream `key`.
extern "C" int synth_fill_normal_f32(float* dst, int64_t n, uint64_t key, int64_t start, float sigma, void* stream) {
  if (n <= 0) return 0;
  fill_normal_f32<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, n, key, start, sigma);
  return finish();
}

extern "C" int synth_fill_normal_bf16trunc(uint16_t* dst, int64_t n, uint64_t key, int64_t start, float sigma,
                                           void* stream) {
  if (n <= 0) return 0;
  fill_normal_bf16trunc<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, n, key, start, sigma);
  return finish();
}

extern "C" int synth_fill_uniform_f32(float* dst, int64_t n, uint64_t key, int64_t start, float hi, void* stream) {
  if (n <= 0) return 0;
  fill_uniform_f32<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, n, key, start, hi);
  return finish();
}
