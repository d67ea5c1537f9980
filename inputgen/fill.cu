// Device side of the seeded input generator (see inputgen/__init__.py for the
// definition). Produces, for flat indices start .. start+n-1, exactly the values
// the numpy implementation produces: SplitMix64 bits, an Irwin-Hall sum of twelve
// 16-bit uniforms (exact in fp32), one fp32 multiply by sigma, then an optional
// round-to-nearest-even to bf16. Holds no arithmetic of the MoE layer.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kM1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kM2 = 0x94D049BB133111EBull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * kM1;
  z = (z ^ (z >> 27)) * kM2;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float draw_one(uint64_t key, uint64_t i, float sigma) {
  int acc = 0;
#pragma unroll
  for (int m = 0; m < 3; ++m) {
    uint64_t h = mix64(key + (3ull * i + (uint64_t)(m + 1)) * kGamma);
    acc += (int)(h & 0xFFFFull) + (int)((h >> 16) & 0xFFFFull) +
           (int)((h >> 32) & 0xFFFFull) + (int)((h >> 48) & 0xFFFFull);
  }
  float z = (float)(acc + 6 - 393216) * (1.0f / 65536.0f);  // exact
  return __fmul_rn(z, sigma);
}

__global__ void fill_f32(float* __restrict__ out, long long n, long long start, uint64_t key,
                         float sigma) {
  long long stride = (long long)gridDim.x * blockDim.x;
  for (long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = draw_one(key, (uint64_t)(start + j), sigma);
}

__global__ void fill_bf16(__nv_bfloat16* __restrict__ out, long long n, long long start,
                          uint64_t key, float sigma) {
  long long stride = (long long)gridDim.x * blockDim.x;
  for (long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = __float2bfloat16_rn(draw_one(key, (uint64_t)(start + j), sigma));
}

}  // namespace

extern "C" int inputgen_fill_normal(void* out, long long n, long long start,
                                    unsigned long long key, float sigma, int dtype,
                                    cudaStream_t stream) {
  if (n <= 0) return 0;
  if (out == nullptr || start < 0 || (dtype != 0 && dtype != 1)) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n + 255) / 256;
  long long cap = (long long)(sms > 0 ? sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  if (dtype == 0)
    fill_f32<<<(unsigned)blocks, 256, 0, stream>>>((float*)out, n, start, key, sigma);
  else
    fill_bf16<<<(unsigned)blocks, 256, 0, stream>>>((__nv_bfloat16*)out, n, start, key, sigma);
  return (int)cudaGetLastError();
}
