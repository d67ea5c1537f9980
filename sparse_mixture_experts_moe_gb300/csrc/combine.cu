// Combine: out[t, :] = sum_{j=0..k-1} y_perm[row_of[t, j], :], fp32 in slot order, one rounding.
// csdn/6a462027 §4.2 step 7 (sum the expert outputs back per token). The gate was
// already applied per row by the down-projection epilogue.
//
// One warp per (token, 256-column chunk), so a single decode token still spreads over many
// warps; each lane owns 8 consecutive columns and reads the fp32 rows with 128-bit loads.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]); u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]); u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// y_perm is fp32 for every element type, so the output is rounded exactly once.
template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ y_perm, const int32_t* __restrict__ row_of, int Tn, int d, int k, int A,
               T* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int groups = d / 8;
  const int chunks = (groups + 31) / 32;  // a warp item: one token, 32 groups of 8 columns
  const long long items = (long long)Tn * chunks;
  for (long long item = gwarp; item < items; item += nwarps) {
    const int t = (int)(item / chunks);
    const int g = (int)(item % chunks) * 32 + lane;
    int rows[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rows[j] = j < k ? row_of[(size_t)t * k + j] : -1;
    if (g >= groups) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= k) break;
      const int r = rows[j];
      if (r < 0 || r >= A) continue;
      float v[8];
      load8(y_perm + (size_t)r * d + 8 * g, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    store8(out + (size_t)t * d + 8 * g, acc);
  }
}

}  // namespace

cudaError_t launch_combine(const void* y_perm, const int32_t* row_of, int Tn, int d, int k, int dt, void* out,
                           cudaStream_t s) {
  if (Tn == 0) return cudaSuccess;
  const long long items = (long long)Tn * ((d / 8 + 31) / 32);
  int blocks = (int)((items + 7) / 8 < 0x7fffffff ? (items + 7) / 8 : 0x7fffffff);
  const int cap = device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  const int A = Tn * k;
  if (dt == MOE_DTYPE_BF16)
    return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s, (const float*)y_perm, row_of, Tn,
                      d, k, A, (__nv_bfloat16*)out);
  return launch_pdl(combine_kernel<float>, dim3(blocks), dim3(256), 0, s, (const float*)y_perm, row_of, Tn, d, k, A,
                    (float*)out);
}

}  // namespace moe
