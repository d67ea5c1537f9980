// CUDA-core grouped expert GEMM with the GeLU or gate epilogue (the fp32 path).
// csdn/6a462027 §3.2 (d -> d_ff -> d GELU experts) and §4.2 step 6 (grouped GEMM over experts).
//
// Work item = one 64-row tile of one expert's row range x one 64-column tile.
// 256 threads, 4x4 outputs each, K staged in 16-deep slabs through shared memory.
// fp32 accumulation in a fixed order (k ascending).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

// up (STAGE 1) writes h in the layer's element type; down (STAGE 2) writes fp32 y_perm.
template <typename T, int STAGE, typename OutT>
__global__ void __launch_bounds__(256)
ffn_simt_kernel(const T* __restrict__ a, const T* __restrict__ w, const int32_t* __restrict__ offsets,
                const float* __restrict__ row_gate, int K, int N, int E, OutT* __restrict__ out) {
  __shared__ float sA[BK][BM + 4];
  __shared__ float sB[BK][BN + 4];
  __shared__ int s_e, s_m0, s_mend;
  const int tid = threadIdx.x;
  griddep_launch_dependents();
  griddep_wait();
  if (tid == 0) {
    // Locate work item blockIdx.y in the list of (expert, 64-row tile) pairs.
    int item = blockIdx.y, e_found = -1, m0 = 0, mend = 0;
    for (int e = 0; e < E; ++e) {
      const int lo = offsets[e], hi = offsets[e + 1];
      const int nt = (hi - lo + BM - 1) / BM;
      if (item < nt) { e_found = e; m0 = lo + item * BM; mend = hi; break; }
      item -= nt;
    }
    s_e = e_found; s_m0 = m0; s_mend = mend;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int m0 = s_m0, mend = s_mend, n0 = blockIdx.x * BN;
  const T* we = w + (size_t)e * K * N;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BK * BM; i += 256) {
      const int r = i / BK, c = i % BK;
      const int gr = m0 + r, gk = k0 + c;
      sA[c][r] = (gr < mend && gk < K) ? to_f32(a[(size_t)gr * K + gk]) : 0.f;
    }
    for (int i = tid; i < BK * BN; i += 256) {
      const int r = i / BN, c = i % BN;
      const int gk = k0 + r, gn = n0 + c;
      sB[r][c] = (gk < K && gn < N) ? to_f32(we[(size_t)gk * N + gn]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = sA[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = sB[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gr = m0 + tr * 4 + i;
    if (gr >= mend) continue;
    const float g = STAGE == 2 ? row_gate[gr] : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tc * 4 + j;
      if (gn >= N) continue;
      const float v = STAGE == 1 ? gelu_erf(acc[i][j]) : g * acc[i][j];
      out[(size_t)gr * N + gn] = from_f32<OutT>(v);
    }
  }
}

template <typename T>
cudaError_t launch_t(const FfnArgs& p, cudaStream_t s) {
  const int max_items = (p.rows + BM - 1) / BM + p.E;  // each expert adds at most one partial tile
  dim3 grid((p.N + BN - 1) / BN, max_items);
  if (max_items > 65535) return cudaErrorInvalidConfiguration;
  if (p.stage == 1)
    return launch_pdl(ffn_simt_kernel<T, 1, T>, grid, dim3(256), 0, s, (const T*)p.a, (const T*)p.w, p.offsets,
                      p.row_gate, p.K, p.N, p.E, (T*)p.out);
  else
    return launch_pdl(ffn_simt_kernel<T, 2, float>, grid, dim3(256), 0, s, (const T*)p.a, (const T*)p.w, p.offsets,
                      p.row_gate, p.K, p.N, p.E, (float*)p.out);
}

}  // namespace

cudaError_t launch_ffn_simt(const FfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  return p.dt == MOE_DTYPE_BF16 ? launch_t<__nv_bfloat16>(p, s) : launch_t<float>(p, s);
}

}  // namespace moe
