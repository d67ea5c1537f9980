// Routing statistics computed inside the router kernels, beside the top-k selection
// (csdn/6a462027 §4.2 expert load; aicoding/6a320eef §3.2 balance term, §5.2 router entropy):
//   out[e]        = (1/T) sum_t p[t, e]                    soft load of expert e
//   out[E + e]    = #{(t, j) : idx[t, j] = e} / (T k)      share of the assignments
//   out[2E]       = sum_e (out[E + e] - 1/E)^2             balance term (times lambda = the loss)
//   out[2E + 1]   = (1/T) sum_t -sum_e p ln p              mean router entropy, nats
// p is the full softmax over the E experts. Each CTA of a router launch writes one row of
// partial sums; the CTA that takes the last ticket reduces the rows in CTA order, in double.
// Every order is fixed, so the statistics are reproducible run to run.
#pragma once

#include "kernels.cuh"

namespace moe {

// v[i] of lane l is element (l, i) of a 32 x 32 block. On return, lane l holds the sum over
// the 32 lanes of column l (recursive halving: each step exchanges half of the live columns
// with the xor partner and keeps the half that the lane's bit selects).
__device__ __forceinline__ float warp_column_sums(float (&v)[32]) {
  const unsigned lane = threadIdx.x & 31u;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & (unsigned)o) != 0u;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Called by every thread of the CTA. s_soft: nw rows (stride ld) of per-warp soft-load sums,
// s_ent: nw per-warp entropy sums, s_cnt: E assignment counts of this CTA's tokens.
// blockDim.x <= 256.
__device__ inline void router_stats_cta(const RouterStats& st, const float* s_soft, int nw, int ld,
                                        const float* s_ent, const int* s_cnt, int E, int Tn, int k) {
  __shared__ int s_last;
  __shared__ double s_red[2][256];
  __syncthreads();
  const size_t W = 2 * (size_t)E + 1;
  float* row = st.part + (size_t)blockIdx.x * W;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < nw; ++w) v += s_soft[w * ld + e];
    row[e] = v;
    reinterpret_cast<int*>(row)[E + e] = s_cnt[e];
  }
  if (threadIdx.x == 0) {
    float h = 0.f;
    for (int w = 0; w < nw; ++w) h += s_ent[w];
    row[2 * E] = h;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(st.ticket, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int ncta = (int)gridDim.x;
  double bal = 0.0, ent = 0.0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    double s = 0.0;
    long long c = 0;
    for (int j = 0; j < ncta; ++j) {
      s += (double)__ldcg(st.part + (size_t)j * W + e);
      c += __ldcg(reinterpret_cast<const int*>(st.part) + (size_t)j * W + E + e);
    }
    const double f = (double)c / ((double)Tn * (double)k);
    st.out[e] = (float)(s / (double)Tn);
    st.out[E + e] = (float)f;
    bal += (f - 1.0 / E) * (f - 1.0 / E);
  }
  for (int j = threadIdx.x; j < ncta; j += blockDim.x) ent += (double)__ldcg(st.part + (size_t)j * W + 2 * E);
  s_red[0][threadIdx.x] = bal;
  s_red[1][threadIdx.x] = ent;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0, h = 0.0;
    for (int i = 0; i < (int)blockDim.x; ++i) { b += s_red[0][i]; h += s_red[1][i]; }
    st.out[2 * E] = (float)b;
    st.out[2 * E + 1] = (float)(h / (double)Tn);
    *st.ticket = 0;  // ready for the next launch
  }
}

}  // namespace moe
