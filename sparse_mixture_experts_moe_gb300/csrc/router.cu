// Router: logits = x W_r (+ b_r), softmax over the E experts, deterministic top-k.
// csdn/6a919c0d §2.2 steps 1-4; aicoding/6a320eef §3.2; csdn/6a919c0d §4.2 (max subtraction).
//
// CUDA-core version, for fp32 layers and for E > 256 or E not a multiple of 8; bf16
// layers with E <= 256 use the tensor-core router in router_tc.cu.
// One CTA = 4 warps and 4*TPW tokens. W_r is staged through shared memory in
// 32-row slabs (as fp32) and shared by every token of the CTA; lane l owns four
// consecutive experts of the current 128-expert chunk and TPW tokens, so each
// 16-byte W load feeds 4*TPW FMAs. Logits land in shared memory; then the warp
// that owns a token does its softmax and k rounds of (max logit, lowest index)
// selection with warp shuffles. All sums use a fixed order: results are
// reproducible run to run.
#include "common.cuh"
#include "kernels.cuh"
#include "router_stats.cuh"

namespace moe {
namespace {

constexpr int kWarps = 4;
constexpr int kDK = 32;      // W_r rows per staged slab
constexpr int kEC = 128;     // experts per chunk (4 per lane)

template <typename T, int TPW>
__global__ void __launch_bounds__(kWarps * 32)
router_topk_kernel(const T* __restrict__ x, const T* __restrict__ w_r, const float* __restrict__ b_r, int Tn,
                   int d, int E, int k, int renorm, RouterStats st, int32_t* __restrict__ topk_idx,
                   float* __restrict__ topk_gate) {
  constexpr int TB = kWarps * TPW;
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ __align__(16) float smem[];
  float* sW = smem;                    // [kDK][kEC]
  float* sX = sW + kDK * kEC;          // [TB][kDK]
  float* sL = sX + TB * kDK;           // [TB][E]
  float* sSoft = sL + TB * E;          // statistics only: [kWarps][E] soft-load sums, per warp
  float* sEnt = sSoft + kWarps * E;    // [kWarps] entropy sums
  int* sCnt = reinterpret_cast<int*>(sEnt + kWarps);  // [E] assignment counts
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tok0 = blockIdx.x * TB;
  const bool stats = st.part != nullptr;
  if (stats)
    for (int i = tid; i < kWarps * E + kWarps + E; i += kWarps * 32) sSoft[i] = 0.f;  // zero bits: also int 0

  for (int ec = 0; ec < E; ec += kEC) {
    float acc[TPW][4];
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
      for (int m = 0; m < 4; ++m) acc[t][m] = 0.f;

    for (int k0 = 0; k0 < d; k0 += kDK) {
      __syncthreads();
      for (int i = tid; i < kDK * kEC; i += kWarps * 32) {
        const int r = i / kEC, c = i % kEC;
        const int gk = k0 + r, ge = ec + c;
        sW[i] = (gk < d && ge < E) ? to_f32(w_r[(size_t)gk * E + ge]) : 0.f;
      }
      for (int i = tid; i < TB * kDK; i += kWarps * 32) {
        const int t = i / kDK, c = i % kDK;
        const int gt = tok0 + t, gk = k0 + c;
        sX[i] = (gt < Tn && gk < d) ? to_f32(x[(size_t)gt * d + gk]) : 0.f;
      }
      __syncthreads();
#pragma unroll 2
      for (int kk = 0; kk < kDK; kk += 4) {
        float4 w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = *reinterpret_cast<const float4*>(&sW[(kk + q) * kEC + 4 * lane]);
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
          const float4 xv = *reinterpret_cast<const float4*>(&sX[(warp * TPW + t) * kDK + kk]);
          acc[t][0] = fmaf(xv.x, w[0].x, acc[t][0]); acc[t][1] = fmaf(xv.x, w[0].y, acc[t][1]);
          acc[t][2] = fmaf(xv.x, w[0].z, acc[t][2]); acc[t][3] = fmaf(xv.x, w[0].w, acc[t][3]);
          acc[t][0] = fmaf(xv.y, w[1].x, acc[t][0]); acc[t][1] = fmaf(xv.y, w[1].y, acc[t][1]);
          acc[t][2] = fmaf(xv.y, w[1].z, acc[t][2]); acc[t][3] = fmaf(xv.y, w[1].w, acc[t][3]);
          acc[t][0] = fmaf(xv.z, w[2].x, acc[t][0]); acc[t][1] = fmaf(xv.z, w[2].y, acc[t][1]);
          acc[t][2] = fmaf(xv.z, w[2].z, acc[t][2]); acc[t][3] = fmaf(xv.z, w[2].w, acc[t][3]);
          acc[t][0] = fmaf(xv.w, w[3].x, acc[t][0]); acc[t][1] = fmaf(xv.w, w[3].y, acc[t][1]);
          acc[t][2] = fmaf(xv.w, w[3].z, acc[t][2]); acc[t][3] = fmaf(xv.w, w[3].w, acc[t][3]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = ec + 4 * lane + m;
        if (e < E) sL[(warp * TPW + t) * E + e] = acc[t][m];
      }
  }
  __syncwarp();

  // Softmax and top-k: each warp finishes its own tokens (it wrote all their logits).
  float went = 0.f;
  for (int t = 0; t < TPW; ++t) {
    const int tok = tok0 + warp * TPW + t;
    if (tok >= Tn) break;
    float* row = sL + (warp * TPW + t) * E;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) {
      const float v = row[e] + (b_r != nullptr ? b_r[e] : 0.f);
      row[e] = v;
      m = fmaxf(m, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += expf(row[e] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (stats) {
      // p = exp(z) / s with z = l - max; entropy = ln s - sum p z. Lane l owns columns l mod 32.
      float hs = 0.f;
      for (int e = lane; e < E; e += 32) {
        const float z = row[e] - m;
        const float p = expf(z) / s;
        sSoft[warp * E + e] += p;
        hs += p * z;
      }
      went += logf(s) - warp_sum_xor(hs);
    }
    __syncwarp();
    float sel[8];
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
      for (int e = lane; e < E; e += 32) {
        const float v = row[e];
        if (v > bv) { bv = v; be = e; }  // ascending e within a lane: ties keep the lower index
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      sel[j] = bv;
      if (lane == 0) {
        topk_idx[(size_t)tok * k + j] = be;
        if (stats) atomicAdd(&sCnt[be], 1);
      }
      if ((be & 31) == lane) row[be] = -INFINITY;
      __syncwarp();
    }
    // gates: softmax probabilities, or (renorm) the softmax over the k chosen logits
    float ks = 0.f;
    if (renorm)
      for (int j = 0; j < k; ++j) ks += expf(sel[j] - m);
    if (lane == 0)
      for (int j = 0; j < k; ++j) topk_gate[(size_t)tok * k + j] = expf(sel[j] - m) / (renorm ? ks : s);
  }
  if (stats) {
    if (lane == 0) sEnt[warp] = went;
    router_stats_cta(st, sSoft, kWarps, E, sEnt, sCnt, E, Tn, k);
  }
}

template <typename T, int TPW>
cudaError_t launch_router_t(const void* x, const void* w_r, const float* b_r, int Tn, int d, int E, int k,
                            int renorm, const RouterStats& st, int32_t* idx, float* gate, cudaStream_t s) {
  constexpr int TB = kWarps * TPW;
  static_assert(TB >= kRouterStatsTokensPerCta, "statistics rows are sized for 8 tokens per CTA");
  const size_t stat_words = st.part != nullptr ? (size_t)(kWarps * E + kWarps + E) : 0;
  const size_t smem = (size_t)(kDK * kEC + TB * kDK + TB * E + stat_words) * sizeof(float);
  auto kern = router_topk_kernel<T, TPW>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = (Tn + TB - 1) / TB;
  return launch_pdl(kern, dim3(grid), dim3(kWarps * 32), smem, s, (const T*)x, (const T*)w_r, b_r, Tn, d, E, k,
                    renorm, st, idx, gate);
}

}  // namespace

cudaError_t launch_router_topk(const void* x, const void* w_r, const float* b_r, int Tn, int d, int E, int k,
                               int dt, int flags, const RouterStats& st, int32_t* idx, float* gate, int* status,
                               uint64_t timeout_ns, cudaStream_t s, bool* wrote_hist) {
  const int renorm = (flags & MOE_GATES_RENORMALISE) != 0;
  if (wrote_hist != nullptr) *wrote_hist = false;
  if (Tn == 0) return cudaSuccess;
  // bf16 with E <= 256 (E % 8 == 0 for TMA row strides): tensor cores; otherwise this CUDA-core kernel.
  if (dt == MOE_DTYPE_BF16 && E <= 256 && E % 8 == 0) {
    const cudaError_t e = launch_router_tc(x, w_r, b_r, Tn, d, E, k, renorm, st, idx, gate, status, timeout_ns, s);
    if (e != cudaErrorNotSupported) {
      if (wrote_hist != nullptr) *wrote_hist = e == cudaSuccess && st.hist != nullptr;
      return e;
    }
  }
  // the CUDA-core router fills no histogram
  const RouterStats st_nohist{st.part, st.out, st.ticket, nullptr};
  const bool small_e = E <= 256;
  if (dt == MOE_DTYPE_BF16)
    return small_e ? launch_router_t<__nv_bfloat16, 8>(x, w_r, b_r, Tn, d, E, k, renorm, st_nohist, idx, gate, s)
                   : launch_router_t<__nv_bfloat16, 2>(x, w_r, b_r, Tn, d, E, k, renorm, st_nohist, idx, gate, s);
  return small_e ? launch_router_t<float, 8>(x, w_r, b_r, Tn, d, E, k, renorm, st_nohist, idx, gate, s)
                 : launch_router_t<float, 2>(x, w_r, b_r, Tn, d, E, k, renorm, st_nohist, idx, gate, s);
}

}  // namespace moe
