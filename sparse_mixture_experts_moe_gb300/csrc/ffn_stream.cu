// Weight-streaming grouped expert FFN for batches with few rows per expert (decode).
// csdn/6a919c0d §2.3: with top-2 routing each token reads two experts' full W1 and W2
// from HBM, so the layer is bound by moving weights, not by arithmetic.
//
// Work unit = (expert with at least one row, 64-column slab of its weight matrix).
// A CTA owns the slab for the full depth K, so the GeLU (up) or gate (down)
// epilogue applies locally and no partial sums leave the CTA. Each k-row of the
// slab is 128 contiguous bytes read by 8 lanes with 16-byte loads; two batches of 8
// loads per thread are in flight (software pipelining), two CTAs per SM. The expert's
// rows (2 or 4 per pass, by batch size; more rows take more passes) are staged in
// shared memory as fp32 in 1024-deep chunks.
// Partial sums are combined in a fixed order (xor-butterfly in the warp, then
// warps in index order), so results are reproducible.
// Units are ordered slab-fastest, so CTAs running together stream neighbouring
// slabs of the same matrix rows.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256, kWarps = 8;
constexpr int NS = 64;            // columns per slab
constexpr int LPR = NS / 8;       // lanes per k-row: 8 (16 bytes each)
constexpr int RPW = 32 / LPR;     // k-rows per warp per step: 4
constexpr int KSTEP = kWarps * RPW;  // k-rows per CTA step: 32
// k-depth of activations staged per chunk: 32 KB of fp32 rows. Each chunk restarts the weight
// stream behind two barriers, so chunks are made as deep as the two-CTAs-per-SM budget allows.
template <int RMAX>
constexpr int kc_for() { return RMAX <= 2 ? 4096 : 2048; }
// Weight loads per thread per batch (two batches in flight): 8 with 2 rows a pass; with 4 rows
// the accumulators take the registers, and 8 would spill.
template <int RMAX>
constexpr int unroll_for() { return RMAX == 1 ? 9 : RMAX <= 2 ? 8 : 7; }

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&v)[8]) {
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}

// Rows rp .. rp+R-1 (through a_rows when given), k-range [kc, kc+kn) of the bf16 activations ->
// sA as fp32 (row stride KC), with 16-byte loads; K and kn are multiples of 8 and the rows 16-byte
// aligned.
template <int KC>
__device__ __forceinline__ void stage_rows(const __nv_bfloat16* __restrict__ a, const int32_t* __restrict__ a_rows,
                                           int K, int rp, int R, int kc, int kn, float* sA) {
  const int per_row = KC / 8;
  for (int i = threadIdx.x; i < R * per_row; i += kThreads) {
    const int r = i / per_row, kk = (i % per_row) * 8;
    const size_t src = a_rows != nullptr ? (size_t)a_rows[rp + r] : (size_t)(rp + r);
    float v[8];
    if (kk < kn) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a + src * K + kc + kk)), v);
    else
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;
    float4* dst = reinterpret_cast<float4*>(sA + r * KC + kk);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// up (STAGE 1) writes bf16 h; down (STAGE 2) writes fp32 y_perm.
// RMAX rows of an expert per pass over its weights (more rows take more passes).
template <int STAGE, typename OutT, int RMAX>
__global__ void __launch_bounds__(kThreads, 2)
ffn_stream_kernel(const __nv_bfloat16* __restrict__ a, const int32_t* __restrict__ a_rows,
                  const __nv_bfloat16* __restrict__ w, const int32_t* __restrict__ offsets,
                  const float* __restrict__ row_gate, int K, int N, int E, OutT* __restrict__ out) {
  constexpr int kUnroll = unroll_for<RMAX>();
  constexpr int KC = kc_for<RMAX>();
  extern __shared__ __align__(16) float smem[];
  float* sA = smem;                         // [RMAX][KC]
  float* sRed = sA + RMAX * KC;             // [kWarps][RMAX][NS]
  int* sAct = reinterpret_cast<int*>(sRed + kWarps * RMAX * NS);  // [E] experts with rows
  __shared__ int s_nact;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool act = e < E && offsets[e + 1] > offsets[e];
      const unsigned m = __ballot_sync(0xffffffffu, act);
      if (act) sAct[base + __popc(m & ((1u << lane) - 1u))] = e;
      base += __popc(m);
    }
    if (lane == 0) s_nact = base;
  }
  __syncthreads();
  const int nslab = (N + NS - 1) / NS;
  const int units = s_nact * nslab;
  const int kr = lane / LPR;            // k-row of this lane within the warp's group of RPW
  const int cg = lane % LPR;            // 8-column group of this lane

  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int e = sAct[u / nslab];
    const int n0 = (u % nslab) * NS;
    const int col = n0 + cg * 8;
    const bool col_ok = col < N;
    const __nv_bfloat16* we = w + (size_t)e * K * N;
    const int r_begin = offsets[e], r_end = offsets[e + 1];
    for (int rp = r_begin; rp < r_end; rp += RMAX) {
      const int R = min(RMAX, r_end - rp);
      uint64_t acc2[RMAX][4];  // column pairs (2p, 2p+1) of each row, fp32x2
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc2[r][p] = 0ull;

      for (int kc = 0; kc < K; kc += KC) {
        const int kn = min(KC, K - kc);
        // Software-pipelined: the next batch of kUnroll weight loads is issued before the
        // current batch is consumed, so two batches per thread are in flight. The first batch
        // goes out before the activations are staged, so staging overlaps the weight stream.
        auto load_batch = [&](int k0, uint4 (&wv)[kUnroll]) {
#pragma unroll
          for (int i = 0; i < kUnroll; ++i) {
            const int kk = k0 + i * KSTEP + warp * RPW + kr;
            if (col_ok && kk < kn)
              wv[i] = __ldg(reinterpret_cast<const uint4*>(we + (size_t)(kc + kk) * N + col));
            else
              wv[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        };
        uint4 cur[kUnroll], nxt[kUnroll];
        load_batch(0, cur);
        __syncthreads();
        stage_rows<KC>(a, a_rows, K, rp, R, kc, kn, sA);
        __syncthreads();
        for (int k0 = 0; k0 < kn; k0 += KSTEP * kUnroll) {
          if (k0 + KSTEP * kUnroll < kn) load_batch(k0 + KSTEP * kUnroll, nxt);
#pragma unroll
          for (int i = 0; i < kUnroll; ++i) {
            const int kk = k0 + i * KSTEP + warp * RPW + kr;
            if (kk >= kn) break;
            // bf16 pair (lo, hi) of each 32-bit word -> two fp32 in one 64-bit register
            const uint32_t wv[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
            uint64_t w2[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) w2[p] = ((uint64_t)(wv[p] & 0xFFFF0000u) << 32) | (uint64_t)(wv[p] << 16);
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
              if (r >= R) break;
              const float av = sA[r * KC + kk];
              const uint64_t av2 = f2_pack(av, av);
#pragma unroll
              for (int p = 0; p < 4; ++p) acc2[r][p] = ffma2(av2, w2[p], acc2[r][p]);
            }
          }
#pragma unroll
          for (int i = 0; i < kUnroll; ++i) cur[i] = nxt[i];
        }
      }
      // Combine the RPW k-row groups of the warp (lanes cg, cg+8, cg+16, cg+24), then the warps.
      float acc[RMAX][8];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float v = c & 1 ? f2_hi(acc2[r][c >> 1]) : f2_lo(acc2[r][c >> 1]);
          v += __shfl_xor_sync(0xffffffffu, v, LPR);
          v += __shfl_xor_sync(0xffffffffu, v, 2 * LPR);
          acc[r][c] = v;
        }
      if (lane < LPR) {
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int c = 0; c < 8; ++c) sRed[(warp * RMAX + r) * NS + cg * 8 + c] = acc[r][c];
      }
      __syncthreads();
      for (int i = tid; i < R * NS; i += kThreads) {
        const int r = i / NS, c = i % NS;
        const int gn = n0 + c;
        if (gn >= N) continue;
        float v = 0.f;
#pragma unroll
        for (int wi = 0; wi < kWarps; ++wi) v += sRed[(wi * RMAX + r) * NS + c];
        const int grow = rp + r;
        v = STAGE == 1 ? gelu_as(v) : row_gate[grow] * v;
        out[(size_t)grow * N + gn] = from_f32<OutT>(v);
      }
    }
  }
}

template <int STAGE, typename OutT, int RMAX>
cudaError_t launch_t(const FfnArgs& p, cudaStream_t s) {
  const size_t smem = (size_t)(RMAX * kc_for<RMAX>() + kWarps * RMAX * NS) * sizeof(float) + (size_t)p.E * sizeof(int);
  auto kern = ffn_stream_kernel<STAGE, OutT, RMAX>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int nslab = (p.N + NS - 1) / NS;
  const long long max_units = (long long)(p.rows < p.E ? p.rows : p.E) * nslab;
  long long grid = (long long)device_sm_count() * (RMAX <= 2 ? 8 : 4);
  if (grid > max_units) grid = max_units;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, (const __nv_bfloat16*)p.a, p.a_rows,
                    (const __nv_bfloat16*)p.w, p.offsets, p.row_gate, p.K, p.N, p.E, (OutT*)p.out);
}

}  // namespace

cudaError_t launch_ffn_stream(const FfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  if (p.dt != MOE_DTYPE_BF16) return cudaErrorNotSupported;
  // Rows per expert are at most T*k; small batches keep fewer accumulators (more CTAs per SM).
  // An expert with more rows than a pass holds streams its weights again for the rest.
  if (p.max_rows_per_expert == 1)
    return p.stage == 1 ? launch_t<1, __nv_bfloat16, 1>(p, s) : launch_t<2, float, 1>(p, s);
  if (p.rows <= 32)
    return p.stage == 1 ? launch_t<1, __nv_bfloat16, 2>(p, s) : launch_t<2, float, 2>(p, s);
  return p.stage == 1 ? launch_t<1, __nv_bfloat16, 4>(p, s) : launch_t<2, float, 4>(p, s);
}

}  // namespace moe
