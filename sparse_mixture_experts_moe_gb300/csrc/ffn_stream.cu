// Weight-streaming grouped expert FFN for batches with few rows per expert (decode).
// csdn/6a919c0d §2.3: with top-2 routing each token reads two experts' full W1 and W2
// from HBM, so the layer is bound by moving weights, not by arithmetic.
//
// Work unit = (expert with at least one row, 64-column slab of its weight matrix).
// A CTA owns the slab for the full depth K, so the GeLU (up) or gate (down)
// epilogue applies locally and no partial sums leave the CTA. Units are ordered
// slab-fastest, so CTAs running together stream neighbouring slabs of the same
// matrix rows.
//
// The weights arrive by TMA: one producer warp keeps a ring of five 16 KB boxes
// (64 columns x 128 k-rows of one expert) in flight per CTA, two CTAs per SM, so the
// bytes in flight do not depend on registers. The eight consumer warps read each box
// from shared memory, 8 lanes x 16 bytes per k-row, and release it to the producer.
// The expert's rows (1, 2 or 4 per pass, by batch size; more rows take more passes)
// are staged as fp32 in shared memory between named barriers of the consumer warps
// only, so the weight stream never waits for them.
// Partial sums are combined in a fixed order (xor-butterfly in the warp, then
// warps in index order), so results are reproducible.
//
// Ring depth, box height and L2 promotion were swept on decode shapes (d = d_ff =
// 8192, 1/8/64 tokens): 128-row boxes five deep without promotion were best or
// within noise of the best everywhere; three deep fell to 0.83 of HBM for one token,
// and 64-row boxes lost 2-5%.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256, kWarps = 8;  // consumer warps
constexpr int NS = 64;                     // columns per slab
constexpr int LPR = NS / 8;                // lanes per k-row: 8 (16 bytes each)
constexpr int RPW = 32 / LPR;              // k-rows per warp per step: 4
constexpr int KSTEP = kWarps * RPW;        // k-rows per CTA step: 32

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

constexpr int kTmaRows = 128;                    // k-rows per box
constexpr int kTmaBoxBytes = kTmaRows * NS * 2;  // 16 KB
constexpr int kTmaStages = 5;                    // boxes in flight per CTA
constexpr int kTmaThreads = kThreads + 32;       // 8 consumer warps + the producer warp
constexpr int kTmaActFloats = 4096;              // staged activations: RMAX rows x 4096/RMAX
constexpr int kBarSlotBytes = 128;               // the ring's mbarriers: 2 x kTmaStages x 8 bytes
static_assert(2 * kTmaStages * 8 <= kBarSlotBytes, "the mbarriers fit their slot");

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
// The weights' copies at L2 evict-first priority (see stream_evict_first).
__device__ __forceinline__ uint64_t policy_evict_first_s() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_3d_first(uint32_t dst, const void* tmap, int c0, int c1, int c2,
                                                  uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol) : "memory");
}

template <int STAGE, typename OutT, int RMAX>
__global__ void __launch_bounds__(kTmaThreads, 2)
ffn_stream_tma_kernel(const __grid_constant__ CUtensorMap tmW, const __nv_bfloat16* __restrict__ a,
                      const int32_t* __restrict__ a_rows, const int32_t* __restrict__ offsets,
                      const float* __restrict__ row_gate, int K, int N, int E, int nst, OutT* __restrict__ out,
                      int* status, uint64_t timeout_ns, int evict_first) {
  constexpr int KC = kTmaActFloats / RMAX;  // a multiple of kTmaRows
  extern __shared__ uint8_t smem_raw[];
  // ring [nst][kTmaRows][NS] bf16 (128-byte aligned) | full [nst], empty [nst] mbarriers in a
  // 128-byte slot | sA [RMAX][KC] fp32 (the epilogue's per-warp sums reuse it) | sAct [E]
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 127u) & ~127u;
  uint8_t* gring = smem_raw + (ring - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gring + nst * kTmaBoxBytes);
  float* sA = reinterpret_cast<float*>(gring + nst * kTmaBoxBytes + kBarSlotBytes);
  float* sRed = sA;  // [kWarps][RMAX][NS]
  int* sAct = reinterpret_cast<int*>(sA + RMAX * KC);
  __shared__ int s_nact, s_abort;
  volatile int* abort_flag = &s_abort;
  auto full = [&](int st) { return smem_u32(bars + st); };
  auto empty = [&](int st) { return smem_u32(bars + nst + st); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == kWarps && lane == 0) {
    for (int st = 0; st < nst; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), kWarps);
    }
    fence_mbar_init();
    *abort_flag = 0;
    tma_prefetch_desc(&tmW);
  }
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
  const int KB = (K + kTmaRows - 1) / kTmaRows;  // boxes per pass; rows past K arrive as zeros

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int st = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int e = sAct[u / nslab], n0 = (u % nslab) * NS;
        const int passes = (offsets[e + 1] - offsets[e] + RMAX - 1) / RMAX;
        for (int ps = 0; ps < passes; ++ps)
          for (int kb = 0; kb < KB; ++kb) {
            if (!wait_or_abort(empty(st), phase ^ 1u, timeout_ns, abort_flag, status, 51)) goto producer_out;
            mbar_arrive_expect_tx(full(st), kTmaBoxBytes);
            if (evict_first)
              tma_load_3d_first(ring + st * kTmaBoxBytes, &tmW, n0, kb * kTmaRows, e, full(st), policy_evict_first_s());
            else
              tma_load_3d(ring + st * kTmaBoxBytes, &tmW, n0, kb * kTmaRows, e, full(st));
            filled |= 1u << st;
            fill_phase = (fill_phase & ~(1u << st)) | (phase << st);
            if (++st == nst) { st = 0; phase ^= 1u; }
          }
      }
    producer_out:
      // copies in flight land before the CTA (and its shared memory) goes away
      for (int q = 0; q < nst; ++q)
        if (filled & (1u << q)) mbar_wait_bounded(full(q), (fill_phase >> q) & 1u, timeout_ns);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers (warps 0..7)
  // Every consumer warp runs the same trip counts, so the named barriers always match; after a
  // failed wait (recorded in the status word) the warps skip the arithmetic and run to the end.
  const int kr = lane / LPR, cg = lane % LPR;
  int st = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int e = sAct[u / nslab];
    const int n0 = (u % nslab) * NS;
    const int r_begin = offsets[e], r_end = offsets[e + 1];
    for (int rp = r_begin; rp < r_end; rp += RMAX) {
      const int R = min(RMAX, r_end - rp);
      uint64_t acc2[RMAX][4];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc2[r][q] = 0ull;
      for (int kc = 0; kc < K; kc += KC) {
        const int kn = min(KC, K - kc);
        consumer_sync();  // the previous chunk's activations (or the last epilogue's sums) are read
        stage_rows<KC>(a, a_rows, K, rp, R, kc, kn, sA);
        consumer_sync();
        for (int kb = 0; kb < kn; kb += kTmaRows) {
          if (ok) ok = wait_or_abort(full(st), phase, timeout_ns, abort_flag, status, 52);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            const uint8_t* box = gring + st * kTmaBoxBytes;
#pragma unroll
            for (int i = 0; i < kTmaRows / KSTEP; ++i) {
              const int kk = i * KSTEP + warp * RPW + kr;  // k-row within the box
              const uint4 v = *reinterpret_cast<const uint4*>(box + kk * (NS * 2) + cg * 16);
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
              uint64_t w2[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) w2[q] = ((uint64_t)(wv[q] & 0xFFFF0000u) << 32) | (uint64_t)(wv[q] << 16);
#pragma unroll
              for (int r = 0; r < RMAX; ++r) {
                if (r >= R) break;
                const float av = sA[r * KC + kb + kk];
                const uint64_t av2 = f2_pack(av, av);
#pragma unroll
                for (int q = 0; q < 4; ++q) acc2[r][q] = ffma2(av2, w2[q], acc2[r][q]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty(st));  // the box's slot goes back to the producer
          if (++st == nst) { st = 0; phase ^= 1u; }
        }
      }
      // the warp's RPW k-row groups (lanes cg, cg+8, cg+16, cg+24), then the warps in index order
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
      consumer_sync();  // sRed overlays the activations
      if (lane < LPR) {
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int c = 0; c < 8; ++c) sRed[(warp * RMAX + r) * NS + cg * 8 + c] = acc[r][c];
      }
      consumer_sync();
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

constexpr size_t kSmPerSmBytes = 228 * 1024;  // shared memory per SM, of which 1 KB per resident CTA is reserved

size_t tma_smem_bytes(int nst, int E) {
  return 128 + (size_t)nst * kTmaBoxBytes + kBarSlotBytes + (size_t)kTmaActFloats * sizeof(float) + (size_t)E * 4;
}

template <int STAGE, typename OutT, int RMAX>
cudaError_t launch_tma(const FfnArgs& p, EncodeTiledFn enc, cudaStream_t s) {
  // the deepest ring that keeps two CTAs per SM
  // five boxes deep, fewer where a large E leaves no room for two CTAs per SM
  int nst = kTmaStages;
  while (nst > 2 && 2 * (tma_smem_bytes(nst, p.E) + 1024) > kSmPerSmBytes) --nst;
  const size_t smem = tma_smem_bytes(nst, p.E);
  auto kern = ffn_stream_tma_kernel<STAGE, OutT, RMAX>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // weights [E][K][N] as a 3D map: 64 columns x 128 k-rows of one expert per box, no swizzle, no L2
  // promotion (each weight byte is read once); rows past K and columns past N arrive as zeros
  CUtensorMap tmW;
  const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.K, (cuuint64_t)p.E};
  const cuuint64_t str[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.K * p.N * 2};
  const cuuint32_t box[3] = {NS, kTmaRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.w), dims, str, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int nslab = (p.N + NS - 1) / NS;
  const long long max_units = (long long)(p.rows < p.E ? p.rows : p.E) * nslab;
  long long grid = 2LL * device_sm_count();  // persistent: the resident CTAs loop over the units
  if (grid > max_units) grid = max_units;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kTmaThreads), smem, s, tmW, (const __nv_bfloat16*)p.a, p.a_rows,
                    p.offsets, p.row_gate, p.K, p.N, p.E, nst, (OutT*)p.out, p.status, p.timeout_ns,
                    (int)stream_evict_first(p.rows, p.E, p.K, p.N, 16));
}

}  // namespace

cudaError_t launch_ffn_stream(const FfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  if (p.dt != MOE_DTYPE_BF16) return cudaErrorNotSupported;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // Rows per expert are at most T*k; one row a pass for one token, two for small batches, four
  // otherwise. An expert with more rows than a pass holds streams its weights again for the rest.
  if (p.max_rows_per_expert == 1)
    return p.stage == 1 ? launch_tma<1, __nv_bfloat16, 1>(p, enc, s) : launch_tma<2, float, 1>(p, enc, s);
  if (p.rows <= 32)
    return p.stage == 1 ? launch_tma<1, __nv_bfloat16, 2>(p, enc, s) : launch_tma<2, float, 2>(p, enc, s);
  return p.stage == 1 ? launch_tma<1, __nv_bfloat16, 4>(p, enc, s) : launch_tma<2, float, 4>(p, enc, s);
}

}  // namespace moe
