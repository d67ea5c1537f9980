// Grouped expert GEMM on CTA pairs (tcgen05 cta_group::2), for experts with many routed rows.
// Same math and epilogues as ffn_tc.cu (csdn/6a462027 §3.2 and §4.2 step 6; gate:
// csdn/6a919c0d §2.2 step 4):
//   up   (stage 1): h[r]      = GeLU(x_perm[r] W1[e])            (bf16 out)
//   down (stage 2): y_perm[r] = row_gate[r] * (h[r] W2[e])        (fp32 out)
//
// A cluster of two CTAs on two SMs computes a 256-row x 256-column tile with one
// tcgen05.mma.cta_group::2 per 16-deep k-step (M = 256, N = 256): each CTA holds its own 128
// rows of A and its own 128 columns of B in shared memory, and its TMEM receives its 128 rows
// of the result. Per SM this halves the weight bytes per FLOP compared with one-CTA 128x256
// tiles (32 KB instead of 48 KB per 64-deep k-block), so six stages fit in shared memory and
// cover about twice as much load latency.
//
// Roles (both CTAs run 10 warps):
//   warp 0      TMA producer of this CTA's halves; its loads complete on the leader CTA's
//               "full" barrier (the leader arms it with both CTAs' bytes)
//   warp 1      TMEM allocation for the pair; in the leader CTA also the MMA issuer, whose
//               commits arrive on both CTAs' "empty" / "accumulator full" barriers
//   warps 2..9  epilogue of this CTA's 128 rows (two warps per TMEM lane quarter), then an
//               arrival on the leader's "accumulator empty" barrier
// All waits are bounded; on a timeout the CTA records MOE_ERR_DEVICE_TIMEOUT and unwinds.
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BMP = 256;                            // rows per pair tile
constexpr int BM = 128, BN = 256, BK = 64;           // per CTA: 128 rows, 256 columns of D
constexpr int kTileABytes = BM * BK * 2;             // 16 KB: this CTA's rows of A
constexpr int kTileBSubBytes = BK * 64 * 2;          // 8 KB: 64 k-rows x 64 columns
constexpr int kTileBBytes = BK * (BN / 2) * 2;       // 16 KB: this CTA's 128 columns of B
constexpr int kStageBytes = kTileABytes + kTileBBytes;
constexpr int kEpiWarps = 8;
constexpr int kStagingBytes = 32 * 128;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kMaxSmem = 232448;

__host__ __device__ constexpr int num_bars(int nst) { return 2 * nst + 5; }
__host__ __device__ constexpr size_t smem_bytes_for(int E, int nst) {
  return 1024 + (size_t)nst * kStageBytes + (size_t)kEpiWarps * kStagingBytes + 8 * num_bars(nst) + 16 +
         4 * (size_t)(E + 1);
}

struct Item {
  int e, row0, row_end, n0;
};

// Item w of the list (expert, 256-column block, 256-row pair tile), pair tile fastest.
__device__ __forceinline__ Item decode_item(int w, const int* P, int E, int NB, const int32_t* offsets) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P[mid] * NB <= w) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mt = P[e + 1] - P[e];
  const int r = w - P[e] * NB;
  Item it;
  it.e = e;
  it.row0 = offsets[e] + (r % mt) * BMP;
  it.row_end = offsets[e + 1];
  it.n0 = (r / mt) * BN;
  return it;
}

template <int STAGE>
struct EpiOut { using T = __nv_bfloat16; };
template <>
struct EpiOut<2> { using T = float; };

template <int STAGE, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
ffn_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, typename EpiOut<STAGE>::T* __restrict__ out,
               const int32_t* __restrict__ offsets, const float* __restrict__ row_gate, int K, int N, int E,
               int* status, uint64_t timeout_ns) {
  using OutT = typename EpiOut<STAGE>::T;
  constexpr int CW = 128 / (int)sizeof(OutT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + STAGES * kTileABytes;
  const uint32_t sStg = sB + STAGES * kTileBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * kStageBytes + kEpiWarps * kStagingBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + num_bars(STAGES));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* P = reinterpret_cast<int*>(tmem_slot + 4);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, TEMPTY = 2 * STAGES + 2, DONE = 2 * STAGES + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(bar(FULL + s), 1); mbar_init(bar(EMPTY + s), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(bar(TFULL + a), 1); mbar_init(bar(TEMPTY + a), 2 * kEpiWarps); }
    mbar_init(bar(DONE), 1);
    fence_mbar_init();
    *abort_flag = 0;
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  griddep_launch_dependents();
  griddep_wait();
  if (warp == 2) {
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int mt = 0;
      if (e < E) {
        const int cnt = offsets[e + 1] - offsets[e];
        mt = cnt > 0 ? (cnt + BMP - 1) / BMP : 0;
      }
      int incl = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) P[e] = run + incl - mt;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) P[E] = run;
  }
  // Both CTAs' barriers must be initialised before any signal crosses to the peer.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int NB = (N + BN - 1) / BN;
  const int KB = (K + BK - 1) / BK;
  const int total_items = P[E] * NB;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int w = pair; w < total_items && !*abort_flag; w += npairs) {
        const Item it = decode_item(w, P, E, NB, offsets);
        const int row0 = it.row0 + BM * (int)rank;
        const int col0 = it.n0 + (BN / 2) * (int)rank;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(bar(EMPTY + stage), phase ^ 1u, timeout_ns, abort_flag, status, 31)) goto producer_out;
          const uint32_t full_leader = map_to_cta(bar(FULL + stage), 0);
          if (leader) mbar_arrive_expect_tx(bar(FULL + stage), 2 * kStageBytes);
          tma_load_2d_pair(sA + stage * kTileABytes, &tmA, kb * BK, row0, full_leader);
#pragma unroll
          for (int j = 0; j < BN / 128; ++j)
            tma_load_3d_pair(sB + stage * kTileBBytes + j * kTileBSubBytes, &tmB, col0 + 64 * j, kb * BK, it.e,
                             full_leader);
          filled |= 1u << stage;
          fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    producer_out:
      // Copies in flight must land before shared memory goes away: the leader waits for the phases
      // it armed (they count both CTAs' bytes); the peer waits until the MMAs released its last fills.
      for (int s = 0; s < STAGES; ++s) {
        if (!(filled & (1u << s))) continue;
        const uint32_t ph = (fill_phase >> s) & 1u;
        if (leader) mbar_wait_bounded(bar(FULL + s), ph, timeout_ns);
        else mbar_wait_bounded(bar(EMPTY + s), ph, timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // ---------------------------------------------------------- MMA issuer (leader only)
        constexpr uint32_t idesc = make_idesc_bf16_f32(BMP, BN, /*b_mn_major=*/true);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        for (int w = pair; w < total_items && !*abort_flag; w += npairs) {
          if (!wait_or_abort(bar(TEMPTY + acc), acc_phase ^ 1u, timeout_ns, abort_flag, status, 32)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          for (int kb = 0; kb < KB; ++kb) {
            if (!wait_or_abort(bar(FULL + stage), phase, timeout_ns, abort_flag, status, 32)) goto mma_out;
            tc_fence_after();
            const uint64_t a_desc = make_smem_desc_sw128(sA + stage * kTileABytes, 16, 1024);
            const uint64_t b_desc = make_smem_desc_sw128(sB + stage * kTileBBytes, kTileBSubBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_f16_pair(d_tmem, a_desc + (uint64_t)((kk * 32) >> 4),
                              b_desc + (uint64_t)((kk * 16 * 128) >> 4), idesc, (kb | kk) != 0 ? 1u : 0u);
            tc_commit_pair(bar(EMPTY + stage), 0x3);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          tc_commit_pair(bar(TFULL + acc), 0x3);
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
      mma_out:
        tc_commit_pair(bar(DONE), 0x3);
      }
      // Both CTAs: every MMA writing this CTA's TMEM has completed before TMEM is freed.
      mbar_wait_bounded(bar(DONE), 0, timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- epilogue (warps 2..9)
    const int q = warp & 3;
    const int c_begin = ((warp - 2) >> 2) * (BN / 2);
    const uint32_t stg = sStg + (uint32_t)((warp - 2) * kStagingBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = pair; w < total_items && !*abort_flag; w += npairs) {
      const Item it = decode_item(w, P, E, NB, offsets);
      if (!wait_or_abort(bar(TFULL + acc), acc_phase, timeout_ns, abort_flag, status, 33)) break;
      tc_fence_after();
      const int row0 = it.row0 + BM * (int)rank;
      const int grow = row0 + 32 * q + lane;
      const bool row_ok = grow < it.row_end;
      const bool group_full = row0 + 32 * q + 31 < it.row_end;
      float g = 1.f;
      if (STAGE == 2 && row_ok) g = row_gate[grow];
      for (int c = c_begin; c < c_begin + BN / 2; c += CW) {
        if (it.n0 + c >= N) break;
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN + c);
        uint32_t packed[32];
        if (STAGE == 1) {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(taddr, v0);
          tmem_ld_32x32b_x32(taddr + 32, v1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            packed[i] = pack_bf16x2(gelu_as(__uint_as_float(v0[2 * i])), gelu_as(__uint_as_float(v0[2 * i + 1])));
            packed[16 + i] =
                pack_bf16x2(gelu_as(__uint_as_float(v1[2 * i])), gelu_as(__uint_as_float(v1[2 * i + 1])));
          }
        } else {
          uint32_t v0[32];
          tmem_ld_32x32b_x32(taddr, v0);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) packed[i] = __float_as_uint(g * __uint_as_float(v0[i]));
        }
        if (group_full) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t dst = stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) * 16));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[4 * j]),
                         "r"(packed[4 * j + 1]), "r"(packed[4 * j + 2]), "r"(packed[4 * j + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, stg, it.n0 + c, row0 + 32 * q);
            bulk_commit_group();
          }
        } else if (row_ok) {
          OutT* dst = out + (size_t)grow * N + it.n0 + c;
          constexpr int per16 = 16 / (int)sizeof(OutT);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (it.n0 + c + per16 * j < N)
              *reinterpret_cast<uint4*>(dst + per16 * j) =
                  make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(TEMPTY + acc), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  // No signal may target a CTA that has left, and no MMA may still write TMEM being freed.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_ffn_tensor_pair(const FfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  if (p.dt != MOE_DTYPE_BF16) return cudaErrorNotSupported;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmA, tmB, tmC;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.rows};
    const cuuint64_t str[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!encode_tmap(enc, &tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.a, 2, dims, str, box))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.K, (cuuint64_t)p.E};
    const cuuint64_t str[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.K * p.N * 2};
    const cuuint32_t box[3] = {64, BK, 1};
    if (!encode_tmap(enc, &tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.w, 3, dims, str, box))
      return cudaErrorInvalidValue;
  }
  {
    const bool f32_out = p.stage == 2;
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.rows};
    const cuuint64_t str[1] = {(cuuint64_t)p.N * (f32_out ? 4 : 2)};
    const cuuint32_t box[2] = {f32_out ? 32u : 64u, 32};
    if (!encode_tmap(enc, &tmC, f32_out ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.out,
                     2, dims, str, box))
      return cudaErrorInvalidValue;
  }
  const bool six = smem_bytes_for(p.E, 6) <= (size_t)kMaxSmem;
  const size_t smem = smem_bytes_for(p.E, six ? 6 : 5);
  const int NB = (p.N + BN - 1) / BN;
  const long long max_items = ((long long)(p.rows + BMP - 1) / BMP + p.E) * NB;
  // Persistent: as many pairs as can be resident at once (two-SM clusters may not tile every SM).
  auto resident_pairs = [&](auto kern) -> long long {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(device_sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0)
      return device_sm_count() / 2;
    return clusters;
  };
  cudaError_t err;
  if (p.stage == 1) {
    auto kern = six ? ffn_tc2_kernel<1, 6> : ffn_tc2_kernel<1, 5>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    long long pairs = resident_pairs(kern);
    if (pairs > max_items) pairs = max_items;
    err = launch_pdl(kern, dim3((unsigned)(2 * pairs)), dim3(kThreads), smem, s, tmA, tmB, tmC,
                     (__nv_bfloat16*)p.out, p.offsets, p.row_gate, p.K, p.N, p.E, p.status, p.timeout_ns);
  } else {
    auto kern = six ? ffn_tc2_kernel<2, 6> : ffn_tc2_kernel<2, 5>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    long long pairs = resident_pairs(kern);
    if (pairs > max_items) pairs = max_items;
    err = launch_pdl(kern, dim3((unsigned)(2 * pairs)), dim3(kThreads), smem, s, tmA, tmB, tmC, (float*)p.out,
                     p.offsets, p.row_gate, p.K, p.N, p.E, p.status, p.timeout_ns);
  }
  return err;
}

}  // namespace moe
