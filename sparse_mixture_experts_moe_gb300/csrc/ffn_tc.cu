// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
// csdn/6a462027 §3.2 and §4.2 step 6 (grouped GEMM over the routed rows of each expert),
// with GeLU fused into the up-projection epilogue and the gate into the down-projection's
// (csdn/6a919c0d §2.2 step 4).
//
// out[r, n] = epi( sum_k a[r, k] * w[e][k, n] ) for every row r of expert e's range.
//   up   (stage 1): a = x_perm [rows, d], w = W1 [E, d, F], epi = GeLU (erf form, gelu_as)
//   down (stage 2): a = h [rows, F],      w = W2 [E, F, d], epi = row_gate[r] * ., fp32 output
//
// Tiles: 128 rows x 256 columns x 64-deep k-blocks, one tcgen05.mma of M=128, N=256, K=16
// per 16 k. A tiles are K-major, B tiles MN-major (the weights are stored [K, N], N
// contiguous), both 128-byte swizzled exactly as TMA writes them. The fp32 accumulator
// lives in TMEM; two accumulators (512 columns) let the epilogue of one tile overlap the
// main loop of the next.
//
// Persistent CTAs, one per SM, 10 warps:
//   warp 0      TMA producer (one lane): A tile + 4 B sub-tiles per stage, 4 stages (3 when E is
//               large)
//   warp 1      TMEM allocator and MMA issuer (one lane)
//   warps 2..9  epilogue (two per TMEM lane quarter, half the columns each): tcgen05.ld ->
//               GeLU -> bf16 (up) or gate -> fp32 (down) -> swizzled staging -> TMA store
// Work items are (expert, 256-column block, 128-row tile), the row tile fastest, so the
// CTAs that run at the same time share the same weight tile (read once from HBM, then from
// L2). The item list is derived on the device from `offsets`: no host round trip.
// Rows of a tile that lie past the expert's end are computed but never stored.
//
// Every wait is bounded (globaltimer); on a timeout the CTA records
// MOE_ERR_DEVICE_TIMEOUT, raises a CTA-wide abort flag, waits (bounded) for its own
// copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kTileABytes = BM * BK * 2;           // 16 KB
constexpr int kTileBSubBytes = BK * 64 * 2;        // 8 KB: 64 k-rows x 64 columns
constexpr int kTileBBytes = BK * BN * 2;           // 32 KB
constexpr int kStageBytes = kTileABytes + kTileBBytes;
// Two epilogue warps per TMEM lane quarter, each taking half of the tile's 256 columns.
constexpr int kEpiWarps = 8;
constexpr int kStagingBytes = 32 * 128;            // per epilogue warp: 32 rows x 128 bytes
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kMaxSmem = 232448;                   // opt-in shared memory per CTA on sm_103a

__host__ __device__ constexpr int num_bars(int nst) { return 2 * nst + 5; }
__host__ __device__ constexpr size_t smem_bytes_for(int E, int nst) {
  return 1024 /* alignment slack */ + (size_t)nst * kStageBytes + (size_t)kEpiWarps * kStagingBytes +
         8 * num_bars(nst) + 16 + 4 * (size_t)(E + 1);
}

struct Item {
  int e, row0, row_end, n0;
};

// Largest e with NB*P[e] <= w (the expert holding item w; empty experts share P with the next one).
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
  it.row0 = offsets[e] + (r % mt) * BM;
  it.row_end = offsets[e + 1];
  it.n0 = (r / mt) * BN;
  return it;
}

template <int STAGE>
struct EpiOut { using T = __nv_bfloat16; };
template <>
struct EpiOut<2> { using T = float; };

template <int STAGE, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
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
  int* P = reinterpret_cast<int*>(tmem_slot + 4);  // [E+1] exclusive scan of 128-row tiles per expert
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, TEMPTY = 2 * STAGES + 2, DONE = 2 * STAGES + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(bar(FULL + s), 1); mbar_init(bar(EMPTY + s), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(bar(TFULL + a), 1); mbar_init(bar(TEMPTY + a), kEpiWarps); }
    mbar_init(bar(DONE), 1);
    fence_mbar_init();
    *abort_flag = 0;
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  griddep_launch_dependents();
  griddep_wait();  // offsets, rows and weights may come from earlier kernels in the stream
  if (warp == 2) {
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int mt = 0;
      if (e < E) {
        const int cnt = offsets[e + 1] - offsets[e];
        mt = cnt > 0 ? (cnt + BM - 1) / BM : 0;
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int NB = (N + BN - 1) / BN;
  const int KB = (K + BK - 1) / BK;
  const int total_items = P[E] * NB;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int w = blockIdx.x; w < total_items && !*abort_flag; w += gridDim.x) {
        const Item it = decode_item(w, P, E, NB, offsets);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(bar(EMPTY + stage), phase ^ 1u, timeout_ns, abort_flag, status, 1)) goto producer_out;
          mbar_arrive_expect_tx(bar(FULL + stage), kStageBytes);
          tma_load_2d(sA + stage * kTileABytes, &tmA, kb * BK, it.row0, bar(FULL + stage));
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_3d(sB + stage * kTileBBytes + j * kTileBSubBytes, &tmB, it.n0 + 64 * j, kb * BK, it.e,
                        bar(FULL + stage));
          filled |= 1u << stage;
          fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    producer_out:
      // Every copy this CTA issued must have landed before its shared memory goes away.
      for (int s = 0; s < STAGES; ++s)
        if (filled & (1u << s)) mbar_wait_bounded(bar(FULL + s), (fill_phase >> s) & 1u, timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16_f32(BM, BN, /*b_mn_major=*/true);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int w = blockIdx.x; w < total_items && !*abort_flag; w += gridDim.x) {
        if (!wait_or_abort(bar(TEMPTY + acc), acc_phase ^ 1u, timeout_ns, abort_flag, status, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(bar(FULL + stage), phase, timeout_ns, abort_flag, status, 2)) goto mma_out;
          tc_fence_after();
          const uint64_t a_desc = make_smem_desc_sw128(sA + stage * kTileABytes, 16, 1024);
          const uint64_t b_desc = make_smem_desc_sw128(sB + stage * kTileBBytes, kTileBSubBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_f16(d_tmem, a_desc + (uint64_t)((kk * 32) >> 4), b_desc + (uint64_t)((kk * 16 * 128) >> 4),
                       idesc, (kb | kk) != 0 ? 1u : 0u);
          tc_commit(bar(EMPTY + stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        tc_commit(bar(TFULL + acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    mma_out:
      // All issued MMAs complete before TMEM is freed.
      tc_commit(bar(DONE));
      mbar_wait_bounded(bar(DONE), 0, timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- epilogue (warps 2..9)
    const int q = warp & 3;                   // TMEM lanes 32q .. 32q+31 belong to this warp
    const int c_begin = ((warp - 2) >> 2) * (BN / 2);  // and this half of the tile's columns
    const uint32_t stg = sStg + (uint32_t)((warp - 2) * kStagingBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = blockIdx.x; w < total_items && !*abort_flag; w += gridDim.x) {
      const Item it = decode_item(w, P, E, NB, offsets);
      if (!wait_or_abort(bar(TFULL + acc), acc_phase, timeout_ns, abort_flag, status, 3)) break;
      tc_fence_after();
      const int grow = it.row0 + 32 * q + lane;
      const bool row_ok = grow < it.row_end;
      const bool group_full = it.row0 + 32 * q + 31 < it.row_end;
      float g = 1.f;
      if (STAGE == 2 && row_ok) g = row_gate[grow];
      // One staging row is 128 bytes: 64 bf16 columns (up) or 32 fp32 columns (down).
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
          if (lane == 0) bulk_wait_group_read0();  // the previous store has finished reading the buffer
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
            tma_store_2d(&tmC, stg, it.n0 + c, it.row0 + 32 * q);
            bulk_commit_group();
          }
        } else if (row_ok) {
          // The 32-row group straddles the end of the expert's rows: plain stores of the valid rows.
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
      if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// One CTA waits on a barrier that nothing completes; the bounded wait gives up,
// records MOE_ERR_DEVICE_TIMEOUT and the kernel returns normally.
__global__ void selftest_wait_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    wait_or_abort(smem_u32(&never), 0, timeout_ns, &abort_flag, status, 99);
  __syncthreads();
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool encode_tmap(EncodeTiledFn enc, CUtensorMap* m, CUtensorMapDataType type, const void* ptr, int rank,
                 const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, type, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides_bytes, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
bool encode_tmap_plain(EncodeTiledFn enc, CUtensorMap* m, CUtensorMapDataType type, const void* ptr, int rank,
                       const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, type, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides_bytes, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_ffn_tensor(const FfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  if (p.dt != MOE_DTYPE_BF16) return cudaErrorNotSupported;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmA, tmB, tmC;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.rows};
    const cuuint64_t str[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!encode_tmap(enc, &tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.a, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.K, (cuuint64_t)p.E};
    const cuuint64_t str[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.K * p.N * 2};
    const cuuint32_t box[3] = {64, BK, 1};
    if (!encode_tmap(enc, &tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.w, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // up writes bf16 h (64-column boxes), down writes fp32 y_perm (32-column boxes): 128-byte rows
    const bool f32_out = p.stage == 2;
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.rows};
    const cuuint64_t str[1] = {(cuuint64_t)p.N * (f32_out ? 4 : 2)};
    const cuuint32_t box[2] = {f32_out ? 32u : 64u, 32};
    if (!encode_tmap(enc, &tmC, f32_out ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.out, 2,
                dims, str, box))
      return cudaErrorInvalidValue;
  }
  const bool four = smem_bytes_for(p.E, 4) <= (size_t)kMaxSmem;
  const size_t smem = smem_bytes_for(p.E, four ? 4 : 3);
  const int NB = (p.N + BN - 1) / BN;
  const long long max_items = ((long long)(p.rows + BM - 1) / BM + p.E) * NB;
  int grid = device_sm_count();
  if ((long long)grid > max_items) grid = (int)max_items;
  cudaError_t err;
  if (p.stage == 1) {
    auto kern = four ? ffn_tc_kernel<1, 4> : ffn_tc_kernel<1, 3>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, tmA, tmB, tmC, (__nv_bfloat16*)p.out, p.offsets,
                     p.row_gate, p.K, p.N, p.E, p.status, p.timeout_ns);
  } else {
    auto kern = four ? ffn_tc_kernel<2, 4> : ffn_tc_kernel<2, 3>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, tmA, tmB, tmC, (float*)p.out, p.offsets, p.row_gate,
                     p.K, p.N, p.E, p.status, p.timeout_ns);
  }
  return err;
}

cudaError_t launch_selftest_wait(int* status, uint64_t timeout_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
