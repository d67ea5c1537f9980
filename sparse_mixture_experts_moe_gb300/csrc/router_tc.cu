// Router on the tensor cores: logits = x W_r (+ b_r), softmax over the E experts and
// deterministic top-k, fused in one kernel.
// csdn/6a919c0d §2.2 steps 1-4; aicoding/6a320eef §3.2; csdn/6a919c0d §4.2 (max subtraction).
//
// The router is a dense [T, d] x [d, E] contraction, so each CTA computes the logits of
// 128 tokens with tcgen05.mma (M = 128 tokens, N = E rounded up to 64, K = d in 64-deep
// blocks fed by TMA) into a TMEM accumulator. In TMEM, lane r holds token r's logits, so
// each epilogue thread owns one token: it reads its row 32 columns at a time with
// tcgen05.ld, keeps the k best (logit, expert) pairs in registers (a strictly greater
// logit displaces, so equal logits keep the lower expert index first) and the maximum,
// then sums exp(l - max) in ascending expert order and writes the k gates
// exp(l_j - max) / sum. Fixed orders everywhere: results are reproducible.
//
// Warps: 0 = TMA producer, 1 = TMEM allocator + MMA issuer, 2..5 = one token per thread.
// For at most 128 tokens, deep d (at least 16 k-blocks) and E <= 128, a cluster of eight CTAs
// splits d (router_tc_split_kernel).
// All waits are bounded (see wait_or_abort).
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"
#include "router_stats.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int kTileXBytes = BM * BK * 2;     // 16 KB
constexpr int kTileWSubBytes = BK * 64 * 2;  // 8 KB: 64 k-rows x 64 experts
constexpr int kThreads = 192;
__host__ __device__ constexpr int num_bars(int nst) { return 2 * nst + 2; }

// Pipeline depth: about 192 KB of x and W_r tiles in flight per CTA (the router streams x once and
// is bound by load latency): 8 stages of 24 KB (E <= 64), 6 of 32 KB (E <= 128), 4 of 48 KB.
template <int EN>
constexpr int stages_plain() { return EN <= 64 ? 8 : EN <= 128 ? 6 : 4; }
// The split kernel also holds the 128 x EN partial-logit table.
template <int EN>
constexpr int stages_split() { return EN <= 64 ? 6 : 4; }

template <int EN, int NST>
constexpr size_t router_smem_bytes() {
  return 1024 + (size_t)NST * (kTileXBytes + EN / 64 * kTileWSubBytes) + 8 * num_bars(NST) + 16;
}

// Routing statistics: [4][EN] per-warp soft-load sums, [4] entropy sums, [EN] counts.
template <int EN>
constexpr size_t router_stat_bytes() {
  return (size_t)(5 * EN + 4) * sizeof(float);
}

// Insert (v, e) into the descending list bv/bi of length k (k <= KMAX). A value equal to an
// entry already present goes after it: the scan is in ascending e, so lower indices stay first.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&bv)[KMAX], int (&bi)[KMAX], int k, float v, int e) {
#pragma unroll
  for (int p = 0; p < KMAX; ++p) {
    if (p < k && v > bv[p]) {
      const float tv = bv[p];
      const int ti = bi[p];
      bv[p] = v; bi[p] = e;
      v = tv; e = ti;
    }
  }
}

template <int EN, int KMAX, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const float* __restrict__ b_r, int Tn, int d, int E, int k, int renorm, RouterStats st,
                 int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, int* status, uint64_t timeout_ns) {
  constexpr int kTileWBytes = EN / 64 * kTileWSubBytes;
  constexpr int kStageBytes = kTileXBytes + kTileWBytes;
  constexpr uint32_t kCols = EN;  // 64, 128 or 256: a power of two >= 32
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sX = base;
  const uint32_t sW = base + STAGES * kTileXBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + num_bars(STAGES));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_soft = reinterpret_cast<float*>(gbase + STAGES * kStageBytes + 8 * num_bars(STAGES) + 16);  // [4][EN]
  float* s_ent = s_soft + 4 * EN;                                                             // [4]
  int* s_cnt = reinterpret_cast<int*>(s_ent + 4);                                             // [EN]
  const bool stats = st.part != nullptr;
  const bool hist = st.hist != nullptr;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, DONE = 2 * STAGES + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * BM;
  const int KB = (d + BK - 1) / BK;
  if (stats || hist)
    for (int i = threadIdx.x; i < 5 * EN + 4; i += kThreads) s_soft[i] = 0.f;  // zero bits: also int 0

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(bar(FULL + s), 1); mbar_init(bar(EMPTY + s), 1); }
    mbar_init(bar(TFULL), 1);
    mbar_init(bar(DONE), 1);
    fence_mbar_init();
    *abort_flag = 0;
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kCols);
    tmem_relinquish();
  }
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // x may come from the previous kernel in the stream

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_or_abort(bar(EMPTY + stage), phase ^ 1u, timeout_ns, abort_flag, status, 11)) break;
        mbar_arrive_expect_tx(bar(FULL + stage), kStageBytes);
        tma_load_2d(sX + stage * kTileXBytes, &tmX, kb * BK, t0, bar(FULL + stage));
#pragma unroll
        for (int j = 0; j < EN / 64; ++j)
          tma_load_2d(sW + stage * kTileWBytes + j * kTileWSubBytes, &tmW, 64 * j, kb * BK, bar(FULL + stage));
        filled |= 1u << stage;
        fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      for (int s = 0; s < STAGES; ++s)
        if (filled & (1u << s)) mbar_wait_bounded(bar(FULL + s), (fill_phase >> s) & 1u, timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16_f32(BM, EN, /*b_mn_major=*/true);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_or_abort(bar(FULL + stage), phase, timeout_ns, abort_flag, status, 12)) { ok = false; break; }
        tc_fence_after();
        const uint64_t a_desc = make_smem_desc_sw128(sX + stage * kTileXBytes, 16, 1024);
        const uint64_t b_desc = make_smem_desc_sw128(sW + stage * kTileWBytes, kTileWSubBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_f16(tmem_base, a_desc + (uint64_t)((kk * 32) >> 4), b_desc + (uint64_t)((kk * 16 * 128) >> 4),
                     idesc, (kb | kk) != 0 ? 1u : 0u);
        tc_commit(bar(EMPTY + stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok) tc_commit(bar(TFULL));
      tc_commit(bar(DONE));
      mbar_wait_bounded(bar(DONE), 0, timeout_ns);
    }
  } else {
    const int q = warp & 3;
    const int tok = t0 + 32 * q + lane;
    // warp-uniform: the TMEM loads and shuffles below are warp-collective
    const bool ok = __all_sync(0xffffffffu, wait_or_abort(bar(TFULL), 0, timeout_ns, abort_flag, status, 13));
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16);
      float bv[KMAX];
      int bi[KMAX];
#pragma unroll
      for (int p = 0; p < KMAX; ++p) { bv[p] = -INFINITY; bi[p] = 0x7fffffff; }
      // pass 1: the k largest logits (the first of them is the maximum)
#pragma unroll 1
      for (int c = 0; c < E; c += 32) {  // the padding columns past E are not read
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int e = c + j;
          if (e < E) topk_insert<KMAX>(bv, bi, k, __uint_as_float(v[j]) + (b_r != nullptr ? b_r[e] : 0.f), e);
        }
      }
      const float m = bv[0];
      // pass 2: sum of exp(l - max) in ascending expert order (the softmax denominator; skipped
      // for renormalised gates unless the statistics want it), and for renormalised gates the
      // sum over the k chosen logits in slot order
      float ssum = 0.f, ksum = 0.f;
      if (renorm) {
#pragma unroll
        for (int p = 0; p < KMAX; ++p)
          if (p < k) ksum += expf(bv[p] - m);
      }
#pragma unroll 1
      for (int c = 0; c < (renorm && !stats ? 0 : E); c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int e = c + j;
          if (e < E) ssum += expf(__uint_as_float(v[j]) + (b_r != nullptr ? b_r[e] : 0.f) - m);
        }
      }
      const float gden = renorm ? ksum : ssum;
      if (tok < Tn) {
#pragma unroll
        for (int p = 0; p < KMAX; ++p) {
          if (p < k) {
            topk_idx[(size_t)tok * k + p] = bi[p];
            topk_gate[(size_t)tok * k + p] = expf(bv[p] - m) / gden;
            if (stats || hist) atomicAdd(&s_cnt[bi[p]], 1);
          }
        }
      }
      if (stats) {
        // pass 3: p = exp(z) / ssum with z = l - max; per-warp column sums of p over the warp's
        // 32 tokens, and the token entropy ln ssum - sum p z
        float hs = 0.f;
#pragma unroll 1
        for (int c = 0; c < E; c += 32) {  // the padding columns past E are not read
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)c, v);
          tmem_ld_wait();
          float pv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int e = c + j;
            const float z = __uint_as_float(v[j]) + (b_r != nullptr && e < E ? b_r[e] : 0.f) - m;
            const float p = (tok < Tn && e < E) ? expf(z) / ssum : 0.f;
            pv[j] = p;
            hs += p * z;
          }
          s_soft[q * EN + c + lane] = warp_column_sums(pv);
        }
        const float ent = warp_sum_xor(tok < Tn ? logf(ssum) - hs : 0.f);
        if (lane == 0) s_ent[q] = ent;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCols);
  }
  if (hist)
    for (int e = threadIdx.x; e < E; e += kThreads) st.hist[(size_t)blockIdx.x * E + e] = s_cnt[e];
  if (stats) router_stats_cta(st, s_soft, 4, EN, s_ent, s_cnt, E, Tn, k);
}

// Split-K version: one cluster of kSplit CTAs per 128-token tile, CTA r accumulating the
// k-blocks [r*KB/kSplit, (r+1)*KB/kSplit) in its own TMEM. Each epilogue thread copies its
// token's partial logits to shared memory; after a cluster barrier, CTA r finishes tokens
// [r*16, r*16+16): one warp per token sums the kSplit partials in rank order (DSMEM loads),
// then softmax and top-k with warp shuffles (lane l owns experts l, l+32, ...).
constexpr int kSplit = 8;

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

template <int EN>
constexpr size_t router_split_smem_bytes() {
  return router_smem_bytes<EN, stages_split<EN>()>() + (size_t)BM * (EN + 1) * sizeof(float) +
         router_stat_bytes<EN>();
}

template <int EN, int KMAX, int STAGES>
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kThreads, 1)
router_tc_split_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const float* __restrict__ b_r, int Tn, int d, int E, int k, int renorm,
                       RouterStats st, int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
                       int* status, uint64_t timeout_ns) {
  constexpr int kTileWBytes = EN / 64 * kTileWSubBytes;
  constexpr int kStageBytes = kTileXBytes + kTileWBytes;
  constexpr uint32_t kCols = EN;
  constexpr int RS = EN + 1;  // padded row stride of the partial-logit table
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sX = base;
  const uint32_t sW = base + STAGES * kTileXBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + num_bars(STAGES));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(gbase + STAGES * kStageBytes + 8 * num_bars(STAGES) + 16);  // [BM][RS]
  float* s_soft = red + BM * RS;                   // statistics: [4][EN] per-warp soft-load sums
  float* s_ent = s_soft + 4 * EN;                  // [4]
  int* s_cnt = reinterpret_cast<int*>(s_ent + 4);  // [EN]
  const bool stats = st.part != nullptr;
  const bool hist = st.hist != nullptr;
  if (stats || hist)
    for (int i = threadIdx.x; i < 5 * EN + 4; i += kThreads) s_soft[i] = 0.f;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, DONE = 2 * STAGES + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int t0 = (blockIdx.x / kSplit) * BM;  // this cluster's 128-token tile
  const int KB = (d + BK - 1) / BK;
  const int kb0 = (int)rank * KB / kSplit, kb1 = ((int)rank + 1) * KB / kSplit;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(bar(FULL + s), 1); mbar_init(bar(EMPTY + s), 1); }
    mbar_init(bar(TFULL), 1);
    mbar_init(bar(DONE), 1);
    fence_mbar_init();
    *abort_flag = 0;
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kCols);
    tmem_relinquish();
  }
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_or_abort(bar(EMPTY + stage), phase ^ 1u, timeout_ns, abort_flag, status, 14)) break;
        mbar_arrive_expect_tx(bar(FULL + stage), kStageBytes);
        tma_load_2d(sX + stage * kTileXBytes, &tmX, kb * BK, t0, bar(FULL + stage));
#pragma unroll
        for (int j = 0; j < EN / 64; ++j)
          tma_load_2d(sW + stage * kTileWBytes + j * kTileWSubBytes, &tmW, 64 * j, kb * BK, bar(FULL + stage));
        filled |= 1u << stage;
        fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      for (int s = 0; s < STAGES; ++s)
        if (filled & (1u << s)) mbar_wait_bounded(bar(FULL + s), (fill_phase >> s) & 1u, timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16_f32(BM, EN, /*b_mn_major=*/true);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_or_abort(bar(FULL + stage), phase, timeout_ns, abort_flag, status, 15)) { ok = false; break; }
        tc_fence_after();
        const uint64_t a_desc = make_smem_desc_sw128(sX + stage * kTileXBytes, 16, 1024);
        const uint64_t b_desc = make_smem_desc_sw128(sW + stage * kTileWBytes, kTileWSubBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_f16(tmem_base, a_desc + (uint64_t)((kk * 32) >> 4), b_desc + (uint64_t)((kk * 16 * 128) >> 4),
                     idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
        tc_commit(bar(EMPTY + stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok) tc_commit(bar(TFULL));
      tc_commit(bar(DONE));
      mbar_wait_bounded(bar(DONE), 0, timeout_ns);
    }
  } else {
    // partial logits of this CTA's k-range -> shared memory (row = token)
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const bool ok = __all_sync(0xffffffffu, wait_or_abort(bar(TFULL), 0, timeout_ns, abort_flag, status, 16));
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
      for (int c = 0; c < E; c += 32) {  // the padding columns past E are not read
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) red[row * RS + c + j] = __uint_as_float(v[j]);
      }
    } else {
      for (int c = 0; c < EN; ++c) red[row * RS + c] = 0.f;
    }
  }
  tc_fence_before();
  cluster_sync_all();  // every CTA's partials are in its shared memory

  if (warp >= 2) {
    constexpr int kRowsPerCta = BM / kSplit;  // 16
    constexpr int kEpi = 4;
    float accp[EN / 32];  // statistics: this lane's soft-load sums (experts lane + 32 j)
#pragma unroll
    for (int j = 0; j < EN / 32; ++j) accp[j] = 0.f;
    float went = 0.f;
    for (int i = warp - 2; i < kRowsPerCta; i += kEpi) {
      const int row = (int)rank * kRowsPerCta + i;
      const int tok = t0 + row;
      if (tok >= Tn) break;
      float lv[EN / 32];
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < EN / 32; ++j) {
        const int e = lane + 32 * j;
        float v = 0.f;
        const uint32_t local = smem_u32(red + row * RS + e);
#pragma unroll
        for (int c = 0; c < kSplit; ++c) v += ld_shared_cluster_f32(map_to_cta(local, c));
        v += (b_r != nullptr && e < E) ? b_r[e] : 0.f;
        lv[j] = e < E ? v : -INFINITY;
        m = fmaxf(m, lv[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float ssum = 0.f;
#pragma unroll
      for (int j = 0; j < EN / 32; ++j)
        if (lane + 32 * j < E) ssum += expf(lv[j] - m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
      if (stats) {
        float hs = 0.f;
#pragma unroll
        for (int j = 0; j < EN / 32; ++j) {
          if (lane + 32 * j < E) {
            const float z = lv[j] - m;
            const float p = expf(z) / ssum;
            accp[j] += p;
            hs += p * z;
          }
        }
        went += logf(ssum) - warp_sum_xor(hs);
      }
      float sel[8];
      for (int p = 0; p < k; ++p) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < EN / 32; ++j)
          if (lv[j] > bv) { bv = lv[j]; be = lane + 32 * j; }  // ascending e in a lane: lower index kept
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        sel[p] = bv;
        if (lane == 0) {
          topk_idx[(size_t)tok * k + p] = be;
          if (stats || hist) atomicAdd(&s_cnt[be], 1);
        }
#pragma unroll
        for (int j = 0; j < EN / 32; ++j)
          if (lane + 32 * j == be) lv[j] = -INFINITY;
      }
      float ksum = 0.f;
      if (renorm)
        for (int p = 0; p < k; ++p) ksum += expf(sel[p] - m);
      if (lane == 0)
        for (int p = 0; p < k; ++p) topk_gate[(size_t)tok * k + p] = expf(sel[p] - m) / (renorm ? ksum : ssum);
    }
    if (stats) {
#pragma unroll
      for (int j = 0; j < EN / 32; ++j) s_soft[(warp - 2) * EN + lane + 32 * j] = accp[j];
      if (lane == 0) s_ent[warp - 2] = went;
    }
  }
  if (hist) {
    // the tile's histogram: every CTA moves its rows' counts into rank 0's (integer adds: exact), so
    // the statistics partials still sum to each expert's count once
    __syncthreads();
    if (rank != 0)
      for (int e = threadIdx.x; e < E; e += kThreads) {
        const int v = s_cnt[e];
        s_cnt[e] = 0;
        if (v != 0)
          asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(map_to_cta(smem_u32(s_cnt + e), 0)), "r"(v)
                       : "memory");
      }
  }
  cluster_sync_all();  // no CTA leaves while a peer may still read its partials (or add to its counts)
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCols);
  }
  if (hist && rank == 0)
    for (int e = threadIdx.x; e < E; e += kThreads) st.hist[(size_t)(blockIdx.x / kSplit) * E + e] = s_cnt[e];
  if (stats) router_stats_cta(st, s_soft, 4, EN, s_ent, s_cnt, E, Tn, k);
}

template <int EN, int KMAX>
cudaError_t launch_en(const CUtensorMap& tmX, const CUtensorMap& tmW, const float* b_r, int Tn, int d, int E,
                      int k, int renorm, const RouterStats& st, int32_t* idx, float* gate, int* status,
                      uint64_t timeout_ns, cudaStream_t s) {
  if (EN <= 128 && Tn <= BM && (d + BK - 1) / BK >= 2 * kSplit) {
    // one token tile and deep d: a single CTA would stream all of W_r alone, so a cluster of
    // kSplit CTAs splits d (measured: 51 -> 14 us at T = 1, d = 8192). With more tiles the
    // DSMEM reduction costs more than it saves (T = 4096, d = 1024: 14.6 -> 27.6 us), so
    // larger batches keep one CTA per tile.
    const size_t smem = router_split_smem_bytes<EN>();
    auto kern = router_tc_split_kernel<EN, KMAX, stages_split<EN>()>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(kSplit * ((Tn + BM - 1) / BM)), dim3(kThreads), smem, s, tmX, tmW, b_r, Tn, d, E,
                      k, renorm, st, idx, gate, status, timeout_ns);
  }
  const size_t smem = router_smem_bytes<EN, stages_plain<EN>()>() + router_stat_bytes<EN>();
  auto kern = router_tc_kernel<EN, KMAX, stages_plain<EN>()>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3((Tn + BM - 1) / BM), dim3(kThreads), smem, s, tmX, tmW, b_r, Tn, d, E, k, renorm, st,
                    idx, gate, status, timeout_ns);
}

template <int KMAX>
cudaError_t launch_k(const CUtensorMap& tmX, const CUtensorMap& tmW, const float* b_r, int Tn, int d, int E, int k,
                     int renorm, const RouterStats& st, int32_t* idx, float* gate, int* status, uint64_t timeout_ns,
                     cudaStream_t s) {
  if (E <= 64) return launch_en<64, KMAX>(tmX, tmW, b_r, Tn, d, E, k, renorm, st, idx, gate, status, timeout_ns, s);
  if (E <= 128) return launch_en<128, KMAX>(tmX, tmW, b_r, Tn, d, E, k, renorm, st, idx, gate, status, timeout_ns, s);
  return launch_en<256, KMAX>(tmX, tmW, b_r, Tn, d, E, k, renorm, st, idx, gate, status, timeout_ns, s);
}

}  // namespace

cudaError_t launch_router_tc(const void* x, const void* w_r, const float* b_r, int Tn, int d, int E, int k,
                             int renorm, const RouterStats& st, int32_t* idx, float* gate, int* status,
                             uint64_t timeout_ns, cudaStream_t s) {
  if (Tn == 0) return cudaSuccess;
  if (E > 256 || E % 8 != 0) return cudaErrorNotSupported;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmX, tmW;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)Tn};
    const cuuint64_t str[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!encode_tmap(enc, &tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)d};
    const cuuint64_t str[1] = {(cuuint64_t)E * 2};
    const cuuint32_t box[2] = {64, BK};
    if (!encode_tmap(enc, &tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_r, 2, dims, str, box))
      return cudaErrorInvalidValue;
  }
  if (k <= 2) return launch_k<2>(tmX, tmW, b_r, Tn, d, E, k, renorm, st, idx, gate, status, timeout_ns, s);
  return launch_k<8>(tmX, tmW, b_r, Tn, d, E, k, renorm, st, idx, gate, status, timeout_ns, s);
}

}  // namespace moe
