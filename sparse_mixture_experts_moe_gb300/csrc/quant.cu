// Block quantisation of expert weights and the weight-streaming expert FFN that reads them.
// csdn/6a462500 §4.3 (64 x 64 blocks, each with its own min and max); csdn/6a919c0d §2.3 (decode
// is bound by moving expert weights, so fewer bytes per weight is the lever).
//
// Quantiser: per 64 x 64 block, scale = (max - min) / (2^bits - 1) and
// code = round((w - min) / scale), in fp32 with correctly rounded subtraction and division and
// rounding half to even, so the codes are a deterministic function of the weights; w is restored
// as min + code * scale (the page's dequantisation would lose the block minimum).
//
// Memory format of the codes of one [K, N] matrix: the fragment layouts of the tensor-core streaming
// kernels (quantize_kernel describes the orders). INT4: [N/64 slabs][K/16 steps][32 lanes][4 words],
// INT8: [N/64 slabs][K/16 steps][2 halves][32 lanes][16 bytes]. Scales: one (scale, min) float pair
// per block, [K/64][N/64] per expert.
//
// Streaming kernels (ffn_stream_q4_kernel, ffn_stream_q8_kernel): the structure of ffn_stream.cu
// (work unit = (expert with rows, 64-column slab), full depth per CTA, fixed-order reductions) with
// the dequantisation folded into the dot product:
//   sum_k a_k (min_b + c_k scale_b) = sum_b [ scale_b (a . (c - m)) + (min_b + m scale_b) sum_b a ]
// with the centre m = 8 (INT4) or 128 (INT8); the products a . (c - m) run on the tensor cores.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int QB = 64;  // block edge
constexpr int kThreads = 256, kWarps = 8;  // consumer threads and warps (and the quantiser's)
constexpr int NS = 64;              // columns per slab (one block column)

// ------------------------------------------------------------------ quantiser
template <typename T, int BITS>
__global__ void __launch_bounds__(256)
quantize_kernel(const T* __restrict__ w, int K, int N, uint4* __restrict__ codes, float2* __restrict__ sm) {
  static_assert(BITS == 4 || BITS == 8, "INT4 or INT8 codes");
  constexpr float levels = (float)((1 << BITS) - 1);
  __shared__ float blk[QB][QB + 1];
  __shared__ float s_lo[kWarps], s_hi[kWarps];
  const int nbj = N / QB, nbi = K / QB;
  const int bj = blockIdx.x % nbj;
  const int bi = (blockIdx.x / nbj) % nbi;
  const int e = blockIdx.x / (nbj * nbi);
  const T* src = w + ((size_t)e * K + (size_t)bi * QB) * N + (size_t)bj * QB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float lo = INFINITY, hi = -INFINITY;
  for (int i = tid; i < QB * QB; i += 256) {
    const int r = i / QB, c = i % QB;
    const float v = to_f32(src[(size_t)r * N + c]);
    blk[r][c] = v;
    lo = fminf(lo, v);
    hi = fmaxf(hi, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) { s_lo[warp] = lo; s_hi[warp] = hi; }
  __syncthreads();
  lo = s_lo[0];
  hi = s_hi[0];
  for (int i = 1; i < kWarps; ++i) { lo = fminf(lo, s_lo[i]); hi = fmaxf(hi, s_hi[i]); }
  const float scale = __fdiv_rn(__fsub_rn(hi, lo), levels);
  if (tid == 0) sm[((size_t)e * nbi + bi) * nbj + bj] = make_float2(scale, lo);
  auto code = [&](int r, int c) -> uint32_t {
    if (!(scale > 0.f)) return 0u;
    return (uint32_t)rintf(__fdiv_rn(__fsub_rn(blk[r][c], lo), scale));
  };
  if constexpr (BITS == 4) {
    // INT4: the fragment layout of the tensor-core streaming kernel. Per (64-column slab, 16-deep
    // step j of a 64-deep block) 512 bytes: lane l = 4g + t holds four words, word m covering columns
    // 16m + g (c0) and 16m + g + 8 (c1) at the block's k-rows kp .. kp+3, kp = 16t + 4j, nibbles (k, c):
    //   0: (kp, c0)  1: (kp, c1)  2: (kp+2, c0)  3: (kp+2, c1)  4: (kp+1, c0)  5: (kp+1, c1)
    //   6: (kp+3, c0)  7: (kp+3, c1),
    // so that (word >> 4i) & 0x000F000F puts register i of an m16n8k16 A fragment (rows = columns of
    // w) in place, nibble i in the low half and nibble i + 4 in the high half, with the fragment's
    // k-rows 2t, 2t+1, 2t+8, 2t+9 standing for kp .. kp+3: then lane t's B fragments for the four
    // steps are the block's 16 consecutive activations 16t .. 16t+15.
    uint32_t* cw = reinterpret_cast<uint32_t*>(codes);
    for (int wi = tid; wi < (QB / 16) * 32 * 4; wi += 256) {
      const int m = wi & 3, lane = (wi >> 2) & 31, j = wi >> 7;
      const int g = lane >> 2, t = lane & 3;
      const int c0 = 16 * m + g, c1 = c0 + 8, k0 = 16 * t + 4 * j;
      const uint32_t v = code(k0, c0) | code(k0, c1) << 4 | code(k0 + 2, c0) << 8 | code(k0 + 2, c1) << 12 |
                         code(k0 + 1, c0) << 16 | code(k0 + 1, c1) << 20 | code(k0 + 3, c0) << 24 |
                         code(k0 + 3, c1) << 28;
      const size_t k16 = (size_t)bi * (QB / 16) + j;
      cw[((((size_t)e * nbj + bj) * (K / 16) + k16) * 32 + lane) * 4 + m] = v;
    }
  } else {
    // INT8: the fragment layout of the tensor-core streaming kernel, fp16 A operands. Per (64-column
    // slab, 16-deep step) 1 KB, [2 halves][32 lanes][16 bytes]: half h of lane l = 4g + t holds the A
    // fragments of column tiles 2h and 2h + 1, 8 bytes each in register order a0 .. a7; the tile m
    // covers columns c0 = 16m + g and c1 = c0 + 8, and step 2p + s of the block's 32-deep range p
    // (k-rows kp .. kp+3, kp = 32p + 8t + 4s) holds (k, column) = (kp, c0), (kp+1, c0), (kp, c1),
    // (kp+1, c1), (kp+2, c0), (kp+3, c0), (kp+2, c1), (kp+3, c1): the fragment's k-rows 2t, 2t+1, 2t+8,
    // 2t+9 stand for kp .. kp+3, so lane t's B fragments for the range's two steps are its 8
    // consecutive activations 32p + 8t .. 32p + 8t + 7.
    for (int q = tid; q < (QB / 16) * 64; q += 256) {
      const int lane = q & 31, h = (q >> 5) & 1, j = q >> 6;
      const int g = lane >> 2, t = lane & 3;
      const int kp = 32 * (j >> 1) + 8 * t + 4 * (j & 1);
      uint32_t word[4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int c0 = 16 * (2 * h + mi) + g, c1 = c0 + 8;
        word[2 * mi] = code(kp, c0) | code(kp + 1, c0) << 8 | code(kp, c1) << 16 | code(kp + 1, c1) << 24;
        word[2 * mi + 1] = code(kp + 2, c0) | code(kp + 3, c0) << 8 | code(kp + 2, c1) << 16 | code(kp + 3, c1) << 24;
      }
      const size_t k16 = (size_t)bi * (QB / 16) + j;
      codes[(((size_t)e * nbj + bj) * (K / 16) + k16) * 64 + h * 32 + lane] =
          make_uint4(word[0], word[1], word[2], word[3]);
    }
  }
}

// ------------------------------------------------------------------ streaming FFN on the tensor cores
// The codes of a 64-column slab arrive by TMA in the fragment layout the quantiser writes: one
// producer warp keeps a ring of 16 KB boxes in flight (two CTAs per SM), and eight consumer warps
// multiply them on mma.sync m16n8k16 (fp32 accumulate): A = 16 weight columns x 16 k-rows decoded
// in registers, B = 16 k-rows x 8 activation rows (tokens), so one instruction does 2048
// multiply-adds and a pass takes up to 8 rows at the cost of one.
//   INT4, bf16 operands: one shift and one LOP3 put two nibbles n into the low mantissa bits of
//   bf16 128.0 (128 + n, exact), one packed bf16 subtraction of 136 leaves the centred code n - 8
//   (exact). A box holds 32 steps of 16 k-rows; each warp takes one 64-deep block of it.
//   INT8, fp16 operands: one byte permute puts two codes b into the low mantissa bytes of fp16
//   1024.0 (1024 + b, exact: fp16 keeps 10 mantissa bits where bf16 keeps 7), one packed fp16
//   subtraction of 1152 leaves the centred code b - 128 (exact): two instructions per two weights.
//   The activations become fp16, exactly for bf16 values in fp16's normal range (values below 2^-14
//   keep fp16's subnormal spacing, 2^-24). A box holds 16 steps; each warp takes a 32-deep range.
// Within a warp's range the code layout numbers k so that the B fragments of lane 4g + t for all the
// range's steps are consecutive k-rows of activation row g: the lane loads them from global memory
// (16-byte loads, one box ahead of use) and nothing is staged in shared memory. A range lies in one
// 64 x 64 block, whose (scale, min) pair scales the range's accumulator once per box; the
// column-independent term (min + centre * scale) * (sum of the range's activations) takes one more
// MMA per step, with an A fragment of ones, whose result is each row's sum over the step's k-rows.
constexpr int kTmaBoxBytes = 16384;         // one box of codes
constexpr int kTmaStages = 5;               // boxes in flight per CTA (fewer where shared memory runs short)
constexpr int kTmaThreads = kThreads + 32;  // 8 consumer warps + the producer warp
constexpr int kBarSlotBytes = 128;          // the ring's mbarriers: 2 x kTmaStages x 8 bytes
static_assert(2 * kTmaStages * 8 <= kBarSlotBytes, "the mbarriers fit their slot");
constexpr int kQRows = 8;                   // activation rows per pass: the MMA's N

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
// An 8-byte asynchronous copy global -> shared (n = 0: zero fill, nothing read), and an arrive on an
// mbarrier once this thread's earlier such copies have landed (counted in the barrier's init count).
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src, int n) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// The codes' copies at L2 evict-first priority (see stream_evict_first).
__device__ __forceinline__ uint64_t policy_evict_first_q() {
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

template <int BITS>
struct QCodes {
  static constexpr int kStepBytes = BITS * 128;                      // one 16-deep step of a slab: 512 / 1024
  static constexpr int kWarpSteps = BITS == 4 ? 4 : 2;               // steps per warp per box
  static constexpr int kBoxSteps = kTmaBoxBytes / kStepBytes;        // 32 / 16
  static constexpr int kWarpK = 16 * kWarpSteps;                     // k-rows per warp per box: 64 / 32
  static constexpr int kBoxK = 16 * kBoxSteps;                       // k-rows per box: 512 / 256
  static constexpr float kCentre = (float)(1 << (BITS - 1));
  static constexpr uint32_t kOnePair = BITS == 4 ? 0x3F803F80u : 0x3C003C00u;  // 1.0 in both halves
  // INT8: the producer warp copies each box's (scale, min) pairs into shared memory beside the box
  // (an INT8 box passes in about 0.8 us, too short to hide the pairs' global load one box ahead).
  // INT4: each consumer warp loads its pair one box ahead (measured: the copy made INT4 5% slower).
  static constexpr bool kScalesInSmem = BITS == 8;
  static_assert(kWarps * kWarpSteps == kBoxSteps, "the warps split a box");
  static_assert(QB % kWarpK == 0, "a warp's range lies in one block");
};

__device__ __forceinline__ uint32_t q4_pair(uint32_t word, int shift) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(word >> shift), "r"(0x000F000Fu), "r"(0x43004300u));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(0x43084308u));  // (128 + n) - 136 = n - 8, exact
  return r;
}
// bytes (sel & 0xF) and ((sel >> 8) & 0xF) of word as centred fp16 codes
__device__ __forceinline__ uint32_t q8_pair(uint32_t word, uint32_t sel) {
  uint32_t r = __byte_perm(word, 0x64646464u, sel);  // fp16 (1024 + b) in both halves
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(0x64806480u));  // (1024 + b) - 1152 = b - 128, exact
  return r;
}
// two bf16 values (low, high) -> the same two as fp16
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(w & 0xFFFF0000u)), "f"(__uint_as_float(w << 16)));
  return r;
}
template <int BITS>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BITS == 4)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int BITS, int STAGE, typename OutT>
__device__ __forceinline__ void stream_q_body(const CUtensorMap* tmC, const __nv_bfloat16* __restrict__ a,
                                              const int32_t* __restrict__ a_rows, const float2* __restrict__ sm,
                                              const int32_t* __restrict__ offsets, const float* __restrict__ row_gate,
                                              int K, int N, int E, int nst, OutT* __restrict__ out, int* status,
                                              uint64_t timeout_ns, int evict_first) {
  using C = QCodes<BITS>;
  extern __shared__ uint8_t smem_raw[];
  // ring [nst][16 KB] (128-byte aligned) | full [nst], empty [nst] mbarriers in a 128-byte slot |
  // sQ [kTmaStages][kWarps] (each box's (scale, min) per warp) | sRed [kWarps][kQRows][NS] (warp sums) |
  // sMinW [kWarps][kQRows] (warp block-minimum terms) | sAct [E]
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 127u) & ~127u;
  uint8_t* gring = smem_raw + (ring - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gring + nst * kTmaBoxBytes);
  float2* sQ = reinterpret_cast<float2*>(gring + nst * kTmaBoxBytes + kBarSlotBytes);
  float* sRed = reinterpret_cast<float*>(sQ + kTmaStages * kWarps);
  float* sMinW = sRed + kWarps * kQRows * NS;
  int* sAct = reinterpret_cast<int*>(sMinW + kWarps * kQRows);
  __shared__ int s_nact, s_abort;
  volatile int* abort_flag = &s_abort;
  auto full = [&](int st) { return smem_u32(bars + st); };
  auto empty = [&](int st) { return smem_u32(bars + nst + st); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == kWarps && lane == 0) {
    for (int st = 0; st < nst; ++st) {
      mbar_init(full(st), C::kScalesInSmem ? 1 + kWarps : 1);  // expect-tx arrive (+ the sQ copies)
      mbar_init(empty(st), kWarps);
    }
    fence_mbar_init();
    *abort_flag = 0;
    tma_prefetch_desc(tmC);
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
  const int nslab = N / NS;
  const int units = s_nact * nslab;
  const int K16 = K / 16;
  const int KB = (K16 + C::kBoxSteps - 1) / C::kBoxSteps;  // boxes per pass; steps past K arrive as zeros

  const int NB = N / QB, KQ = K / QB;
  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    // Lane 0 waits for a free slot and copies the box (TMA). INT8: lanes 0..kWarps-1 also copy the
    // (scale, min) pair of each consumer warp's range beside it; both land on the slot's full barrier.
    if (C::kScalesInSmem || lane == 0) {
      int st = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int e = sAct[u / nslab], slab = u % nslab;
        const float2* sm_e = sm + (size_t)e * KQ * NB + slab;  // block b's (scale, min) at sm_e[b * NB]
        const int passes = (offsets[e + 1] - offsets[e] + kQRows - 1) / kQRows;
        for (int ps = 0; ps < passes; ++ps)
          for (int kb = 0; kb < KB; ++kb) {
            bool free_slot = true;
            if (lane == 0) free_slot = wait_or_abort(empty(st), phase ^ 1u, timeout_ns, abort_flag, status, 55);
            if constexpr (C::kScalesInSmem) {
              if (!__shfl_sync(0xffffffffu, free_slot, 0)) goto producer_out;
              if (lane < kWarps) {
                const int kw = kb * C::kBoxK + lane * C::kWarpK;  // past K: zeros
                cp_async_8(smem_u32(sQ + st * kWarps + lane), kw < K ? sm_e + (size_t)(kw / QB) * NB : sm,
                           kw < K ? 8 : 0);
                cp_async_arrive_noinc(full(st));
              }
            } else if (!free_slot) {
              goto producer_out;
            }
            if (lane == 0) {
              mbar_arrive_expect_tx(full(st), kTmaBoxBytes);
              if (evict_first)
                tma_load_3d_first(ring + st * kTmaBoxBytes, tmC, 0, kb * C::kBoxSteps, e * nslab + slab, full(st),
                                  policy_evict_first_q());
              else
                tma_load_3d(ring + st * kTmaBoxBytes, tmC, 0, kb * C::kBoxSteps, e * nslab + slab, full(st));
              filled |= 1u << st;
              fill_phase = (fill_phase & ~(1u << st)) | (phase << st);
            }
            if (++st == nst) { st = 0; phase ^= 1u; }
          }
      }
    producer_out:
      if (lane == 0)
        for (int q = 0; q < nst; ++q)
          if (filled & (1u << q)) mbar_wait_bounded(full(q), (fill_phase >> q) & 1u, timeout_ns);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers (warps 0..7)
  // Every consumer warp runs the same trip counts, so the named barriers always match; after a
  // failed wait (recorded in the status word) the warps skip the arithmetic and run to the end.
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ones[4] = {C::kOnePair, C::kOnePair, C::kOnePair, C::kOnePair};
  int st = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int e = sAct[u / nslab];
    const int slab = u % nslab;
    const int n0 = slab * NS;
    const float2* sm_e = sm + (size_t)e * KQ * NB + slab;  // block b's (scale, min) at sm_e[b * NB] (INT4)
    const int r_begin = offsets[e], r_end = offsets[e + 1];
    for (int rp = r_begin; rp < r_end; rp += kQRows) {
      const int R = min(kQRows, r_end - rp);
      // lane (g, t) feeds activation row g of the pass (column g of B); rows past R stay zero. Its
      // k-rows within a warp's range start at 16t (INT4) or 8t (INT8).
      const __nv_bfloat16* xrow = nullptr;
      if (g < R) xrow = a + (size_t)(a_rows != nullptr ? a_rows[rp + g] : rp + g) * K + (C::kWarpK / 4) * t;
      // the B fragments (and, INT4, the (scale, min) pair) of this warp's range of the box at k = kb
      auto fetch = [&](int kb, uint4& x0, uint4& x1, float2& q) {
        const int kw = kb + warp * C::kWarpK;
        x0 = make_uint4(0u, 0u, 0u, 0u);
        x1 = x0;
        q = make_float2(0.f, 0.f);
        if (kw < K) {
          if constexpr (!C::kScalesInSmem) q = sm_e[(size_t)(kw / QB) * NB];
          if (xrow != nullptr) {
            x0 = __ldg(reinterpret_cast<const uint4*>(xrow + kw));
            if constexpr (BITS == 4) x1 = __ldg(reinterpret_cast<const uint4*>(xrow + kw + 8));
          }
        }
      };
      float acc[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;
      float macc0 = 0.f, macc1 = 0.f;  // rows 2t and 2t + 1: sums of (min + centre scale) * (range sum of a)
      uint4 nx0, nx1;
      float2 nq;
      fetch(0, nx0, nx1, nq);
      for (int kb = 0; kb < K; kb += C::kBoxK) {
        const uint4 x0 = nx0, x1 = nx1;
        const float2 pq = nq;
        if (kb + C::kBoxK < K) fetch(kb + C::kBoxK, nx0, nx1, nq);  // in flight during this box
        if (ok) ok = wait_or_abort(full(st), phase, timeout_ns, abort_flag, status, 56);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && kb + warp * C::kWarpK < K) {
          // this warp's block (scale, min): copied with the box (INT8) or loaded a box ahead (INT4)
          const float2 q = C::kScalesInSmem ? sQ[st * kWarps + warp] : pq;
          const uint8_t* box = gring + st * kTmaBoxBytes + warp * C::kWarpSteps * C::kStepBytes + lane * 16;
          float blk[4][4], bs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) blk[m][i] = 0.f;
          if constexpr (BITS == 4) {
            const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 wd = *reinterpret_cast<const uint4*>(box + j * C::kStepBytes);
              const uint32_t words[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const uint32_t af[4] = {q4_pair(words[m], 0), q4_pair(words[m], 4), q4_pair(words[m], 8),
                                        q4_pair(words[m], 12)};
                mma_16816<4>(blk[m], af, xb[2 * j], xb[2 * j + 1]);
              }
              mma_16816<4>(bs, ones, xb[2 * j], xb[2 * j + 1]);  // bs[0], bs[1]: rows 2t, 2t+1
            }
          } else {
            const uint32_t xb[4] = {bf16x2_to_f16x2(x0.x), bf16x2_to_f16x2(x0.y), bf16x2_to_f16x2(x0.z),
                                    bf16x2_to_f16x2(x0.w)};
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
              // half 0: column tiles 0 and 1, half 1: tiles 2 and 3; a tile's 8 bytes in register order
              const uint4 h0 = *reinterpret_cast<const uint4*>(box + s2 * C::kStepBytes);
              const uint4 h1 = *reinterpret_cast<const uint4*>(box + s2 * C::kStepBytes + 512);
              const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const uint32_t af[4] = {q8_pair(w[2 * m], 0x5140u), q8_pair(w[2 * m], 0x5342u),
                                        q8_pair(w[2 * m + 1], 0x5140u), q8_pair(w[2 * m + 1], 0x5342u)};
                mma_16816<8>(blk[m], af, xb[2 * s2], xb[2 * s2 + 1]);
              }
              mma_16816<8>(bs, ones, xb[2 * s2], xb[2 * s2 + 1]);  // bs[0], bs[1]: rows 2t, 2t+1
            }
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][i] = fmaf(q.x, blk[m][i], acc[m][i]);
          const float mq = fmaf(C::kCentre, q.x, q.y);  // w = (min + centre scale) + (code - centre) scale
          macc0 = fmaf(mq, bs[0], macc0);
          macc1 = fmaf(mq, bs[1], macc1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(st));  // the box's slot goes back to the producer
        if (++st == nst) { st = 0; phase ^= 1u; }
      }
      // Warp sums to shared memory ([warp][row][column], and the block-minimum terms [warp][row]),
      // then every (row, column) adds the warps in a fixed order. acc[m]: columns 16m + g (0, 1) and
      // 16m + g + 8 (2, 3), rows 2t and 2t + 1.
      consumer_sync();  // the previous pass's sums have been read
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int c = 16 * m + g;
        if (2 * t < R) {
          sRed[(warp * kQRows + 2 * t) * NS + c] = acc[m][0];
          sRed[(warp * kQRows + 2 * t) * NS + c + 8] = acc[m][2];
        }
        if (2 * t + 1 < R) {
          sRed[(warp * kQRows + 2 * t + 1) * NS + c] = acc[m][1];
          sRed[(warp * kQRows + 2 * t + 1) * NS + c + 8] = acc[m][3];
        }
      }
      if (g == 0) {
        if (2 * t < R) sMinW[warp * kQRows + 2 * t] = macc0;
        if (2 * t + 1 < R) sMinW[warp * kQRows + 2 * t + 1] = macc1;
      }
      consumer_sync();
      for (int i = tid; i < R * NS; i += kThreads) {
        const int r = i / NS, c = i % NS;
        float v = 0.f, mt = 0.f;
#pragma unroll
        for (int wi = 0; wi < kWarps; ++wi) {
          v += sRed[(wi * kQRows + r) * NS + c];
          mt += sMinW[wi * kQRows + r];
        }
        v += mt;
        const int grow = rp + r;
        v = STAGE == 1 ? gelu_as(v) : row_gate[grow] * v;
        out[(size_t)grow * N + n0 + c] = from_f32<OutT>(v);
      }
    }
  }
}

#define MOE_STREAM_Q_PARAMS                                                                                   \
  const __grid_constant__ CUtensorMap tmC, const __nv_bfloat16* __restrict__ a,                               \
      const int32_t* __restrict__ a_rows, const float2* __restrict__ sm, const int32_t* __restrict__ offsets, \
      const float* __restrict__ row_gate, int K, int N, int E, int nst, OutT* __restrict__ out, int* status,  \
      uint64_t timeout_ns, int evict_first
template <int STAGE, typename OutT>
__global__ void __launch_bounds__(kTmaThreads, 2) ffn_stream_q4_kernel(MOE_STREAM_Q_PARAMS) {
  stream_q_body<4, STAGE, OutT>(&tmC, a, a_rows, sm, offsets, row_gate, K, N, E, nst, out, status, timeout_ns,
                                evict_first);
}
template <int STAGE, typename OutT>
__global__ void __launch_bounds__(kTmaThreads, 2) ffn_stream_q8_kernel(MOE_STREAM_Q_PARAMS) {
  stream_q_body<8, STAGE, OutT>(&tmC, a, a_rows, sm, offsets, row_gate, K, N, E, nst, out, status, timeout_ns,
                                evict_first);
}
#undef MOE_STREAM_Q_PARAMS

size_t q_smem_bytes(int nst, int E) {
  return 128 + (size_t)nst * kTmaBoxBytes + kBarSlotBytes + (size_t)kTmaStages * kWarps * sizeof(float2) +
         (size_t)kWarps * kQRows * (NS + 1) * sizeof(float) + (size_t)E * 4;
}

constexpr size_t kSmPerSmBytes = 228 * 1024;  // shared memory per SM, of which 1 KB per resident CTA is reserved

template <int BITS, int STAGE, typename OutT>
cudaError_t launch_q(const QFfnArgs& p, EncodeTiledFn enc, cudaStream_t s) {
  using C = QCodes<BITS>;
  int nst = kTmaStages;
  while (nst > 2 && 2 * (q_smem_bytes(nst, p.E) + 64 + 1024) > kSmPerSmBytes) --nst;
  const size_t smem = q_smem_bytes(nst, p.E);
  auto kern = BITS == 4 ? ffn_stream_q4_kernel<STAGE, OutT> : ffn_stream_q8_kernel<STAGE, OutT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // codes [E][N/64][K/16][step] viewed as [E * N/64][K/16][256] elements of 2 (INT4) or 4 (INT8)
  // bytes: kBoxSteps steps of one slab per box, no swizzle; steps past K/16 arrive as zeros
  CUtensorMap tmC;
  const cuuint64_t dims[3] = {256, (cuuint64_t)(p.K / 16), (cuuint64_t)p.E * (p.N / NS)};
  const cuuint64_t str[2] = {(cuuint64_t)C::kStepBytes, (cuuint64_t)(p.K / 16) * C::kStepBytes};
  const cuuint32_t box[3] = {256, (cuuint32_t)C::kBoxSteps, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&tmC, BITS == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 3,
          const_cast<void*>(p.codes), dims, str, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int nslab = p.N / NS;
  const long long max_units = (long long)(p.rows < p.E ? p.rows : p.E) * nslab;
  long long grid = 2LL * device_sm_count();  // persistent: the resident CTAs loop over the units
  if (grid > max_units) grid = max_units;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kTmaThreads), smem, s, tmC, (const __nv_bfloat16*)p.a,
                    p.a_rows, (const float2*)p.scale_min, p.offsets, p.row_gate, p.K, p.N, p.E, nst, (OutT*)p.out,
                    p.status, p.timeout_ns, (int)stream_evict_first(p.rows, p.E, p.K, p.N, BITS));
}

}  // namespace

cudaError_t launch_quantize(const void* w, int K, int N, int E, int dt, int bits, void* codes, float* scale_min,
                            cudaStream_t s) {
  const long long blocks = (long long)E * (K / QB) * (N / QB);
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks);
  if (dt == MOE_DTYPE_BF16) {
    if (bits == 4)
      quantize_kernel<__nv_bfloat16, 4><<<grid, 256, 0, s>>>((const __nv_bfloat16*)w, K, N, (uint4*)codes,
                                                             (float2*)scale_min);
    else
      quantize_kernel<__nv_bfloat16, 8><<<grid, 256, 0, s>>>((const __nv_bfloat16*)w, K, N, (uint4*)codes,
                                                             (float2*)scale_min);
  } else {
    if (bits == 4)
      quantize_kernel<float, 4><<<grid, 256, 0, s>>>((const float*)w, K, N, (uint4*)codes, (float2*)scale_min);
    else
      quantize_kernel<float, 8><<<grid, 256, 0, s>>>((const float*)w, K, N, (uint4*)codes, (float2*)scale_min);
  }
  return cudaGetLastError();
}

cudaError_t launch_ffn_stream_q(const QFfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  if (p.bits == 4)
    return p.stage == 1 ? launch_q<4, 1, __nv_bfloat16>(p, enc, s) : launch_q<4, 2, float>(p, enc, s);
  return p.stage == 1 ? launch_q<8, 1, __nv_bfloat16>(p, enc, s) : launch_q<8, 2, float>(p, enc, s);
}

}  // namespace moe
