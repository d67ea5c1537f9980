// Block quantisation of expert weights and the weight-streaming expert FFN that reads them.
// csdn/6a462500 §4.3 (64 x 64 blocks, each with its own min and max); csdn/6a919c0d §2.3 (decode
// is bound by moving expert weights, so fewer bytes per weight is the lever).
//
// Quantiser: per 64 x 64 block, scale = (max - min) / (2^bits - 1) and
// code = round((w - min) / scale), in fp32 with correctly rounded subtraction and division and
// rounding half to even, so the codes are a deterministic function of the weights; w is restored
// as min + code * scale (the page's dequantisation would lose the block minimum).
//
// Memory format of the codes of one [K, N] matrix. INT8: 16-byte tiles of 8 consecutive columns by 2
// consecutive k-rows, tiles row-major over (k / 2, n / 8); 64-bit half j holds k-row j, byte c is
// column c. Eight lanes reading one tile each cover a 64-column slab of 2 k-rows with one coalesced
// 128-byte request, and a tile never straddles a 64 x 64 block. INT4: the fragment layout of the
// tensor-core kernel, [N/64 slabs][K/16 k-blocks][32 lanes][4 words] (quantize_kernel describes
// the nibble order). Scales: one (scale, min) float pair per block, [K/64][N/64] per expert.
//
// INT8 streaming kernel: the structure of ffn_stream.cu (work unit = (expert with rows, 64-column
// slab), full depth per CTA, fixed-order reductions) with the dequantisation folded into the
// dot product: sum_k a_k (min_b + c_k scale_b) = sum_b [ (a scale_b) . (c - m) + (min_b + m scale_b) sum a ]
// with the centre m = 128.
// Per weight that is one byte permute into a 2^23-offset float, one subtraction (exact) and one
// FMA per activation row. The activations are staged already multiplied by their block's scale,
// and the column-independent term (min_b times the block's activation sum) is formed once per row
// from block sums taken while staging, not by every lane of the slab.
// INT4 streaming kernel (ffn_stream_q4_kernel): the same units and code stream, the dot products on
// mma.sync (see there).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int QB = 64;  // block edge
constexpr int kThreads = 256, kWarps = 8;  // consumer threads and warps (and the quantiser's)
constexpr int NS = 64;              // columns per slab (one block column)
constexpr int LPR = NS / 8;         // lanes per tile row: 8
constexpr int RPW = 32 / LPR;       // tile rows per warp per step: 4
constexpr int GSTEP = kWarps * RPW; // tile rows per CTA step: 32
constexpr float kMagic = 8388608.0f;  // 2^23: a byte b placed in the low mantissa bits reads 2^23 + b

// ------------------------------------------------------------------ quantiser
template <typename T, int BITS>
__global__ void __launch_bounds__(256)
quantize_kernel(const T* __restrict__ w, int K, int N, uint4* __restrict__ codes, float2* __restrict__ sm) {
  constexpr int KT = 16 / BITS;  // k-rows per tile: 128 bits / (8 columns x BITS)
  static_assert(KT * 8 * BITS == 128, "a tile is 16 bytes");
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
  if (BITS == 4) {
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
    return;
  }
  constexpr int tiles = (QB / KT) * (QB / 8);  // 256 (INT8)
  for (int t = tid; t < tiles; t += 256) {
    const int kgl = t / (QB / 8), ngl = t % (QB / 8);
    uint32_t word[4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) v |= code(kgl * KT + j, ngl * 8 + 4 * h + c) << (8 * c);
        word[2 * j + h] = v;
      }
    const size_t kg = (size_t)bi * (QB / KT) + kgl, ng = (size_t)bj * (QB / 8) + ngl;
    codes[((size_t)e * (K / KT) + kg) * (N / 8) + ng] = make_uint4(word[0], word[1], word[2], word[3]);
  }
}

// ------------------------------------------------------------------ streaming FFN
// Codes of the 8 columns of one k-row as exact centred floats c - 2^(bits-1) (-8 .. 7 for INT4,
// -128 .. 127 for INT8), in column pairs (2p, 2p+1) packed for the fp32x2 instructions: a byte
// permute places each code in the low mantissa bits of 2^23, one packed subtraction of
// 2^23 + 2^(bits-1) (exact) leaves the centred code. Centring halves the scaled term that the
// block-minimum term otherwise cancels in part, and with it the term's rounding error.
template <int BITS>
constexpr float kCentre = (float)(1 << (BITS - 1));
__device__ __forceinline__ uint32_t magic_byte(uint32_t w, uint32_t sel) { return __byte_perm(w, 0x4B000000u, sel); }
__device__ __forceinline__ void int8_row(uint32_t w0, uint32_t w1, uint64_t (&c)[4]) {
  const uint64_t neg = f2_pack(-(kMagic + kCentre<8>), -(kMagic + kCentre<8>));
  c[0] = fadd2(((uint64_t)magic_byte(w0, 0x7541) << 32) | magic_byte(w0, 0x7540), neg);
  c[1] = fadd2(((uint64_t)magic_byte(w0, 0x7543) << 32) | magic_byte(w0, 0x7542), neg);
  c[2] = fadd2(((uint64_t)magic_byte(w1, 0x7541) << 32) | magic_byte(w1, 0x7540), neg);
  c[3] = fadd2(((uint64_t)magic_byte(w1, 0x7543) << 32) | magic_byte(w1, 0x7542), neg);
}

// Rows rp .. rp+R-1, k-range [kc, kc+kn) of the bf16 activations -> sA as fp32 (row stride KC),
// each multiplied by its block's scale (the same for every lane of the slab, so done once here
// instead of by each of the eight lanes that share a k-row); sBS[r][b] receives the plain sum of the
// row's 64 activations of block b (eight 8-value partials of consecutive lanes, added as a fixed
// xor tree), for the block-minimum term. 16-byte loads (K and kn are multiples of 64, rows 16-byte
// aligned); every lane of a warp runs the same number of iterations (R * KC / 8 is a multiple of the
// block size).
template <int KC>
__device__ __forceinline__ void stage_rows_q(const __nv_bfloat16* __restrict__ a, const int32_t* __restrict__ a_rows,
                                             int K, int rp, int R, int kc, int kn, const float2* sSM, float* sA,
                                             float* sBS) {
  const int per_row = KC / 8;
  for (int i = threadIdx.x; i < R * per_row; i += kThreads) {
    const int r = i / per_row, kk = (i % per_row) * 8;
    const size_t src = a_rows != nullptr ? (size_t)a_rows[rp + r] : (size_t)(rp + r);
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (kk < kn) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(a + src * K + kc + kk));
      v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
      v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
    }
    const float sc = kk < kn ? sSM[(kc + kk) / QB].x : 0.f;
    float4* dst = reinterpret_cast<float4*>(sA + r * KC + kk);
    dst[0] = make_float4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
    dst[1] = make_float4(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
    float s8 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s8 += v[j];
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) s8 += __shfl_xor_sync(0xffffffffu, s8, o);
    if ((threadIdx.x & 7) == 0) sBS[r * (KC / QB) + kk / QB] = s8;
  }
}

// Activations of rows rp .. rp+R-1 (through a_rows when given), k-range [kc, kc+kn), in two steps so
// that the loads can be issued well before they are needed: load_rows_q fetches them into registers
// (16-byte loads; K and kn are multiples of 64, rows 16-byte aligned), and store_rows_q writes them
// to sA as fp32 (row stride KC), each multiplied by its block's scale (the same for every lane of
// the slab, so done once here instead of by each of the eight lanes that share a k-row), with
// sBS[r][b] = the plain sum of row r's 64 activations of block b (eight 8-value partials of
// consecutive lanes, added as a fixed xor tree), for the block-minimum term. Thread i of the
// consumers holds the 8-value groups i, i + kThreads, ...; a row's KC / 8 groups are a multiple of
// the warp size, so every lane of a warp takes the same branches.
template <int KC, int NIT>
__device__ __forceinline__ void load_rows_q(const __nv_bfloat16* __restrict__ a, const int32_t* __restrict__ a_rows,
                                            int K, int rp, int R, int kc, int kn, uint4 (&xv)[NIT]) {
  constexpr int per_row = KC / 8;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int i = threadIdx.x + it * kThreads;
    const int r = i / per_row, kk = (i % per_row) * 8;
    xv[it] = make_uint4(0u, 0u, 0u, 0u);
    if (r < R && kk < kn) {
      const size_t src = a_rows != nullptr ? (size_t)a_rows[rp + r] : (size_t)(rp + r);
      xv[it] = __ldg(reinterpret_cast<const uint4*>(a + src * K + kc + kk));
    }
  }
}
template <int KC, int NIT>
__device__ __forceinline__ void store_rows_q(const uint4 (&xv)[NIT], int R, int kc, int kn, const float2* sSM,
                                             float* sA, float* sBS) {
  constexpr int per_row = KC / 8;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int i = threadIdx.x + it * kThreads;
    const int r = i / per_row, kk = (i % per_row) * 8;
    if (r >= R) continue;  // warp-uniform
    const uint4 u = xv[it];
    const float v[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                        bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
    const float sc = kk < kn ? sSM[(kc + kk) / QB].x : 0.f;
    float4* dst = reinterpret_cast<float4*>(sA + r * KC + kk);
    dst[0] = make_float4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
    dst[1] = make_float4(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
    float s8 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s8 += v[j];
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) s8 += __shfl_xor_sync(0xffffffffu, s8, o);
    if ((threadIdx.x & 7) == 0) sBS[r * (KC / QB) + kk / QB] = s8;
  }
}

constexpr int kTmaTileRows = 128;                      // tile rows per box (128 x KT k-rows)
constexpr int kTmaBoxBytes = kTmaTileRows * LPR * 16;  // 16 KB: 8 tiles (64 columns) per tile row
constexpr int kTmaStages = 5;                          // boxes in flight per CTA
constexpr int kTmaThreads = kThreads + 32;             // 8 consumer warps + the producer warp
constexpr int kTmaActFloats = 4096;                    // staged activations: RMAX rows x 4096/RMAX
constexpr int kBarSlotBytes = 128;                     // the ring's mbarriers: 2 x kTmaStages x 8 bytes
static_assert(2 * kTmaStages * 8 <= kBarSlotBytes, "the mbarriers fit their slot");

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// The code stream arrives by TMA: one producer warp keeps a ring of 16 KB boxes (the 8 tiles of a
// 64-column slab for 128 consecutive tile rows of one expert) in flight, two CTAs per SM, and the
// eight consumer warps read the tiles from shared memory, one 16-byte tile per lane, and release
// each box. The activations, the slab's (scale, min) pairs and the block sums are staged between
// named barriers of the consumer warps only, so the code stream never waits for them.
template <int BITS, int STAGE, typename OutT, int RMAX>
__global__ void __launch_bounds__(kTmaThreads, 2)
ffn_stream_q_kernel(const __grid_constant__ CUtensorMap tmC, const __nv_bfloat16* __restrict__ a,
                    const int32_t* __restrict__ a_rows, const float2* __restrict__ sm,
                    const int32_t* __restrict__ offsets, const float* __restrict__ row_gate, int K, int N, int E,
                    int nst, OutT* __restrict__ out, int* status, uint64_t timeout_ns) {
  constexpr int KT = 16 / BITS;  // k-rows per tile: 128 bits / (8 columns x BITS)
  static_assert(BITS == 8 && KT == 2, "the tile kernel streams INT8 codes (INT4: ffn_stream_q4_kernel)");
  constexpr int KC = kTmaActFloats / RMAX;  // a multiple of the k-rows of a box (128 KT)
  static_assert(KC % (kTmaTileRows * KT) == 0, "a chunk holds whole boxes");
  constexpr int kSets = RMAX == 2 ? 2 : 1;  // accumulator sets
  constexpr int kXIt = RMAX * KC / 8 / kThreads;  // 16-byte activation loads per consumer thread per chunk
  constexpr bool kPrefetch = RMAX == 2;          // the next chunk's activations in flight during the boxes
  static_assert(kXIt * kThreads * 8 == RMAX * KC && (KC / 8) % 32 == 0, "whole warps per activation row");
  static_assert(RMAX <= kWarps, "one warp per row forms the block-minimum terms");
  extern __shared__ uint8_t smem_raw[];
  // ring [nst][128 tile rows][8 tiles] (128-byte aligned) | full [nst], empty [nst] mbarriers in
  // a 128-byte slot | sA [RMAX][KC] (the epilogue's per-warp sums reuse it) | sSM [K/64]
  // | sBS [RMAX][KC/64] | sMin [RMAX] | sAct [E]
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 127u) & ~127u;
  uint8_t* gring = smem_raw + (ring - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gring + nst * kTmaBoxBytes);
  float* sA = reinterpret_cast<float*>(gring + nst * kTmaBoxBytes + kBarSlotBytes);
  float* sRed = sA;  // [kWarps][RMAX][NS]
  float2* sSM = reinterpret_cast<float2*>(sA + RMAX * KC);
  float* sBS = reinterpret_cast<float*>(sSM + K / QB);
  float* sMin = sBS + RMAX * (KC / QB);
  int* sAct = reinterpret_cast<int*>(sMin + RMAX);
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
    tma_prefetch_desc(&tmC);
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
  const int KG = K / KT;                                   // tile rows of a matrix
  const int KB = (KG + kTmaTileRows - 1) / kTmaTileRows;  // boxes per pass; rows past KG arrive as zeros

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int st = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int e = sAct[u / nslab], slab = u % nslab;
        const int passes = (offsets[e + 1] - offsets[e] + RMAX - 1) / RMAX;
        for (int ps = 0; ps < passes; ++ps)
          for (int kb = 0; kb < KB; ++kb) {
            if (!wait_or_abort(empty(st), phase ^ 1u, timeout_ns, abort_flag, status, 53)) goto producer_out;
            mbar_arrive_expect_tx(full(st), kTmaBoxBytes);
            tma_load_3d(ring + st * kTmaBoxBytes, &tmC, slab * NS, kb * kTmaTileRows, e, full(st));
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
  const int kr = lane / LPR;  // tile row of this lane within the warp's group of RPW
  const int cg = lane % LPR;  // 8-column group of this lane
  const int NB = N / QB;
  int st = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int e = sAct[u / nslab];
    const int slab = u % nslab;
    const int n0 = slab * NS;
    if (!kPrefetch) {
      consumer_sync();  // the previous unit is done with sSM
      for (int b = tid; b < K / QB; b += kThreads) sSM[b] = sm[((size_t)e * (K / QB) + b) * NB + slab];
    }
    const int r_begin = offsets[e], r_end = offsets[e + 1];
    for (int rp = r_begin; rp < r_end; rp += RMAX) {
      const int R = min(RMAX, r_end - rp);
      // column pairs (2p, 2p+1) of each row; with two rows a pass, even and odd k-rows of a tile go
      // to separate sets, for twice the independent FMA chains (3% faster at 8 tokens; no faster
      // with one or four rows a pass)
      uint64_t acc2[kSets][RMAX][4];
#pragma unroll
      for (int h = 0; h < kSets; ++h)
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc2[h][r][q] = 0ull;
      float min_term = 0.f;  // warp r < R: row r's sum over blocks of (min_b + m scale_b) * (sum of a over b)
      // With two rows a pass, the pass's first chunk of activations is loaded together with (on a
      // new unit) the slab's scale pairs, which the previous unit stopped reading before its
      // epilogue's barriers, and each later chunk while the boxes of the one before are consumed:
      // 10% faster at 8 tokens. With one row a pass the same made one token 9% slower, and with
      // four the registers run short, so there each chunk is loaded and staged between barriers.
      uint4 xv[kPrefetch ? kXIt : 1];
      if (kPrefetch) {
        load_rows_q<KC>(a, a_rows, K, rp, R, 0, min(KC, K), xv);
        if (rp == r_begin)
          for (int b = tid; b < K / QB; b += kThreads) sSM[b] = sm[((size_t)e * (K / QB) + b) * NB + slab];
      }
      for (int kc = 0; kc < K; kc += KC) {
        const int kn = min(KC, K - kc);  // a multiple of 64
        consumer_sync();  // sSM is written; the previous chunk's activations (or sums) are read
        if (kPrefetch) store_rows_q<KC>(xv, R, kc, kn, sSM, sA, sBS);
        else stage_rows_q<KC>(a, a_rows, K, rp, R, kc, kn, sSM, sA, sBS);
        consumer_sync();
        if (kPrefetch && kc + KC < K) load_rows_q<KC>(a, a_rows, K, rp, R, kc + KC, min(KC, K - kc - KC), xv);
        // w = (min + centre * scale) + (c - centre) * scale: warp r adds row r's block terms of this
        // chunk (lanes strided over the blocks, then a fixed xor tree; every lane ends with the sum)
        if (warp < R) {
          float p = 0.f;
          for (int b = lane; b < kn / QB; b += 32) {
            const float2 q = sSM[kc / QB + b];
            p = fmaf(fmaf(kCentre<BITS>, q.x, q.y), sBS[warp * (KC / QB) + b], p);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
          min_term += p;
        }
        for (int kb = 0; kb < kn; kb += kTmaTileRows * KT) {
          if (ok) ok = wait_or_abort(full(st), phase, timeout_ns, abort_flag, status, 54);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            const uint8_t* box = gring + st * kTmaBoxBytes;
#pragma unroll
            for (int i = 0; i < kTmaTileRows / GSTEP; ++i) {
              const int g = i * GSTEP + warp * RPW + kr;  // tile row within the box
              const uint4 t = *reinterpret_cast<const uint4*>(box + g * (LPR * 16) + cg * 16);
              const uint32_t wd[4] = {t.x, t.y, t.z, t.w};
              const int k0 = kb + g * KT;  // first k-row of the tile within the chunk
#pragma unroll
              for (int j = 0; j < KT; ++j) {
                uint64_t cp[4];
                int8_row(wd[2 * j], wd[2 * j + 1], cp);
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                  if (r >= R) break;
                  const float as = sA[r * KC + k0 + j];  // activation times its block's scale
                  const uint64_t as2 = f2_pack(as, as);
#pragma unroll
                  for (int q = 0; q < 4; ++q) acc2[j % kSets][r][q] = ffma2(as2, cp[q], acc2[j % kSets][r][q]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty(st));  // the box's slot goes back to the producer
          if (++st == nst) { st = 0; phase ^= 1u; }
        }
      }
      // Combine the warp's RPW tile rows (lanes cg, cg+8, cg+16, cg+24) and the warps in fixed
      // orders, then add each row's column-independent block-minimum term.
      float acc[RMAX][8];
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float v = 0.f;
#pragma unroll
          for (int h = 0; h < kSets; ++h) v += c & 1 ? f2_hi(acc2[h][r][c >> 1]) : f2_lo(acc2[h][r][c >> 1]);
          v += __shfl_xor_sync(0xffffffffu, v, LPR);
          v += __shfl_xor_sync(0xffffffffu, v, 2 * LPR);
          acc[r][c] = v;
        }
      consumer_sync();  // sRed overlays the activations
      if (lane == 0 && warp < R) sMin[warp] = min_term;
      if (lane < LPR) {
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int c = 0; c < 8; ++c) sRed[(warp * RMAX + r) * NS + cg * 8 + c] = acc[r][c];
      }
      consumer_sync();
      for (int i = tid; i < R * NS; i += kThreads) {
        const int r = i / NS, c = i % NS;
        float v = 0.f;
#pragma unroll
        for (int wi = 0; wi < kWarps; ++wi) v += sRed[(wi * RMAX + r) * NS + c];
        v += sMin[r];
        const int grow = rp + r;
        v = STAGE == 1 ? gelu_as(v) : row_gate[grow] * v;
        out[(size_t)grow * N + n0 + c] = from_f32<OutT>(v);
      }
    }
  }
}

// ------------------------------------------------------------------ INT4 on the tensor cores
// The INT4 codes of a 64-column slab arrive by TMA like the tiles above (boxes of 16 KB: 32 k-blocks
// of 16 k-rows, 512 bytes each, in the fragment layout the quantiser writes), and the dot products
// run on mma.sync m16n8k16 (bf16 in, fp32 accumulate): A = 16 weight columns x 16 k-rows, decoded from
// one 32-bit word per lane, B = 16 k-rows x 8 activation rows (tokens), so one instruction does 2048
// multiply-adds and a pass takes up to 8 rows at the cost of one. Decoding a register pair is one
// shift and one LOP3 that puts two nibbles n into the low mantissa bits of bf16 128.0 (128 + n,
// exact), and one packed bf16 subtraction of 136 that leaves the centred code n - 8 (exact).
// Each warp takes one 64-deep k-block of every box. Within a block the code layout numbers k so that
// the B fragments of lane 4g + t for all four 16-deep steps are the 16 consecutive k-rows 16t .. 16t+15
// of activation row g: the lane loads them from global memory (two 16-byte loads, one box ahead of
// use) and no activation is staged in shared memory. The products of a block share one (scale, min)
// pair: they accumulate in a block accumulator that is scaled and added once per block. The
// column-independent term (min + 8 scale) * (sum of the block's activations) takes one more MMA per
// step, with an A fragment of ones, whose result is each row's sum over the step's k-rows.
constexpr int kQ4Rows = 8;                     // activation rows per pass: the MMA's N
constexpr int kQ4BoxK16 = kTmaBoxBytes / 512;  // 16-deep k-blocks per box: 32 (512 k-rows)
constexpr uint32_t kBf16OnePair = 0x3F803F80u;  // bf16 1.0 in both halves

__device__ __forceinline__ uint32_t q4_pair(uint32_t word, int shift) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(word >> shift), "r"(0x000F000Fu), "r"(0x43004300u));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(0x43084308u));  // (128 + n) - 136 = n - 8, exact
  return r;
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int STAGE, typename OutT>
__global__ void __launch_bounds__(kTmaThreads, 2)
ffn_stream_q4_kernel(const __grid_constant__ CUtensorMap tmC, const __nv_bfloat16* __restrict__ a,
                     const int32_t* __restrict__ a_rows, const float2* __restrict__ sm,
                     const int32_t* __restrict__ offsets, const float* __restrict__ row_gate, int K, int N, int E,
                     int nst, OutT* __restrict__ out, int* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  // ring [nst][16 KB] (128-byte aligned) | full [nst], empty [nst] mbarriers in a 128-byte slot |
  // sRed [kWarps][kQ4Rows][NS] (warp sums) | sMinW [kWarps][kQ4Rows] (warp block-minimum terms) | sAct [E]
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 127u) & ~127u;
  uint8_t* gring = smem_raw + (ring - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gring + nst * kTmaBoxBytes);
  float* sRed = reinterpret_cast<float*>(gring + nst * kTmaBoxBytes + kBarSlotBytes);
  float* sMinW = sRed + kWarps * kQ4Rows * NS;
  int* sAct = reinterpret_cast<int*>(sMinW + kWarps * kQ4Rows);
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
    tma_prefetch_desc(&tmC);
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
  const int KB = (K16 + kQ4BoxK16 - 1) / kQ4BoxK16;  // boxes per pass; k-blocks past K arrive as zeros

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int st = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int e = sAct[u / nslab], slab = u % nslab;
        const int passes = (offsets[e + 1] - offsets[e] + kQ4Rows - 1) / kQ4Rows;
        for (int ps = 0; ps < passes; ++ps)
          for (int kb = 0; kb < KB; ++kb) {
            if (!wait_or_abort(empty(st), phase ^ 1u, timeout_ns, abort_flag, status, 55)) goto producer_out;
            mbar_arrive_expect_tx(full(st), kTmaBoxBytes);
            tma_load_3d(ring + st * kTmaBoxBytes, &tmC, 0, kb * kQ4BoxK16, e * nslab + slab, full(st));
            filled |= 1u << st;
            fill_phase = (fill_phase & ~(1u << st)) | (phase << st);
            if (++st == nst) { st = 0; phase ^= 1u; }
          }
      }
    producer_out:
      for (int q = 0; q < nst; ++q)
        if (filled & (1u << q)) mbar_wait_bounded(full(q), (fill_phase >> q) & 1u, timeout_ns);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers (warps 0..7)
  // Every consumer warp runs the same trip counts, so the named barriers always match; after a
  // failed wait (recorded in the status word) the warps skip the arithmetic and run to the end.
  const int g = lane >> 2, t = lane & 3;
  const int NB = N / QB, KQ = K / QB;
  const uint32_t ones[4] = {kBf16OnePair, kBf16OnePair, kBf16OnePair, kBf16OnePair};
  int st = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int e = sAct[u / nslab];
    const int slab = u % nslab;
    const int n0 = slab * NS;
    const float2* sm_e = sm + (size_t)e * KQ * NB + slab;  // block b's (scale, min) at sm_e[b * NB]
    const int r_begin = offsets[e], r_end = offsets[e + 1];
    for (int rp = r_begin; rp < r_end; rp += kQ4Rows) {
      const int R = min(kQ4Rows, r_end - rp);
      // lane (g, t) feeds activation row g of the pass (column g of B); rows past R stay zero
      const __nv_bfloat16* xrow = nullptr;
      if (g < R) xrow = a + (size_t)(a_rows != nullptr ? a_rows[rp + g] : rp + g) * K + 16 * t;
      // the B fragments and the (scale, min) pair of this warp's block of the box at k = kb
      auto fetch = [&](int kb, uint4& x0, uint4& x1, float2& q) {
        const int kw = kb + warp * QB;
        x0 = make_uint4(0u, 0u, 0u, 0u);
        x1 = x0;
        q = make_float2(0.f, 0.f);
        if (kw < K) {
          q = sm_e[(size_t)(kw / QB) * NB];
          if (xrow != nullptr) {
            x0 = __ldg(reinterpret_cast<const uint4*>(xrow + kw));
            x1 = __ldg(reinterpret_cast<const uint4*>(xrow + kw + 8));
          }
        }
      };
      float acc[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;
      float macc0 = 0.f, macc1 = 0.f;  // rows 2t and 2t + 1: sums of (min + 8 scale) * (block sum of a)
      uint4 nx0, nx1;
      float2 nq;
      fetch(0, nx0, nx1, nq);
      for (int kb = 0; kb < K; kb += kQ4BoxK16 * 16) {
        const uint4 x0 = nx0, x1 = nx1;
        const float2 q = nq;
        if (kb + kQ4BoxK16 * 16 < K) fetch(kb + kQ4BoxK16 * 16, nx0, nx1, nq);  // in flight during this box
        if (ok) ok = wait_or_abort(full(st), phase, timeout_ns, abort_flag, status, 56);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && kb + warp * QB < K) {
          const uint8_t* box = gring + st * kTmaBoxBytes + warp * 4 * 512 + lane * 16;
          const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          float blk[4][4], bs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) blk[m][i] = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 wd = *reinterpret_cast<const uint4*>(box + j * 512);
            const uint32_t words[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const uint32_t af[4] = {q4_pair(words[m], 0), q4_pair(words[m], 4), q4_pair(words[m], 8),
                                      q4_pair(words[m], 12)};
              mma_bf16_16816(blk[m], af, xb[2 * j], xb[2 * j + 1]);
            }
            mma_bf16_16816(bs, ones, xb[2 * j], xb[2 * j + 1]);  // bs[0], bs[1]: rows 2t, 2t+1
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][i] = fmaf(q.x, blk[m][i], acc[m][i]);
          const float mq = fmaf(8.0f, q.x, q.y);  // w = (min + 8 scale) + (code - 8) scale
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
          sRed[(warp * kQ4Rows + 2 * t) * NS + c] = acc[m][0];
          sRed[(warp * kQ4Rows + 2 * t) * NS + c + 8] = acc[m][2];
        }
        if (2 * t + 1 < R) {
          sRed[(warp * kQ4Rows + 2 * t + 1) * NS + c] = acc[m][1];
          sRed[(warp * kQ4Rows + 2 * t + 1) * NS + c + 8] = acc[m][3];
        }
      }
      if (g == 0) {
        if (2 * t < R) sMinW[warp * kQ4Rows + 2 * t] = macc0;
        if (2 * t + 1 < R) sMinW[warp * kQ4Rows + 2 * t + 1] = macc1;
      }
      consumer_sync();
      for (int i = tid; i < R * NS; i += kThreads) {
        const int r = i / NS, c = i % NS;
        float v = 0.f, mt = 0.f;
#pragma unroll
        for (int wi = 0; wi < kWarps; ++wi) {
          v += sRed[(wi * kQ4Rows + r) * NS + c];
          mt += sMinW[wi * kQ4Rows + r];
        }
        v += mt;
        const int grow = rp + r;
        v = STAGE == 1 ? gelu_as(v) : row_gate[grow] * v;
        out[(size_t)grow * N + n0 + c] = from_f32<OutT>(v);
      }
    }
  }
}

size_t q4_smem_bytes(int nst, int E) {
  return 128 + (size_t)nst * kTmaBoxBytes + kBarSlotBytes + (size_t)kWarps * kQ4Rows * (NS + 1) * sizeof(float) +
         (size_t)E * 4;
}

constexpr size_t kSmPerSmBytes = 228 * 1024;  // shared memory per SM, of which 1 KB per resident CTA is reserved

template <int STAGE, typename OutT>
cudaError_t launch_q4(const QFfnArgs& p, EncodeTiledFn enc, cudaStream_t s) {
  int nst = kTmaStages;
  while (nst > 2 && 2 * (q4_smem_bytes(nst, p.E) + 64 + 1024) > kSmPerSmBytes) --nst;
  const size_t smem = q4_smem_bytes(nst, p.E);
  auto kern = ffn_stream_q4_kernel<STAGE, OutT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // codes [E][N/64][K/16][512 bytes] viewed as [E * N/64][K/16][256] 16-bit elements: 32 k-blocks of one
  // slab per box, no swizzle; k-blocks past K/16 arrive as zeros
  CUtensorMap tmC;
  const cuuint64_t dims[3] = {256, (cuuint64_t)(p.K / 16), (cuuint64_t)p.E * (p.N / NS)};
  const cuuint64_t str[2] = {512, (cuuint64_t)(p.K / 16) * 512};
  const cuuint32_t box[3] = {256, kQ4BoxK16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(p.codes), dims, str, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int nslab = p.N / NS;
  const long long max_units = (long long)(p.rows < p.E ? p.rows : p.E) * nslab;
  long long grid = 2LL * device_sm_count();
  if (grid > max_units) grid = max_units;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kTmaThreads), smem, s, tmC, (const __nv_bfloat16*)p.a,
                    p.a_rows, (const float2*)p.scale_min, p.offsets, p.row_gate, p.K, p.N, p.E, nst, (OutT*)p.out,
                    p.status, p.timeout_ns);
}

size_t q_smem_bytes(int RMAX, int nst, int K, int E) {
  const int KC = kTmaActFloats / RMAX;
  return 128 + (size_t)nst * kTmaBoxBytes + kBarSlotBytes + (size_t)kTmaActFloats * sizeof(float) +
         (size_t)(K / QB) * sizeof(float2) + (size_t)(RMAX * (KC / QB) + RMAX) * sizeof(float) + (size_t)E * 4;
}

template <int BITS, int STAGE, typename OutT, int RMAX>
cudaError_t launch_q(const QFfnArgs& p, EncodeTiledFn enc, cudaStream_t s) {
  // five boxes deep, fewer where a large K or E leaves no room for two CTAs per SM
  int nst = kTmaStages;
  while (nst > 2 && 2 * (q_smem_bytes(RMAX, nst, p.K, p.E) + 1024) > kSmPerSmBytes) --nst;
  const size_t smem = q_smem_bytes(RMAX, nst, p.K, p.E);
  auto kern = ffn_stream_q_kernel<BITS, STAGE, OutT, RMAX>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // codes [E][K/KT][N/8] 16-byte tiles viewed as [E][K/KT][N] 16-bit elements: 128 tile rows of a
  // 64-column slab per box, no swizzle, no L2 promotion; tile rows past K/KT arrive as zeros
  constexpr int KT = 16 / BITS;
  CUtensorMap tmC;
  const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)(p.K / KT), (cuuint64_t)p.E};
  const cuuint64_t str[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)(p.K / KT) * p.N * 2};
  const cuuint32_t box[3] = {NS, kTmaTileRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(p.codes), dims, str, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int nslab = p.N / NS;
  const long long max_units = (long long)(p.rows < p.E ? p.rows : p.E) * nslab;
  long long grid = 2LL * device_sm_count();  // persistent: the resident CTAs loop over the units
  if (grid > max_units) grid = max_units;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kTmaThreads), smem, s, tmC, (const __nv_bfloat16*)p.a,
                    p.a_rows, (const float2*)p.scale_min, p.offsets, p.row_gate, p.K, p.N, p.E, nst, (OutT*)p.out,
                    p.status, p.timeout_ns);
}

template <int BITS>  // INT8 (the INT4 codes take launch_q4)
cudaError_t launch_q_bits(const QFfnArgs& p, EncodeTiledFn enc, cudaStream_t s) {
  if (p.max_rows_per_expert == 1)  // a single token: one row per expert
    return p.stage == 1 ? launch_q<BITS, 1, __nv_bfloat16, 1>(p, enc, s) : launch_q<BITS, 2, float, 1>(p, enc, s);
  // Four rows a pass only when the experts average three or more (the host assumes an even spread):
  // the two-row kernel, which loads its activations ahead, was 12-15% faster at 64 tokens over 128
  // experts, where the touched experts hold 1.5 rows on average.
  if (p.rows <= 32 || (long long)p.rows < 3LL * p.E)
    return p.stage == 1 ? launch_q<BITS, 1, __nv_bfloat16, 2>(p, enc, s) : launch_q<BITS, 2, float, 2>(p, enc, s);
  return p.stage == 1 ? launch_q<BITS, 1, __nv_bfloat16, 4>(p, enc, s) : launch_q<BITS, 2, float, 4>(p, enc, s);
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
    return p.stage == 1 ? launch_q4<1, __nv_bfloat16>(p, enc, s) : launch_q4<2, float>(p, enc, s);
  return launch_q_bits<8>(p, enc, s);
}

}  // namespace moe
