// Grouped expert GEMM on CTA pairs with the product transposed: D^T = W^T x^T.
// Same math and epilogues as ffn_tc.cu (csdn/6a462027 §3.2 and §4.2 step 6; gate:
// csdn/6a919c0d §2.2 step 4):
//   up   (stage 1): h[r]      = GeLU(x_perm[r] W1[e])            (bf16 out)
//   down (stage 2): y_perm[r] = row_gate[r] * (h[r] W2[e])        (fp32 out)
//
// Why transposed: an expert's routed rows are a ragged count, the output features are not
// (d_ff and d are multiples of 256 in every workload). With the features on the MMA's M side
// (256 per CTA pair, 128 per CTA, from the weights stored N-contiguous: an MN-major A operand)
// and the rows on its N side (K-major B operand from x_perm), a tile covers up to 256 rows and
// its N is the row count rounded up to 16. An expert's last tile therefore wastes at most 15
// rows, where a 256-row M tile wastes up to 255. Per CTA and 64-deep k-block the loads are
// 16 KB of weights + 16 KB of rows (32 KB, against 48 KB for one-CTA 128x256 tiles), so six or
// seven stages fit in shared memory.
//
// Roles (both CTAs run 18 warps):
//   warp 0      TMA producer of this CTA's halves (128 features of W, up to 128 rows of x);
//               the loads complete on the leader CTA's "full" barrier
//   warp 1      TMEM allocation for the pair; in the leader also the MMA issuer
//               (tcgen05.mma.cta_group::2, M = 256, N = rows of the tile)
//   warps 2..17 epilogue: TMEM lane = output feature, TMEM column = row; warp w reads lane
//               quarter w mod 4 (32 features) and a quarter of the tile's rows, 32 rows a step.
//               Up: GeLU, bf16, a [32 rows][32 features] tile in shared memory, one TMA store;
//               down: gate, fp32, 32 consecutive features of a row per store instruction. Then
//               an arrival on the leader's "accumulator empty". Sixteen warps (four per
//               scheduler) hide the GeLU's dependent MUFU/FMA chains, which eight did not.
// All waits are bounded; on a timeout the CTA records MOE_ERR_DEVICE_TIMEOUT and unwinds.
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BF = 256;                           // features per pair tile (MMA M)
constexpr int BR = 256;                           // rows per tile at most (MMA N)
constexpr int BK = 64;                            // k per MMA-operand block (one 128-byte swizzle row)
// A pipeline stage holds KSUB consecutive k-blocks (1 or 2) of both operands.
template <int KSUB> constexpr int kTileASubBytes = KSUB * BK * 64 * 2;  // one 64-feature atom: 8 / 16 KB
template <int KSUB> constexpr int kTileABytes = 2 * kTileASubBytes<KSUB>;  // this CTA's 128 features
template <int KSUB> constexpr int kTileBBytes = KSUB * (BR / 2) * BK * 2;  // up to 128 rows of this CTA's half
template <int KSUB> constexpr int kStageBytes = kTileABytes<KSUB> + kTileBBytes<KSUB>;
constexpr int kEpiWarps = 16;                     // four per TMEM lane quarter: enough warps to hide
constexpr int kThreads = 64 + 32 * kEpiWarps;     // the GeLU's dependent chains and the TMEM loads
constexpr int kSegRows = BR * 4 / kEpiWarps;      // rows of a tile per epilogue warp: 64
constexpr int CR = 32;                            // rows per epilogue step (one tcgen05.ld x32)
constexpr int kStgBytes = CR * 32 * 2;            // per epilogue warp (up): 32 rows x 32 bf16 features
constexpr uint32_t kTmemCols = 2 * BR;            // two accumulators of up to 256 columns
constexpr int kMaxSmem = 232448;
// The rows operand comes in boxes sized to the item: a CTA's half of an item of nt rows (nt / 2, a
// multiple of 8) is copied by the smallest box of 16, 32, ..., 128 rows that covers it, one tensor
// map per height. Fewer bytes per stage for the light experts' items (about 84 rows on skew_e128):
// skew_e128 up 2000-2009 -> 1960 us, down 1983-2006 -> 1952 us; e16 and prefill unchanged.
constexpr int kBoxMaps = BR / 2 / 16;
struct BoxMaps {
  CUtensorMap m[kBoxMaps];
};
__host__ __device__ constexpr int box_rows_for(int nt) { return ((nt / 2 + 15) / 16) * 16; }
// Row tiles per band of a heavy expert's down-projection items. The down-projection's rows (h, 4 MB
// per row tile at d_ff = 8192) are reread by every feature block; banding keeps a band's rows in L2
// across them. skew_e128 down: 1968-2001 -> 1946-1947 us (bands of 4: 1951-1968).
constexpr int kHeavyBandDown = 8;

// The item ring: the leader's producer publishes each item index it takes; the MMA issuer, both
// CTAs' epilogue warps and the peer's producer read it from there (kItemSlots deep).
constexpr int kItemSlots = 8;
constexpr int kItemReaders = 2 + 2 * kEpiWarps;  // leader MMA + peer producer + both CTAs' epilogue warps

__host__ __device__ constexpr int num_bars(int nst) { return 2 * nst + 5 + 2 * kItemSlots; }
__host__ __device__ constexpr size_t stg_bytes(int stage) { return stage == 1 ? (size_t)kEpiWarps * kStgBytes : 0; }
__host__ __device__ constexpr size_t smem_bytes_for(int E, int nst, int stage, int ksub) {
  return 1024 + (size_t)nst * ksub * 32768 + stg_bytes(stage) + 8 * num_bars(nst) + 16 + 4 * kItemSlots +
         8 * (size_t)(E + 1);
}

// Waits with cluster-scope acquire (the phase is completed by an arrival from the peer CTA that
// releases at cluster scope, after a store into this CTA's shared memory). Bounded like
// wait_or_abort.
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_cluster_or_abort(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                      volatile int* abort_flag, int* status, int role) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (true) {
    if (try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      record_error(status, MOE_ERR_DEVICE_TIMEOUT, role);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Two GeLUs at once, GeLU(z) = z/2 (1 + erf(z / sqrt 2)), every multiply-add on the packed fp32x2
// FMA. erf from Abramowitz & Stegun 7.1.28: erf(x) = 1 - 1 / (1 + a1 x + ... + a6 x^6)^16 for
// x >= 0, |error| <= 3e-7 (1.7e-6 evaluated in fp32 this way): one reciprocal and no exponential,
// against two MUFU operations for 7.1.26. The result is rounded to bf16 (2^-9 relative), and the
// absolute error of the GeLU stays below 1e-5 for |z| <= 8 (the tail is 0 or z). On e16 the
// up-projection's launch went from 64.6 us (scalar 7.1.26) to 62.5 (packed) to 62.0 us.
__device__ __forceinline__ void gelu_as2(float z0, float z1, float& g0, float& g1) {
  const uint64_t zero = 0ull;
  auto both = [](float v) { return f2_pack(v, v); };
  const uint64_t x = ffma2(f2_pack(fabsf(z0), fabsf(z1)), both(0.70710678118654752440f), zero);
  uint64_t P = ffma2(both(0.0000430638f), x, both(0.0002765672f));
  P = ffma2(P, x, both(0.0001520143f));
  P = ffma2(P, x, both(0.0092705272f));
  P = ffma2(P, x, both(0.0422820123f));
  P = ffma2(P, x, both(0.0705230784f));
  P = ffma2(P, x, both(1.0f));
#pragma unroll
  for (int i = 0; i < 4; ++i) P = ffma2(P, P, zero);  // P^16 (inf for large x: erfc = 0)
  const float c0 = rcp_approx(f2_lo(P)), c1 = rcp_approx(f2_hi(P));  // erfc(x)
  const uint64_t sel = f2_pack(z0 >= 0.f ? 2.0f - c0 : c0, z1 >= 0.f ? 2.0f - c1 : c1);
  const uint64_t g = ffma2(ffma2(both(0.5f), f2_pack(z0, z1), zero), sel, zero);
  g0 = f2_lo(g);
  g1 = f2_hi(g);
}

__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void* tmap, int c0, int c1, int c2, int c3,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// The same copies with an L2 eviction priority (a policy from createpolicy).
__device__ __forceinline__ void tma_load_4d_pair_hint(uint32_t dst, const void* tmap, int c0, int c1, int c2, int c3,
                                                      uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// kind::f16, bf16 A and B, fp32 D, A MN-major (bit 15), B K-major, N >> 3 at 17, M >> 4 at 24.
__host__ __device__ constexpr uint32_t idesc_tn(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

struct Item {
  int e, row0, nrows, f0, heavy;
};

// The work list. An expert with cnt rows has mt = ceil(cnt / 256) row tiles: of 256 rows and a
// ragged last one, or (balanced) of equal size rounded up to 16, so that few items per pair do not
// leave a round of full items behind a round of tiny ones (cnt = 530: 192 + 192 + 146 rows instead
// of 256 + 256 + 18). Each row tile meets each 256-feature block once: an item.
//
// Experts fall into two classes. A heavy expert (more than heavy_rows rows) reuses each weight slab
// over several row tiles, read once from HBM and then from L2: its items are tensor-core work. A
// light expert's items each stream a weight slab that nothing else reads: HBM work. In index order
// a skewed routing runs all heavy items, then all light ones; the list interleaves the two classes
// in proportion to their item counts instead (item w is heavy when floor((w+1) nH / n) >
// floor(w nH / n)), so the items in flight hold a mix of both. Within a class, items go by expert,
// then feature block, then row tile (fastest): the pairs that run together share a weight slab.
// With band > 0 a heavy expert's items go by band of `band` row tiles first (the down-projection,
// whose row tiles are as large as its weight slabs).
// Both classes share one limit, the rate at which each SM's TMA fills its shared-memory ring (about
// 80 GB/s per SM in every mix measured), so they overlap only a little. When both are present (a
// skewed batch) the items come from a workspace counter through an item ring, so that the items in
// flight are a contiguous stretch of the list, and the weight copies carry an L2 priority:
// evict-last for a heavy expert's slabs (read by each of its row tiles), evict-first for a light
// expert's (read once), so that the light experts' stream does not push a heavy slab out of L2
// before its last row tile has read it. Skew workload (T = 16384, E = 128), against the static
// round-robin list in expert order: down-projection 2060 -> 1963 us, up-projection unchanged, and
// the up-projection's DRAM reads 10.17 -> 9.15 GB (8.87 algorithmic). On evenly routed batches the
// roles walk the list round-robin by themselves, as the hand-off through the ring costs there.
// PH / PL: per-expert prefix sums of the row tiles of the heavy / light experts (the other class
// counts zero tiles).
__device__ __forceinline__ Item decode_item(int w, const int* PH, const int* PL, int E, int NB,
                                            const int32_t* offsets, int balanced, int band, long long nH,
                                            long long n) {
  long long before;  // heavy items listed before w
  bool heavy;
  if (nH == 0 || nH == n) {  // one class: the list in expert order, no division
    heavy = nH != 0;
    before = heavy ? w : 0;
  } else {
    before = (long long)w * nH / n;
    heavy = (long long)(w + 1) * nH / n > before;
  }
  const int* P = heavy ? PH : PL;
  const int i = heavy ? (int)before : w - (int)before;  // index within the class
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P[mid] * NB <= i) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mt = P[e + 1] - P[e];
  int r = i - P[e] * NB;  // item within the expert: row tile r % mt of feature block r / mt
  if (heavy && band > 0 && mt > band) {
    // bands of `band` row tiles: within a band, every feature block meets each of the band's row
    // tiles before the next band starts, so the band's rows stay in L2 across the feature blocks
    const int b = r / (band * NB), nr = min(band, mt - b * band), j = r - b * band * NB;
    r = (j / nr) * mt + b * band + j % nr;
  }
  const int cnt = offsets[e + 1] - offsets[e];
  int rte = BR;
  if (balanced) {
    const int b = ((cnt + mt - 1) / mt + 15) & ~15;
    if ((mt - 1) * b < cnt) rte = b;  // every tile keeps at least one row
  }
  Item it;
  it.e = e;
  it.heavy = heavy;
  it.row0 = offsets[e] + (r % mt) * rte;
  it.nrows = min(rte, offsets[e + 1] - it.row0);
  it.f0 = (r / mt) * BF;
  return it;
}

template <int STAGE>
struct EpiOut { using T = __nv_bfloat16; };
template <>
struct EpiOut<2> { using T = float; };

// tmW: with a_one_box, the weights as [E][N/64][K][64] (4D: one box is this CTA's two 64-feature
// atoms of KSUB k-blocks, a single copy); otherwise [E][K][N] (3D: one box per atom and k-block).
// tmXs: KSUB = 1, x rows as [rows][K] (2D); KSUB = 2, as [K/64][rows][64] (3D: both k-blocks at once,
// the second box_rows rows after the first); map i copies 16 (i + 1) rows.
template <int STAGE, int STAGES, int KSUB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
ffn_tct_kernel(const __grid_constant__ BoxMaps tmXs, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ CUtensorMap tmH, typename EpiOut<STAGE>::T* __restrict__ out,
               const int32_t* __restrict__ offsets, const float* __restrict__ row_gate, int K, int N, int E,
               int balanced, int heavy_rows, int heavy_band, int a_one_box, int l2_hints, int* sched, int* status,
               uint64_t timeout_ns) {
  using OutT = typename EpiOut<STAGE>::T;
  constexpr int kTileABytes_ = kTileABytes<KSUB>, kTileASubBytes_ = kTileASubBytes<KSUB>;
  constexpr int kTileBBytes_ = kTileBBytes<KSUB>, kStageBytes_ = kStageBytes<KSUB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;                            // weights: [stage][2 atoms][KSUB*64 k][64 f]
  const uint32_t sB = base + STAGES * kTileABytes_;    // rows:    [stage][KSUB][128 rows][64 k]
  const uint32_t sStg = base + STAGES * kStageBytes_;  // up: per-warp output staging [32 rows][32 f]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * kStageBytes_ + stg_bytes(STAGE));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + num_bars(STAGES));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* slot_w = reinterpret_cast<volatile int*>(tmem_slot + 4);  // [kItemSlots]: item ring
  int* PH = reinterpret_cast<int*>(tmem_slot + 4 + kItemSlots);  // [E + 1]: heavy experts' row-tile prefix
  int* PL = PH + (E + 1);                                        // [E + 1]: light experts' row-tile prefix
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, TEMPTY = 2 * STAGES + 2, DONE = 2 * STAGES + 4;
  const int IFULL = 2 * STAGES + 5, IEMPTY = IFULL + kItemSlots;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(bar(FULL + s), 1); mbar_init(bar(EMPTY + s), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(bar(TFULL + a), 1); mbar_init(bar(TEMPTY + a), 2 * kEpiWarps); }
    mbar_init(bar(DONE), 1);
    for (int q = 0; q < kItemSlots; ++q) { mbar_init(bar(IFULL + q), 1); mbar_init(bar(IEMPTY + q), kItemReaders); }
    fence_mbar_init();
    *abort_flag = 0;
    for (int i = 0; i < kBoxMaps; ++i) tma_prefetch_desc(&tmXs.m[i]);
    tma_prefetch_desc(&tmW);
    if (STAGE == 1) tma_prefetch_desc(&tmH);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  griddep_launch_dependents();
  griddep_wait();
  if (warp == 2) {
    int run_h = 0, run_l = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int mh = 0, ml = 0;
      if (e < E) {
        const int cnt = offsets[e + 1] - offsets[e];
        const int mt = cnt > 0 ? (cnt + BR - 1) / BR : 0;
        if (cnt > heavy_rows) mh = mt; else ml = mt;
      }
      int ih = mh, il = ml;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int vh = __shfl_up_sync(0xffffffffu, ih, o);
        const int vl = __shfl_up_sync(0xffffffffu, il, o);
        if (lane >= o) { ih += vh; il += vl; }
      }
      if (e < E) { PH[e] = run_h + ih - mh; PL[e] = run_l + il - ml; }
      run_h += __shfl_sync(0xffffffffu, ih, 31);
      run_l += __shfl_sync(0xffffffffu, il, 31);
    }
    if (lane == 0) { PH[E] = run_h; PL[E] = run_l; }
  }
  // Both CTAs' barriers must be initialised before any signal crosses to the peer.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int NB = (N + BF - 1) / BF;
  const int KB = (K + BK * KSUB - 1) / (BK * KSUB);  // pipeline stages per item
  const long long n_heavy = (long long)PH[E] * NB;
  const long long n_items = n_heavy + (long long)PL[E] * NB;
  const int total_items = (int)n_items;
  // Routing with both heavy and light experts (a skewed batch): items from the workspace counter
  // through the item ring, and L2 priorities on the weight copies. Otherwise every role walks the
  // list round-robin by itself (pair, pair + npairs, ...): on evenly routed batches the ring's
  // hand-off and the priorities measured 2-10% slower (e16 up 61.7 against 67.4 us).
  const bool mixed = n_heavy > 0 && n_heavy < n_items && sched != nullptr;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      // The leader's producer takes the pair's items: from the counter *sched (every pair takes the
      // next unclaimed item, so the items in flight are always a contiguous stretch of the list), or
      // pair, pair + npairs, ... without one. It publishes each index in the item ring of both CTAs
      // one item ahead of its own loads (the peer's producer starts an item's loads without waiting
      // for a signal), and asks the counter for the index after that while it loads the current
      // item. The peer's producer and every other role read the ring; an index past the list ends
      // every role's loop.
      int stage = 0, iq = 0;
      uint32_t phase = 0, filled = 0, fill_phase = 0, iphase = 0;
      const uint64_t pol_last = policy_evict_last(), pol_first = policy_evict_first();
      auto take = [&](int prev) { return sched != nullptr ? atomicAdd(sched, 1) : prev + npairs; };
      auto publish = [&](int v) -> bool {
        if (!wait_cluster_or_abort(bar(IEMPTY + iq), iphase ^ 1u, timeout_ns, abort_flag, status, 44)) return false;
        slot_w[iq] = v;
        st_shared_cluster_u32(map_to_cta(smem_u32((const void*)(slot_w + iq)), 1), (uint32_t)v);
        mbar_arrive(bar(IFULL + iq));
        mbar_arrive_cluster(map_to_cta(bar(IFULL + iq), 1));
        if (++iq == kItemSlots) { iq = 0; iphase ^= 1u; }
        return true;
      };
      // leader: w = the item loaded in this iteration, w_next = the one after it (already taken)
      int w = pair, w_next = 0, w_pub = pair + npairs;
      if (mixed && leader) {
        w = atomicAdd(sched, 1);
        if (!publish(w)) goto producer_out;
        if (w < total_items) w_next = take(w);
      }
      while (!*abort_flag) {
        if (!mixed) {
          if (w >= total_items) break;
          w_pub = w + npairs;
        } else if (leader) {
          if (w >= total_items) break;
          if (!publish(w_next)) break;  // the next item, visible before this one's loads start
          w_pub = w_next;
          if (w_next < total_items) w_next = take(w_next);  // the one after: in flight during the loads
        } else {
          if (!wait_cluster_or_abort(bar(IFULL + iq), iphase, timeout_ns, abort_flag, status, 44)) break;
          w = slot_w[iq];
          mbar_arrive_cluster(map_to_cta(bar(IEMPTY + iq), 0));
          if (++iq == kItemSlots) { iq = 0; iphase ^= 1u; }
          if (w >= total_items) break;
        }
        const Item it = decode_item(w, PH, PL, E, NB, offsets, balanced, heavy_band, n_heavy, n_items);
        const int nt = (it.nrows + 15) & ~15;           // MMA N: rows rounded up to 16
        const int frow = it.row0 + (nt / 2) * (int)rank;  // this CTA holds rows [nt/2 * rank, +nt/2)
        const int feat = it.f0 + (BF / 2) * (int)rank;
        const int hbox = box_rows_for(nt);
        const CUtensorMap* tmX = &tmXs.m[hbox / 16 - 1];
        const uint32_t stage_tx = 2u * (uint32_t)(kTileABytes_ + hbox * 128 * KSUB);  // both CTAs' bytes
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(bar(EMPTY + stage), phase ^ 1u, timeout_ns, abort_flag, status, 41)) goto producer_out;
          const uint32_t full_leader = map_to_cta(bar(FULL + stage), 0);
          if (leader) mbar_arrive_expect_tx(bar(FULL + stage), stage_tx);
          if (a_one_box && l2_hints && mixed) {
            // a heavy expert's slab is read by every row tile of the expert: keep it in L2 ahead of
            // the light experts' slabs, which nothing reads twice
            tma_load_4d_pair_hint(sA + stage * kTileABytes_, &tmW, 0, kb * BK * KSUB, feat / 64, it.e, full_leader,
                                  it.heavy ? pol_last : pol_first);
          } else if (a_one_box) {
            tma_load_4d_pair(sA + stage * kTileABytes_, &tmW, 0, kb * BK * KSUB, feat / 64, it.e, full_leader);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int u = 0; u < KSUB; ++u)
                tma_load_3d_pair(sA + stage * kTileABytes_ + j * kTileASubBytes_ + u * BK * 128, &tmW, feat + 64 * j,
                                 (kb * KSUB + u) * BK, it.e, full_leader);
          }
          if (KSUB == 1) tma_load_2d_pair(sB + stage * kTileBBytes_, tmX, kb * BK, frow, full_leader);
          else tma_load_3d_pair(sB + stage * kTileBBytes_, tmX, 0, frow, kb * KSUB, full_leader);
          filled |= 1u << stage;
          fill_phase = (fill_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!mixed || leader) w = w_pub;  // the item published ahead (or the next round-robin one)
      }
    producer_out:
      if (leader && mixed) {
        // This pair takes no more items. The last pair to stop sets the counter back to zero for the
        // next launch (no pair reads it after this point; the next launch reads it only after its
        // griddepcontrol.wait, i.e. after this grid has completed).
        __threadfence();
        if (atomicAdd(sched + 1, 1) == npairs - 1) {
          atomicExch(sched, 0);
          atomicExch(sched + 1, 0);
        }
      }
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
        int stage = 0, acc = 0, iq = 0, w = pair - npairs;
        uint32_t phase = 0, acc_phase = 0, iphase = 0;
        while (!*abort_flag) {
          if (mixed) {
            if (!wait_or_abort(bar(IFULL + iq), iphase, timeout_ns, abort_flag, status, 42)) break;
            w = slot_w[iq];
            mbar_arrive(bar(IEMPTY + iq));
            if (++iq == kItemSlots) { iq = 0; iphase ^= 1u; }
          } else {
            w += npairs;
          }
          if (w >= total_items) break;
          const Item it = decode_item(w, PH, PL, E, NB, offsets, balanced, heavy_band, n_heavy, n_items);
          const uint32_t idesc = idesc_tn(BF, (it.nrows + 15) & ~15);
          const uint32_t b_step = (uint32_t)box_rows_for((it.nrows + 15) & ~15) * 128;  // 64 k of B, KSUB = 2
          if (!wait_or_abort(bar(TEMPTY + acc), acc_phase ^ 1u, timeout_ns, abort_flag, status, 42)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BR);
          const uint64_t a_base = make_smem_desc_sw128(sA, kTileASubBytes_, 1024);
          const uint64_t b_base = make_smem_desc_sw128(sB, 16, 1024);
          const uint64_t b_hi = (uint64_t)(b_step >> 4);
          for (int kb = 0; kb < KB; ++kb) {
            // descriptors ready before the wait, so that the MMAs issue as soon as the stage lands (the
            // address field moves by the stage's offset >> 4; skew_e128 down 1976-1988 -> 1919-1931 us)
            const uint64_t a_desc = a_base + (uint64_t)((stage * kTileABytes_) >> 4);
            const uint64_t b_desc = b_base + (uint64_t)((stage * kTileBBytes_) >> 4);
            if (!wait_or_abort(bar(FULL + stage), phase, timeout_ns, abort_flag, status, 42)) goto mma_out;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < KSUB * BK / 16; ++kk)
              tc_mma_f16_pair(d_tmem, a_desc + (uint64_t)((kk * 16 * 128) >> 4),
                              b_desc + (kk / 4) * b_hi + (uint64_t)(((kk % 4) * 32) >> 4), idesc,
                              (kb | kk) != 0 ? 1u : 0u);
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
    const int q = warp & 3;                              // TMEM lanes 32q .. 32q+31: features
    const int c_begin = ((warp - 2) >> 2) * kSegRows;     // this warp's quarter of the rows
    const uint32_t stg = sStg + (uint32_t)((warp - 2) * kStgBytes);
    int acc = 0, iq = 0, w = pair - npairs;
    uint32_t acc_phase = 0, iphase = 0;
    while (!*abort_flag) {
      if (mixed) {
        if (!__all_sync(0xffffffffu,
                        wait_cluster_or_abort(bar(IFULL + iq), iphase, timeout_ns, abort_flag, status, 43)))
          break;
        w = slot_w[iq];
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(IEMPTY + iq), 0));
        if (++iq == kItemSlots) { iq = 0; iphase ^= 1u; }
      } else {
        w += npairs;
      }
      if (w >= total_items) break;
      const Item it = decode_item(w, PH, PL, E, NB, offsets, balanced, heavy_band, n_heavy, n_items);
      // warp-uniform: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, wait_or_abort(bar(TFULL + acc), acc_phase, timeout_ns, abort_flag, status, 43)))
        break;
      tc_fence_after();
      const int f = it.f0 + (BF / 2) * (int)rank + 32 * q + lane;
      const bool f_ok = f < N;
      // CR rows per step: the epilogue of all CR values as independent chains (no per-row branch
      // inside the arithmetic), then the stores.
      for (int c = c_begin; c < c_begin + kSegRows && c < it.nrows; c += CR) {
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BR + c);
        uint32_t v[CR];
        tmem_ld_32x32b_x32(taddr, v);
        tmem_ld_wait();
        const int nvalid = min(CR, it.nrows - c);
        const int r0 = it.row0 + c;
        float res[CR];
        if (STAGE == 1) {
#pragma unroll
          for (int i = 0; i < CR; i += 2) gelu_as2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), res[i], res[i + 1]);
        } else {
          const float g0 = lane < nvalid ? row_gate[r0 + lane] : 0.f;
#pragma unroll
          for (int i = 0; i < CR; ++i) res[i] = __shfl_sync(0xffffffffu, g0, i) * __uint_as_float(v[i]);
        }
        if (STAGE == 1 && nvalid == CR) {
          // CR rows x 32 features through shared memory, one TMA store (columns past N are clipped)
          if (lane == 0) bulk_wait_group_read0();  // the previous store has finished reading the buffer
          __syncwarp();
#pragma unroll
          for (int i = 0; i < CR; ++i) {
            const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(res[i]));
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg + (uint32_t)(i * 64 + lane * 2)), "h"(b) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmH, stg, it.f0 + (BF / 2) * (int)rank + 32 * q, r0);
            bulk_commit_group();
          }
        } else if (f_ok) {
          // a chunk that crosses the end of the expert's rows (or the fp32 down output): plain stores
          OutT* dst = out + (size_t)r0 * N + f;
#pragma unroll
          for (int i = 0; i < CR; ++i)
            if (i < nvalid) dst[(size_t)i * N] = from_f32<OutT>(res[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(TEMPTY + acc), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (STAGE == 1 && lane == 0) bulk_wait_group0();  // stores read shared memory until they complete
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

// 128-byte-swizzled bf16 tensor map of up to four dimensions (strides in bytes, dims 1..rank-1).
bool encode_sw128(EncodeTiledFn enc, CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides_bytes, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int STAGE, int STAGES, int KSUB>
cudaError_t launch_tct(const FfnArgs& p, EncodeTiledFn enc, const CUtensorMap& tmH, size_t smem, cudaStream_t s) {
  using OutT = typename EpiOut<STAGE>::T;
  auto kern = ffn_tct_kernel<STAGE, STAGES, KSUB>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // Persistent: as many pairs as can be resident at once (two-SM clusters may not tile every SM).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0)
    clusters = device_sm_count() / 2;
  const int NB = (p.N + BF - 1) / BF;
  // Balanced row tiles when there are fewer than three items per resident pair (the estimate
  // spreads the rows evenly over the experts); 256-row tiles otherwise.
  const long long active = p.rows < p.E ? p.rows : p.E;
  const long long rpe = (p.rows + active - 1) / active;
  const int balanced = active * ((rpe + BR - 1) / BR) * NB >= 3LL * clusters ? 0 : 1;
  CUtensorMap tmW;
  BoxMaps tmXs;
  // Weights [E][K][N], MN-major A operand. N a multiple of 64: viewed as [E][N/64][K][64] so one
  // box brings both of this CTA's 64-feature atoms (the fewer copies a stage takes, the faster the
  // SM's copy engine feeds it); otherwise one [KSUB*64 k][64 f] box per atom and k-block.
  const int a_one_box = p.N % 64 == 0;
  if (a_one_box) {
    const cuuint64_t dims[4] = {64, (cuuint64_t)p.K, (cuuint64_t)p.N / 64, (cuuint64_t)p.E};
    const cuuint64_t str[3] = {(cuuint64_t)p.N * 2, 128, (cuuint64_t)p.K * p.N * 2};
    const cuuint32_t box[4] = {64, BK * KSUB, 2, 1};
    if (!encode_sw128(enc, &tmW, p.w, 4, dims, str, box)) return cudaErrorInvalidValue;
  } else {
    const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.K, (cuuint64_t)p.E};
    const cuuint64_t str[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.K * p.N * 2};
    const cuuint32_t box[3] = {64, BK, 1};
    if (!encode_sw128(enc, &tmW, p.w, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  // Rows of x_perm (or h): K-major B operand, up to 128 rows (one CTA's half of a tile) per box: a
  // [rows][K] view for one k-block, a [K/64][rows][64] view (K a multiple of 128) for two; one map per
  // box height 16, 32, ..., 128. A stage copies only the rows its item has (rounded up to 16): an
  // item of 84 rows copies 48 rows per CTA, not 128.
  for (int i = 0; i < kBoxMaps; ++i) {
    const cuuint32_t hrows = 16u * (cuuint32_t)(i + 1);
    if (KSUB == 1) {
      const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.rows};
      const cuuint64_t str[1] = {(cuuint64_t)p.K * 2};
      const cuuint32_t box[2] = {BK, hrows};
      if (!encode_sw128(enc, &tmXs.m[i], p.a, 2, dims, str, box)) return cudaErrorInvalidValue;
    } else {
      const cuuint64_t dims[3] = {64, (cuuint64_t)p.rows, (cuuint64_t)p.K / 64};
      const cuuint64_t str[2] = {(cuuint64_t)p.K * 2, 128};
      const cuuint32_t box[3] = {64, hrows, KSUB};
      if (!encode_sw128(enc, &tmXs.m[i], p.a, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
  }
  const long long max_items = ((long long)(p.rows + BR - 1) / BR + p.E) * NB;
  long long pairs = clusters < max_items ? clusters : max_items;
  // An expert is heavy (its weight slabs serve several row tiles) above one full row tile.
  const int heavy_rows = BR;
  // Item counter (and the count of pairs done with it) in workspace header words 4 and 5.
  int* sched = p.status != nullptr ? p.status + 4 : nullptr;
  const int l2_hints = 1;  // skew_e128 up: DRAM reads 10.17 -> 9.16 GB per launch (8.87 GB algorithmic)
  const int heavy_band = STAGE == 2 ? kHeavyBandDown : 0;
  return launch_pdl(kern, dim3((unsigned)(2 * pairs)), dim3(kThreads), smem, s, tmXs, tmW, tmH, (OutT*)p.out,
                    p.offsets, p.row_gate, p.K, p.N, p.E, balanced, heavy_rows, heavy_band, a_one_box, l2_hints,
                    sched, p.status, p.timeout_ns);
}

}  // namespace

cudaError_t launch_ffn_tensor_t(const FfnArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  if (p.dt != MOE_DTYPE_BF16) return cudaErrorNotSupported;
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // Two k-blocks per stage (64 KB, three stages) when K allows it and the weight slabs serve
  // several row tiles, i.e. are mostly read from L2: fewer, larger copies per MMA (e16 up:
  // 73.7 -> 70.6 us). For the up-projection three 64 KB stages hold as many bytes in flight as its
  // six 32 KB ones (the output staging takes the rest), and an average of one full row tile per
  // expert suffices (skew_e128 up: 2057-2101 -> 1992-1999 us); the down-projection would give up
  // its seventh 32 KB stage, and takes them only at two row tiles per expert (skew_e128 down with
  // three 64 KB stages: 1953-1975 -> 2027 us). When every slab streams from HBM once (prefill),
  // six or seven 32 KB stages hide HBM latency better (1.34 vs 1.35 ms).
  const long long active = p.rows < p.E ? p.rows : p.E;
  const long long rpe = (p.rows + active - 1) / active;
  const bool ksub2_ok = p.K % 128 == 0 && rpe >= (p.stage == 1 ? BR : 2 * BR);
  CUtensorMap tmH{};  // up: h [rows][N] bf16, 32 features x CR rows per store, no swizzle
  if (p.stage == 1) {
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.rows};
    const cuuint64_t str[1] = {(cuuint64_t)p.N * 2};
    const cuuint32_t box[2] = {32, CR};
    if (!encode_tmap_plain(enc, &tmH, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.out, 2, dims, str, box))
      return cudaErrorInvalidValue;
    if (ksub2_ok && smem_bytes_for(p.E, 3, 1, 2) <= (size_t)kMaxSmem)
      return launch_tct<1, 3, 2>(p, enc, tmH, smem_bytes_for(p.E, 3, 1, 2), s);
    const bool six = smem_bytes_for(p.E, 6, 1, 1) <= (size_t)kMaxSmem;
    const size_t smem = smem_bytes_for(p.E, six ? 6 : 5, 1, 1);
    return six ? launch_tct<1, 6, 1>(p, enc, tmH, smem, s) : launch_tct<1, 5, 1>(p, enc, tmH, smem, s);
  }
  if (ksub2_ok && smem_bytes_for(p.E, 3, 2, 2) <= (size_t)kMaxSmem)
    return launch_tct<2, 3, 2>(p, enc, tmH, smem_bytes_for(p.E, 3, 2, 2), s);
  const bool seven = smem_bytes_for(p.E, 7, 2, 1) <= (size_t)kMaxSmem;
  const size_t smem = smem_bytes_for(p.E, seven ? 7 : 6, 2, 1);
  return seven ? launch_tct<2, 7, 1>(p, enc, tmH, smem, s) : launch_tct<2, 6, 1>(p, enc, tmH, smem, s);
}

}  // namespace moe
