// Router and dispatch for decode-sized batches (T <= 8 tokens) in one launch.
// csdn/6a919c0d §2.2 steps 1-4 (logits, softmax, top-k, gates); csdn/6a462027 §4.2 steps 4-5
// (per-expert histogram, offsets, stable grouping); aicoding/6a320eef §3.2 (capacity).
//
// With a handful of tokens the router is a skinny product whose cost is reading W_r (d x E);
// a tile-per-128-tokens kernel streams it from a few SMs, and a separate dispatch launch and
// row gather follow. Here every CTA reads a 64-row slice of W_r (16 KB at d = 8192, E = 128,
// with 16-byte loads of 8 experts, all in flight together with the x slice: the kernel is one
// chain of memory latencies, so each step keeps its loads independent) and forms the partial
// logits of all T tokens on CUDA cores. For T <= 2 each CTA writes its partials and the CTA that
// finishes last (an atomic ticket, nobody waits) adds them in CTA order; for larger T the eight
// CTAs of a cluster first add theirs over DSMEM in rank order and the last cluster adds the
// clusters' sums (clusters of eight 8-token CTAs took microseconds to be placed, so one and two
// tokens use plain CTAs with 2-token accumulators). The last CTA then, for each token, takes the max,
// the softmax denominator and the k largest logits (lower expert index first among equals), and
// writes the routing arrays of the dispatch: counts and offsets (clipped at the capacity), the
// permutation, row_of and row_gate. No x_perm: the weight-streaming FFN reads x rows through
// perm_token. Every sum runs in a fixed order, so results are reproducible run to run.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kCluster = 8;
constexpr int kRowsPerCta = 64;  // W_r rows per CTA when d allows it (T > 2)
constexpr int kMaxGrid = 128;
constexpr int kMaxGridSmall = 64;  // T <= 2: 128 rows per CTA at d = 8192
constexpr int kBatch = 4;        // W_r rows per thread in flight

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void bf16x8(const uint4 u, float (&v)[8]) {
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}

// smem: xs [T][KR] fp32 | sg [G][T][E] per-group partials | sp [T][E] CTA partials (then logits)
// | sidx [T*k] | sgate [T*k] | scnt [E] | soff [E+1]
template <int TMAX, bool kClustered>
__global__ void __launch_bounds__(kThreads, 1)
route_small_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w_r,
                   const float* __restrict__ b_r, int T, int d, int E, int k, int renorm, int cap, int KR,
                   float* __restrict__ partials, int* __restrict__ ticket, int32_t* __restrict__ topk_idx,
                   float* __restrict__ topk_gate, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ perm_token, int32_t* __restrict__ row_of, float* __restrict__ row_gate) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C8 = E / 8;                                // 16-byte chunks (8 experts) of a W_r row
  const int G = kThreads / C8;                         // row groups (E <= 2048)
  float* xs = smem;                                    // [T][KR]
  float* sg = xs + T * KR;                             // [G][T][E]
  float* sp = sg + G * T * E;                          // [T][E]
  int* sidx = reinterpret_cast<int*>(sp + T * E);      // [T*k]
  float* sgate = reinterpret_cast<float*>(sidx + 64);  // [T*k]
  int* scnt = reinterpret_cast<int*>(sgate + 64);      // [E]
  int* soff = scnt + E;                                // [E+1]
  __shared__ int s_last;
  __shared__ int s_wtot[kThreads / 32];

  // ---- 1. this CTA's k-rows [r0, r1): thread (g, c8) takes experts 8 c8 .. 8 c8 + 7 of the rows
  // g, g + G, ...; the first batch of W_r loads and the x slice are issued before anything waits
  const int r0 = min(d, (int)blockIdx.x * KR), r1 = min(d, r0 + KR), nr = r1 - r0;
  const int c8 = tid % C8, g = tid / C8;
  const uint4* wbase = reinterpret_cast<const uint4*>(w_r + (size_t)r0 * E) + c8;
  auto load_rows = [&](int rb, uint4 (&wv)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int r = rb + i * G;
      wv[i] = (g < G && r < nr) ? __ldg(wbase + (size_t)r * C8) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 wv[kBatch];
  load_rows(g, wv);
  const int xchunks = T * (KR / 8);
  uint4 xr[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + j * kThreads;
    const int t = i / (KR / 8), kk = (i % (KR / 8)) * 8;
    xr[j] = (i < xchunks && kk < nr) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d + r0 + kk))
                                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + j * kThreads;
    if (i < xchunks) {
      const int t = i / (KR / 8), kk = (i % (KR / 8)) * 8;
      float v[8];
      bf16x8(xr[j], v);
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[t * KR + kk + q] = v[q];
    }
  }
  __syncthreads();
  float acc[TMAX][8];  // [token][expert of the chunk]
#pragma unroll
  for (int t = 0; t < TMAX; ++t)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[t][q] = 0.f;
  for (int rb = g; rb < nr; rb += kBatch * G) {
    uint4 nxt[kBatch];
    if (rb + kBatch * G < nr) load_rows(rb + kBatch * G, nxt);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int r = rb + i * G;
      if (r < nr) {
        float w[8];
        bf16x8(wv[i], w);
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
          if (t < T) {
            const float xv = xs[t * KR + r];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[t][q] = fmaf(xv, w[q], acc[t][q]);
          }
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) wv[i] = nxt[i];
  }
  if (g < G) {
#pragma unroll
    for (int t = 0; t < TMAX; ++t)
      if (t < T)
#pragma unroll
        for (int q = 0; q < 8; ++q) sg[(g * T + t) * E + 8 * c8 + q] = acc[t][q];
  }
  __syncthreads();
  for (int i = tid; i < T * E; i += kThreads) {
    float v = 0.f;
    for (int gg = 0; gg < G; ++gg) v += sg[gg * T * E + i];  // groups in order
    sp[i] = v;
  }

  // ---- 2. one partial set per cluster (its sum in rank order, by rank 0) or per CTA to global memory
  int ncl = (int)gridDim.x;
  if (kClustered) {
  cluster_sync_all();
  const uint32_t rank = cluster_ctarank();
  const int cl = (int)blockIdx.x / kCluster;
  ncl = (int)gridDim.x / kCluster;
  if (rank == 0) {
    for (int i = tid; i < T * E; i += kThreads) {
      const uint32_t local = smem_u32(sp + i);
      float part[kCluster];
#pragma unroll
      for (int c = 0; c < kCluster; ++c) part[c] = ld_cluster_f32(map_to_cta(local, (uint32_t)c));
      float v = 0.f;
#pragma unroll
      for (int c = 0; c < kCluster; ++c) v += part[c];
      partials[(size_t)cl * T * E + i] = v;
    }
  }
  cluster_sync_all();  // peers keep their shared memory until rank 0 has read it
  if (rank != 0) return;
  } else {
    __syncthreads();
    for (int i = tid; i < T * E; i += kThreads) partials[(size_t)blockIdx.x * T * E + i] = sp[i];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(ticket, 1) == ncl - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- 3. the last CTA: logits in partial-set order (all loads in flight first), then softmax
  // and top-k, one warp per token, the token's logits in registers (lane l: experts l + 32 j)
  constexpr int kParts = kClustered ? kMaxGrid / kCluster : kMaxGridSmall;
  for (int i = tid; i < T * E; i += kThreads) {
    float part[kParts];
#pragma unroll
    for (int c = 0; c < kParts; ++c) part[c] = c < ncl ? __ldcg(partials + (size_t)c * T * E + i) : 0.f;
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < kParts; ++c)
      if (c < ncl) v += part[c];
    sp[i] = v + (b_r != nullptr ? b_r[i % E] : 0.f);
  }
  __syncthreads();
  if (warp < T) {
    const int t = warp;
    const float* lg = sp + t * E;
    float lv[32];  // E <= 1024
#pragma unroll
    for (int j = 0; j < 32; ++j) lv[j] = lane + 32 * j < E ? lg[lane + 32 * j] : -INFINITY;
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) m = fmaxf(m, lv[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ssum = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (lane + 32 * j < E) ssum += expf(lv[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    float sel[8];
    for (int p = 0; p < k; ++p) {
      // the largest remaining logit, the lower index among equals (ascending e within a lane)
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (lane + 32 * j < E && (lv[j] > bv || be == 0x7fffffff)) { bv = lv[j]; be = lane + 32 * j; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      sel[p] = bv;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (lane + 32 * j == be) lv[j] = -INFINITY;
      if (lane == 0) sidx[t * k + p] = be;
    }
    float ksum = 0.f;
    if (renorm)
      for (int p = 0; p < k; ++p) ksum += expf(sel[p] - m);
    if (lane == 0)
      for (int p = 0; p < k; ++p) {
        const float gv = expf(sel[p] - m) / (renorm ? ksum : ssum);
        sgate[t * k + p] = gv;
        topk_idx[t * k + p] = sidx[t * k + p];
        topk_gate[t * k + p] = gv;
      }
  }
  __syncthreads();

  // ---- 4. dispatch: kept counts, offsets, and each assignment's row in (t, j) order
  const int A = T * k;
  int local = 0;
  int kept4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // thread owns experts 4 tid .. 4 tid + 3 (E <= 1024)
    const int e = 4 * tid + j;
    int c = 0;
    if (e < E)
      for (int a = 0; a < A; ++a) c += sidx[a] == e;
    kept4[j] = cap > 0 ? min(c, cap) : c;
    local += kept4[j];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wtot[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += s_wtot[w];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * tid + j;
    if (e < E) {
      scnt[e] = kept4[j];
      soff[e] = run;
      counts[e] = kept4[j];
      offsets[e] = run;
    }
    run += kept4[j];
  }
  if (tid == kThreads - 1) offsets[E] = run;
  __syncthreads();
  if (tid < A) {
    const int e = sidx[tid];
    int rk = 0;
    for (int a = 0; a < tid; ++a) rk += sidx[a] == e;
    const int row = (cap > 0 && rk >= cap) ? -1 : soff[e] + rk;
    row_of[tid] = row;
    if (row >= 0) {
      perm_token[row] = tid / k;
      row_gate[row] = sgate[tid];
    }
  }
  if (tid == 0) *ticket = 0;  // ready for the next launch
}

}  // namespace

// One and two tokens: plain CTAs of 128 W_r rows; more: clusters of eight 64-row CTAs.
size_t route_small_smem_bytes(int T, int d, int E, int k, int* kr_out, int* grid_out) {
  const bool small = T <= 2;
  const int rows = small ? 2 * kRowsPerCta : kRowsPerCta;
  const int want = (d + rows - 1) / rows;
  int grid = small ? want : ((want + kCluster - 1) / kCluster) * kCluster;
  const int cap = small ? kMaxGridSmall : kMaxGrid;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  int KR = (d + grid - 1) / grid;
  KR = (KR + 7) & ~7;
  const int G = kThreads / (E / 8);
  (void)k;
  if (kr_out != nullptr) *kr_out = KR;
  if (grid_out != nullptr) *grid_out = grid;
  return (size_t)(T * KR + G * T * E + T * E) * sizeof(float) + 2 * 64 * sizeof(float) +
         (size_t)(2 * E + 1) * sizeof(int);
}

bool route_small_ok(int T, int d, int E, int k, int dt, size_t partial_bytes_avail) {
  if (dt != MOE_DTYPE_BF16 || T < 1 || T > 8 || k > 8 || E % 8 != 0 || E > 1024 || d % 8 != 0) return false;
  int KR = 0, grid = 0;
  if (route_small_smem_bytes(T, d, E, k, &KR, &grid) > 96 * 1024) return false;
  if (T * (KR / 8) > 2 * kThreads) return false;  // x slice: two 16-byte loads per thread
  const int sets = T <= 2 ? grid : grid / kCluster;
  return (size_t)sets * T * E * sizeof(float) <= partial_bytes_avail;
}

cudaError_t launch_route_small(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                               int renorm, int cap, float* partials, int* ticket, int32_t* idx, float* gate,
                               int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* row_of,
                               float* row_gate, cudaStream_t s) {
  int KR = 0, grid = 0;
  const size_t smem = route_small_smem_bytes(T, d, E, k, &KR, &grid);
  const bool small = T <= 2;
  auto kern = small ? route_small_kernel<2, false> : route_small_kernel<8, true>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = small ? 1 : 2;
  return cudaLaunchKernelEx(&cfg, kern, (const __nv_bfloat16*)x, (const __nv_bfloat16*)w_r, b_r, T, d, E, k, renorm,
                            cap, KR, partials, ticket, idx, gate, counts, offsets, perm_token, row_of, row_gate);
}

}  // namespace moe
