// Dispatch: per-expert histogram, exclusive scan, stable permutation and row gather.
// csdn/6a462027 §4.2 steps 4-5 (group each expert's tokens: "in practice a scatter").
//
// moe_dispatch and moe_dispatch_noalloc run count+scan (one kernel, the last CTA scans) and
// scatter+gather as two launches with programmatic dependent launch (launch_dispatch_fast). Inside
// the layer, with the tensor-core router's per-tile histograms, one launch does it all
// (launch_dispatch_from_hist).
//
// The T*k assignments, in row-major (t, j) order, are cut into chunks of 256
// (one CTA each).
//   count:   shared-memory histogram of a chunk -> blk_counts[chunk][e]
//   scan:    one CTA: counts[e] = sum over chunks, offsets = exclusive scan over
//            experts, blk_base[chunk][e] = offsets[e] + counts of earlier chunks
//   scatter: rank of each assignment among equal experts inside its chunk from
//            __match_any_sync (inside a warp) plus per-warp counts (across warps);
//            row = blk_base + rank. No atomics decide an order: the permutation is
//            the stable one and is bit-reproducible.
//   gather:  x_perm[r] = x[perm_token[r]], one warp per row, 16-byte vectors.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kChunk = kDispatchChunk;
constexpr int kWarpsPerChunk = kChunk / 32;

// Scatter and gather in one kernel: `split` CTAs per 256-assignment chunk each compute the chunk's
// stable ranks (cheap, redundant), the first of them writes row_of / perm_token / row_gate, and
// each copies its share of the chunk's rows x[t] -> x_perm[row] (one warp per row, 16-byte vectors).
// Dropped assignments (capacity) get row -1 and are not copied.
__global__ void __launch_bounds__(kChunk)
dispatch_scatter_gather_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate, int A, int k,
                               int E, const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
                               int cap, int split, const int4* __restrict__ x, int vec_per_row,
                               int32_t* __restrict__ row_of, int32_t* __restrict__ perm_token,
                               float* __restrict__ row_gate, int4* __restrict__ x_perm) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int wcnt[];  // [kWarpsPerChunk][E], then the chunk's rows [kChunk]
  int* srow = wcnt + kWarpsPerChunk * E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x / split, part = blockIdx.x % split;
  for (int i = tid; i < kWarpsPerChunk * E; i += kChunk) wcnt[i] = 0;
  __syncthreads();
  const int a = chunk * kChunk + tid;
  int e = -1;
  if (a < A) {
    e = idx[a];
    if (e < 0 || e >= E) e = -1;
  }
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  int row = -1;
  if (e >= 0) {
    int pre = 0;
    for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
    row = blk_base[(size_t)chunk * E + e] + pre + rank;
    if (cap > 0 && row - offsets[e] >= cap) row = -1;  // past the expert's capacity: dropped
  }
  srow[tid] = row;
  if (part == 0 && a < A) {
    row_of[a] = row;
    if (row >= 0) {
      perm_token[row] = a / k;
      row_gate[row] = gate[a];
    }
  }
  __syncthreads();
  // rows of this part: assignments part, part + split, ... of the chunk, one warp each
  const int n_here = min(kChunk, A - chunk * kChunk);
  for (int i = part + split * warp; i < n_here; i += split * kWarpsPerChunk) {
    const int r = srow[i];
    if (r < 0) continue;
    const int4* src = x + (size_t)((chunk * kChunk + i) / k) * vec_per_row;
    int4* dst = x_perm + (size_t)r * vec_per_row;
    int v = lane;
    for (; v + 96 < vec_per_row; v += 128) {
      const int4 v0 = __ldg(src + v), v1 = __ldg(src + v + 32), v2 = __ldg(src + v + 64), v3 = __ldg(src + v + 96);
      dst[v] = v0; dst[v + 32] = v1; dst[v + 64] = v2; dst[v + 96] = v3;
    }
    for (; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
  }
}

// The same scatter + gather when the per-chunk histograms are already in blk_counts (written by the
// router): every CTA first rebuilds, in a fixed order, the experts' totals (clipped at the capacity),
// their exclusive scan (offsets) and its chunk's bases; CTA 0 writes counts and offsets. Reading
// nb x E counts per CTA replaces a separate count kernel.
__global__ void __launch_bounds__(kChunk)
dispatch_from_hist_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate, int A, int k, int E,
                          int nb, const int32_t* __restrict__ blk_counts, int cap, int split,
                          const int4* __restrict__ x, int vec_per_row, int32_t* __restrict__ counts,
                          int32_t* __restrict__ offsets, int32_t* __restrict__ row_of,
                          int32_t* __restrict__ perm_token, float* __restrict__ row_gate, int4* __restrict__ x_perm) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int sm[];
  int* wcnt = sm;                              // [kWarpsPerChunk][E]
  int* srow = wcnt + kWarpsPerChunk * E;       // [kChunk]
  int* sbase = srow + kChunk;                  // [E]: this chunk's first row per expert
  int* soff = sbase + E;                       // [E]: offsets
  __shared__ int warp_tot[kChunk / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x / split, part = blockIdx.x % split;
  // this thread's assignment and gate: loads in flight while the histograms are summed
  const int a = chunk * kChunk + tid;
  const int e_raw = a < A ? idx[a] : -1;
  const float g_a = (part == 0 && a < A) ? gate[a] : 0.f;
  // totals and this chunk's prefix: thread (g, e) sums the chunks c = g (mod G) of expert e (E <= kChunk),
  // then thread e adds the G partials in order
  __shared__ int s_tp[2][kChunk];
  const int G = kChunk / E;
  if (tid < G * E) {
    const int e = tid % E, g = tid / E;
    int tot = 0, p = 0;
    for (int c = g; c < nb; c += G) {
      const int v = blk_counts[(size_t)c * E + e];
      tot += v;
      if (c < chunk) p += v;
    }
    s_tp[0][tid] = tot;
    s_tp[1][tid] = p;
  }
  for (int i = tid; i < kWarpsPerChunk * E; i += kChunk) wcnt[i] = 0;
  __syncthreads();
  int kept = 0, pre = 0;
  if (tid < E) {
    int tot = 0;
    for (int g = 0; g < G; ++g) {
      tot += s_tp[0][g * E + tid];
      pre += s_tp[1][g * E + tid];
    }
    kept = cap > 0 ? min(tot, cap) : tot;
  }
  int incl = kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int run = incl - kept;
  for (int w = 0; w < warp; ++w) run += warp_tot[w];
  if (tid < E) {
    soff[tid] = run;
    sbase[tid] = run + pre;
    if (blockIdx.x == 0) {
      counts[tid] = kept;
      offsets[tid] = run;
    }
  }
  run += kept;
  if (blockIdx.x == 0 && tid == kChunk - 1) offsets[E] = run;
  const int e = (e_raw < 0 || e_raw >= E) ? -1 : e_raw;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  int row = -1;
  if (e >= 0) {
    int p = 0;
    for (int w = 0; w < warp; ++w) p += wcnt[w * E + e];
    row = sbase[e] + p + rank;
    if (cap > 0 && row - soff[e] >= cap) row = -1;  // past the expert's capacity: dropped
  }
  srow[tid] = row;
  if (part == 0 && a < A) {
    row_of[a] = row;
    if (row >= 0) {
      perm_token[row] = a / k;
      row_gate[row] = g_a;
    }
  }
  __syncthreads();
  // the gather: each warp copies its rows four at a time, all sixteen 16-byte loads per lane in
  // flight before the stores (rows i0 + j * stride)
  const int n_here = min(kChunk, A - chunk * kChunk);
  const int stride = split * kWarpsPerChunk;
  for (int i0 = part + split * warp; i0 < n_here; i0 += 4 * stride) {
    int rr[4];
    const int4* src[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j * stride;
      rr[j] = i < n_here ? srow[i] : -1;
      src[j] = x + (size_t)((chunk * kChunk + (i < n_here ? i : 0)) / k) * vec_per_row;
    }
    for (int v0 = 0; v0 < vec_per_row; v0 += 128) {
      int4 buf[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // unconditional loads from valid addresses; stores predicated
          const int v = v0 + lane + 32 * q;
          const int4* ptr = src[j] + (v < vec_per_row ? v : 0);
          asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(buf[j][q].x), "=r"(buf[j][q].y), "=r"(buf[j][q].z), "=r"(buf[j][q].w)
                       : "l"(ptr));
        }
      asm volatile("" ::: "memory");  // keep all sixteen loads ahead of the stores
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int v = v0 + lane + 32 * q;
          if (rr[j] >= 0 && v < vec_per_row)
            asm volatile("st.global.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(x_perm + (size_t)rr[j] * vec_per_row + v),
                         "r"(buf[j][q].x), "r"(buf[j][q].y), "r"(buf[j][q].z), "r"(buf[j][q].w)
                         : "memory");
        }
    }
  }
}



// Histogram of one chunk, and for the CTA that finishes last (an atomic ticket, nobody waits)
// the scan: counts[e], offsets (exclusive scan over experts) and blk_base[c][e] = offsets[e] +
// counts of chunks before c. The 256 threads are (expert, chunk group) pairs so the chunk tables
// are summed in parallel; every sum runs in a fixed order, so results do not depend on timing.
// `done` is zero before the call and is reset to zero by the last CTA.
__global__ void __launch_bounds__(kChunk)
dispatch_count_scan_kernel(const int32_t* __restrict__ idx, int A, int E, int nb, int cap, int neg_dropped,
                           int32_t* __restrict__ blk_counts, int32_t* __restrict__ blk_base,
                           int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int* status, int* done) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int sm[];
  int* hist = sm;            // [E]
  int* tot = hist + E;       // [E]
  int* offs = tot + E;       // [E + 1]
  int* sgrp = offs + E + 1;  // [kChunk]: per (group, expert) sums, then their exclusive prefixes
  __shared__ int s_last;
  __shared__ int warp_tot[kChunk / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kChunk) hist[e] = 0;
  __syncthreads();
  const int a = blockIdx.x * kChunk + tid;
  if (a < A) {
    const int e = idx[a];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else if (!(neg_dropped && e < 0)) record_error(status, MOE_ERR_DEVICE_CHECK, a);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kChunk) blk_counts[(size_t)blockIdx.x * E + e] = hist[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(done, 1) == nb - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // pass 1: totals per expert; for E <= 256, G groups of consecutive chunks per expert
  const int width = E < kChunk ? E : kChunk;
  const int G = E < kChunk ? kChunk / E : 1;
  const int L = (nb + G - 1) / G;
  const int g = tid / width;
  for (int e0 = 0; e0 < E; e0 += width) {
    const int e = e0 + tid % width;
    const bool valid = g < G && e < E;
    int sum = 0;
    if (valid)
      for (int c = g * L; c < nb && c < (g + 1) * L; ++c) sum += __ldcg(blk_counts + (size_t)c * E + e);
    if (g < G) sgrp[g * width + tid % width] = sum;
    __syncthreads();
    if (tid < width && e0 + tid < E) {
      int run = 0;
      for (int gg = 0; gg < G; ++gg) {
        const int v = sgrp[gg * width + tid];
        sgrp[gg * width + tid] = run;
        run += v;
      }
      tot[e0 + tid] = run;
    }
    __syncthreads();
  }
  // exclusive scan of the totals over experts (thread t owns experts 4t .. 4t+3)
  int loc[4], local = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * tid + j;
    loc[j] = e < E ? (cap > 0 ? min(tot[e], cap) : tot[e]) : 0;  // rows kept per expert
    local += loc[j];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += warp_tot[w];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * tid + j;
    if (e < E) {
      offs[e] = run;
      counts[e] = loc[j];
      offsets[e] = run;
    }
    run += loc[j];
  }
  if (tid == kChunk - 1) offsets[E] = run;
  __syncthreads();
  // pass 2: per-chunk bases (E <= 256: the group prefixes are still in sgrp; E > 256: one group)
  for (int e0 = 0; e0 < E; e0 += width) {
    const int e = e0 + tid % width;
    if (g < G && e < E) {
      int r = offs[e] + (E < kChunk ? sgrp[g * width + tid % width] : 0);
      for (int c = g * L; c < nb && c < (g + 1) * L; ++c) {
        blk_base[(size_t)c * E + e] = r;
        r += __ldcg(blk_counts + (size_t)c * E + e);
      }
    }
  }
  if (tid == 0) *done = 0;
}

// Rerouting at capacity (aicoding/6a320eef §3.2: a token that meets a full expert queue goes to the
// next-best expert; csdn/6a919c0d §3.2: the retry of a dropped request). One warp walks the T*k
// assignments in row-major (t, j) order, 32 at a time. rank_idx / rank_p hold each token's R best
// experts and their probabilities, best first; slot j of token t asks for rank j. While no assignment
// of the group meets a full expert, the whole group is placed at once (ranks among equal experts from
// __match_any_sync, as in the dispatch); at the first that does, the ones before it are final, and
// that one takes the next entry of its token's ranking (ranks k .. R-1, each tried once per token)
// whose expert has room, or is dropped (-1) when none has; then the group goes on from the next lane.
// The result is exactly the sequential rule: held[e] counts the assignments placed on e so far.
// An expert index outside [0, E) is recorded (MOE_ERR_DEVICE_CHECK, detail = assignment) and dropped.
__global__ void __launch_bounds__(32)
dispatch_reroute_kernel(const int32_t* __restrict__ rank_idx, const float* __restrict__ rank_p, int T, int k,
                        int R, int E, int cap, int32_t* __restrict__ final_idx, float* __restrict__ final_gate,
                        int* status) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int held[];  // [E]
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) held[e] = 0;
  __syncwarp();
  const int A = T * k;
  int cur_t = -1, cur_next = 0;  // the token whose ranking is being walked, and its next entry (uniform)
  for (int base = 0; base < A; base += 32) {
    const int a = base + lane;
    const bool valid = a < A;
    const int t = valid ? a / k : 0, j = valid ? a % k : 0;
    int e = valid ? rank_idx[(size_t)t * R + j] : -1;
    if (valid && (e < 0 || e >= E)) {
      record_error(status, MOE_ERR_DEVICE_CHECK, a);
      e = -1;
    }
    const float g = valid ? rank_p[(size_t)t * R + j] : 0.f;
    int start = 0;
    while (start < 32) {
      const bool mine = lane >= start && e >= 0;
      const unsigned peers = __match_any_sync(0xffffffffu, mine ? e : -1 - lane);
      const int before = __popc(peers & ((1u << lane) - 1u));  // earlier lanes of this round, same expert
      const bool fits = mine && held[e] + before < cap;
      const unsigned over = __ballot_sync(0xffffffffu, mine && !fits);
      const int first = over ? __ffs(over) - 1 : 32;
      __syncwarp();  // every lane has read held[] before it changes
      if (valid && lane >= start && lane < first) {
        final_idx[a] = e;
        final_gate[a] = e >= 0 ? g : 0.f;
        if (e >= 0) atomicAdd(&held[e], 1);
      }
      __syncwarp();
      if (first == 32) break;
      const int af = base + first;
      const int tf = af / k;
      if (tf != cur_t) {
        cur_t = tf;
        cur_next = k;
      }
      int tgt = -1;
      float tg = 0.f;
      while (cur_next < R) {
        const int c = rank_idx[(size_t)tf * R + cur_next];
        const float cp = rank_p[(size_t)tf * R + cur_next];
        ++cur_next;
        if (c >= 0 && c < E && held[c] < cap) {
          tgt = c;
          tg = cp;
          break;
        }
      }
      __syncwarp();
      if (lane == 0) {
        final_idx[af] = tgt;
        final_gate[af] = tg;
        if (tgt >= 0) held[tgt] += 1;
      }
      __syncwarp();
      start = first + 1;
    }
  }
}

}  // namespace

// Two launches with programmatic dependent launch: count + scan, then scatter + gather.
cudaError_t launch_dispatch_fast(const void* x, const int32_t* idx, const float* gate, int T, int d, int E, int k,
                                 int dt, int cap, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                 int32_t* row_of, float* row_gate, void* x_perm, int32_t* blk_counts,
                                 int32_t* blk_base, int* status, int* done, cudaStream_t s, int neg_dropped) {
  const int A = T * k;
  if (A == 0) {  // no assignments: every count and offset is zero
    cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    return err;
  }
  const int nb = (A + kChunk - 1) / kChunk;
  const size_t cs_smem = (size_t)(3 * E + 1 + kChunk) * sizeof(int);
  cudaError_t err = launch_pdl(dispatch_count_scan_kernel, dim3(nb), dim3(kChunk), cs_smem, s, idx, A, E, nb, cap,
                               neg_dropped, blk_counts, blk_base, counts, offsets, status, done);
  if (err != cudaSuccess) return err;
  // scatter + gather: enough CTAs per chunk that the row copy is spread over the SMs
  const size_t sc_smem = (size_t)(kWarpsPerChunk * E + kChunk) * sizeof(int);
  err = cudaFuncSetAttribute(dispatch_scatter_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sc_smem);
  if (err != cudaSuccess) return err;
  const size_t elem = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const int vec_per_row = (int)((size_t)d * elem / 16);
  int split = (2 * device_sm_count() + nb - 1) / nb;
  if (split > 8) split = 8;
  if (split < 1) split = 1;
  return launch_pdl(dispatch_scatter_gather_kernel, dim3(nb * split), dim3(kChunk), sc_smem, s, idx, gate, A, k, E,
                    (const int32_t*)blk_base, (const int32_t*)offsets, cap, split, (const int4*)x, vec_per_row,
                    row_of, perm_token, row_gate, (int4*)x_perm);
}

cudaError_t launch_dispatch_reroute(const void* x, const int32_t* rank_idx, const float* rank_p, int T, int d, int E,
                                    int k, int R, int dt, int cap, int32_t* final_idx, float* final_gate,
                                    int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* row_of,
                                    float* row_gate, void* x_perm, int32_t* blk_counts, int32_t* blk_base, int* status,
                                    int* done, cudaStream_t s) {
  if ((long long)T * k > 0) {
    cudaError_t err = launch_pdl(dispatch_reroute_kernel, dim3(1), dim3(32), (size_t)E * sizeof(int), s, rank_idx,
                                 rank_p, T, k, R, E, cap, final_idx, final_gate, status);
    if (err != cudaSuccess) return err;
  }
  return launch_dispatch_fast(x, final_idx, final_gate, T, d, E, k, dt, 0, counts, offsets, perm_token, row_of,
                              row_gate, x_perm, blk_counts, blk_base, status, done, s, 1);
}

cudaError_t launch_dispatch_from_hist(const void* x, const int32_t* idx, const float* gate, int T, int d, int E,
                                      int k, int dt, int cap, const int32_t* blk_counts, int32_t* counts,
                                      int32_t* offsets, int32_t* perm_token, int32_t* row_of, float* row_gate,
                                      void* x_perm, cudaStream_t s) {
  const int A = T * k;
  if (A == 0 || E > kChunk) return cudaErrorInvalidValue;
  const int nb = (A + kChunk - 1) / kChunk;
  const size_t smem = (size_t)(kWarpsPerChunk * E + kChunk + 2 * E) * sizeof(int);
  cudaError_t err = cudaFuncSetAttribute(dispatch_from_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const size_t elem = dt == MOE_DTYPE_BF16 ? 2 : 4;
  const int vec_per_row = (int)((size_t)d * elem / 16);
  int split = (2 * device_sm_count() + nb - 1) / nb;
  if (split > 8) split = 8;
  if (split < 1) split = 1;
  return launch_pdl(dispatch_from_hist_kernel, dim3(nb * split), dim3(kChunk), smem, s, idx, gate, A, k, E, nb,
                    blk_counts, cap, split, (const int4*)x, vec_per_row, counts, offsets, row_of, perm_token,
                    row_gate, (int4*)x_perm);
}

}  // namespace moe
