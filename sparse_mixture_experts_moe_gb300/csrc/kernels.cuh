// Host-side launchers of the layer's kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Launch with programmatic stream serialisation (see griddep_wait in common.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Dispatch processes the T*k assignments in chunks of this many (one CTA each).
constexpr int kDispatchChunk = 256;

// status (nullable) receives a device-side wait timeout of the tensor-core router.
// Routing statistics written by the router launch (part == nullptr: none). part: one row of
// 2E + 1 words per CTA of the launch (at most ceil(T / 8) CTAs); out: 2E + 2 floats; ticket: a
// word that is zero before the launch and that the last CTA resets to zero.
struct RouterStats {
  float* part;
  float* out;
  int* ticket;
  // Optional (nullptr: none): the dispatch histogram of each 128-token tile, written by the
  // tensor-core routers as hist[tile][e] (with k = 2 a tile's assignments are one dispatch chunk).
  int32_t* hist;
};
constexpr int kRouterStatsTokensPerCta = 8;  // fewest tokens any router CTA owns

// *wrote_hist (nullable) tells whether st.hist was filled (only the tensor-core routers do it).
cudaError_t launch_router_topk(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                               int dt, int flags, const RouterStats& st, int32_t* idx, float* gate, int* status,
                               uint64_t timeout_ns, cudaStream_t s, bool* wrote_hist = nullptr);

// Dispatch in two launches (count + scan, then scatter + gather). blk_counts / blk_base:
// [ceil(A / kDispatchChunk), E] int32 scratch each; `done` is an int that is zero before the call and
// zero again after it (the workspace header); status (nullable) receives out-of-range indices.
// Scatter + gather from per-chunk histograms already in blk_counts (written by the router for
// k = 2): every CTA rebuilds totals, offsets and its chunk's bases itself; CTA 0 writes counts and
// offsets. No count kernel.
cudaError_t launch_dispatch_from_hist(const void* x, const int32_t* idx, const float* gate, int T, int d, int E,
                                      int k, int dt, int cap, const int32_t* blk_counts, int32_t* counts,
                                      int32_t* offsets, int32_t* perm_token, int32_t* row_of, float* row_gate,
                                      void* x_perm, cudaStream_t s);
// cap > 0: each expert keeps its first cap assignments in (t, j) order, the rest get row -1.
cudaError_t launch_dispatch_fast(const void* x, const int32_t* idx, const float* gate, int T, int d, int E, int k,
                                 int dt, int cap, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                 int32_t* row_of, float* row_gate, void* x_perm, int32_t* blk_counts,
                                 int32_t* blk_base, int* status, int* done, cudaStream_t s, int neg_dropped = 0);
// Rerouting at capacity: one warp places the T*k assignments in (t, j) order, sending an assignment that
// meets a full expert to the next entry of its token's ranking rank_idx[t, k..R-1] with room (or
// dropping it: final_idx -1), then the two-launch dispatch of final_idx / final_gate, a negative index
// being an assignment with no row.
cudaError_t launch_dispatch_reroute(const void* x, const int32_t* rank_idx, const float* rank_p, int T, int d, int E,
                                    int k, int R, int dt, int cap, int32_t* final_idx, float* final_gate,
                                    int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* row_of,
                                    float* row_gate, void* x_perm, int32_t* blk_counts, int32_t* blk_base, int* status,
                                    int* done, cudaStream_t s);

cudaError_t launch_combine(const void* y_perm, const int32_t* row_of, int T, int d, int k, int dt, void* out,
                           cudaStream_t s);

// Expert FFN halves. stage 1: out = GeLU(a W1[e]) (N = F, K = d);
// stage 2: out = row_gate * (a W2[e]) (N = d, K = F).
struct FfnArgs {
  const void* a;          // [rows, K], or (a_rows != nullptr) row r is a[a_rows[r]]
  const void* w;          // [E, K, N]
  const int32_t* offsets; // [E+1]
  const float* row_gate;  // [rows] (stage 2)
  void* out;              // [rows, N]
  int rows, K, N, E, dt, stage;
  int* status;
  uint64_t timeout_ns;
  const int32_t* a_rows;  // nullable row map of `a` (weight-streaming kernels only)
  int max_rows_per_expert;  // an upper bound (T: a token's k experts are distinct); 0: unknown
};
cudaError_t launch_ffn_simt(const FfnArgs& a, cudaStream_t s);

// Block-quantised weights (quant.cu): codes in 16-byte tiles of 8 columns x 16/bits k-rows,
// (scale, min) per 64 x 64 block.
struct QFfnArgs {
  const void* a;          // [rows, K] bf16
  const void* codes;      // INT8: [E, N/64, K/16, 2, 32, 16] bytes; INT4: [E, N/64, K/16, 32, 4] words
  const float* scale_min; // [E, K/64, N/64] (scale, min) pairs
  const int32_t* offsets; // [E+1]
  const float* row_gate;  // [rows] (stage 2)
  void* out;              // [rows, N]: bf16 (stage 1) or fp32 (stage 2)
  int rows, K, N, E, bits, stage;
  const int32_t* a_rows;    // nullable: row r of `a` is a[a_rows[r]]
  int max_rows_per_expert;  // an upper bound (T: a token's k experts are distinct); 0: unknown
  int* status;              // nullable: where a bounded device wait that gave up is recorded
  uint64_t timeout_ns;
};
cudaError_t launch_quantize(const void* w, int K, int N, int E, int dt, int bits, void* codes, float* scale_min,
                            cudaStream_t s);
cudaError_t launch_ffn_stream_q(const QFfnArgs& a, cudaStream_t s);
cudaError_t launch_ffn_stream(const FfnArgs& a, cudaStream_t s);
// Returns cudaErrorNotSupported when no tensor-map encoder is available.
cudaError_t launch_ffn_tensor(const FfnArgs& a, cudaStream_t s);
// CTA-pair version (cta_group::2, 256-row tiles) for experts with many rows.
cudaError_t launch_ffn_tensor_pair(const FfnArgs& a, cudaStream_t s);
// CTA-pair version with the product transposed (features on M, rows on N in steps of 16).
cudaError_t launch_ffn_tensor_t(const FfnArgs& a, cudaStream_t s);

cudaError_t launch_selftest_wait(int* status, uint64_t timeout_ns, cudaStream_t s);

// Router + dispatch for T <= 8 in one launch (router_small.cu): routing arrays only, no x_perm.
// partials: (#clusters) x T x E floats of scratch; ticket: zero before, reset to zero after.
bool route_small_ok(int T, int d, int E, int k, int dt, size_t partial_bytes_avail);
cudaError_t launch_route_small(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                               int renorm, int cap, float* partials, int* ticket, int32_t* idx, float* gate,
                               int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* row_of,
                               float* row_gate, cudaStream_t s);

// Router on the tensor cores (bf16, E <= 256, E % 8 == 0). Returns cudaErrorNotSupported otherwise.
cudaError_t launch_router_tc(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                             int renorm, const RouterStats& st, int32_t* idx, float* gate, int* status,
                             uint64_t timeout_ns, cudaStream_t s);

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time driver dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
// Tiled tensor map with 128-byte swizzle and zero fill outside the tensor.
bool encode_tmap(EncodeTiledFn enc, CUtensorMap* m, CUtensorMapDataType type, const void* ptr, int rank,
                 const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box);
// The same without swizzle: the shared-memory box is plain row-major.
bool encode_tmap_plain(EncodeTiledFn enc, CUtensorMap* m, CUtensorMapDataType type, const void* ptr, int rank,
                       const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box);

int device_sm_count();
// The current device's L2 size in bytes. A streaming GEMM whose touched weights (at most rows experts)
// come to less than three L2s copies them at L2 evict-first priority, so that what the step reads
// again (the router's weights, the activations) stays in L2: one-token steps ran 2-3% faster. With
// 8 tokens (0.5-2 GB a launch) the bf16 GEMM ran 3% slower with the hint, so larger launches go
// without it.
size_t device_l2_bytes();
inline bool stream_evict_first(long long rows, int E, long long K, long long N, int bits) {
  const double touched = (double)(rows < E ? rows : E) * (double)K * (double)N * bits / 8.0;
  return touched < 3.0 * (double)device_l2_bytes();
}

}  // namespace moe
