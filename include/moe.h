/*
 * moe.h — C ABI of the GB300 (sm_103a) sparse top-k Mixture-of-Experts FFN layer, forward pass.
 *
 * The layer, for T tokens x[T, d], E experts, top-k and expert width d_ff = F:
 *   logits = x W_r (+ b_r), p = softmax(logits), the k largest logits pick the
 *   experts (lower index wins a tie), gate = p of each chosen expert,
 *   out[t] = sum_j gate[t, j] * W2_e (GeLU(W1_e x[t])) over the k chosen experts e.
 *
 * Pages (none has a title of its own; each is named by its address):
 *   csdn/6a919c0d     devpress.csdn.net/awstech/6a919c0d2b83d06f0ec6f601.html
 *   csdn/6a462027     devpress.csdn.net/awstech/6a46202710ee7a33f285c5a4.html
 *   aicoding/6a320eef aicoding.csdn.net/6a320eef10ee7a33f27e52b3.html
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers, allocated and owned by the caller;
 *    the library never allocates, frees or synchronises (moe_get_device_status
 *    alone synchronises its stream). Tensors are dense row-major and 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every call only enqueues work on it and returns.
 *  - Element type `dt`: MOE_DTYPE_F32 (x, W_r, W1, W2, x_perm, h and out in fp32) or
 *    MOE_DTYPE_BF16 (those tensors in bf16, accumulation in fp32). Router bias, gates,
 *    row gates and the gated expert outputs y_perm are always fp32 (so the k-way sum of
 *    the combine rounds once); indices are int32.
 *  - Limits: 0 <= T (T = 0 is a no-op), 1 <= k <= min(E, 8), E <= 1024,
 *    d and F multiples of 8 and >= 8, T*k < 2^31, T*max(d,F) < 2^40.
 *  - Host-side argument checks fail with MOE_ERR_INVALID_ARG before anything is
 *    launched. A failed launch returns MOE_ERR_CUDA. Checks made on the device
 *    (an expert index out of range, a wait that timed out) do not fault: they
 *    record the first error in the workspace's status word, skip the offending
 *    item, and are read back with moe_get_device_status.
 *  - Workspace: caller-allocated device scratch of at least
 *    moe_workspace_bytes(T, d, F, E, k, dt) bytes (one such block serves every
 *    call with those sizes), 256-byte aligned, prepared once with
 *    moe_workspace_init. Calls that share a workspace must not overlap in time.
 *  - The library holds no global mutable state; distinct workspaces may be used
 *    from distinct host threads.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* bad sizes, null pointer, misalignment, workspace too small */
  MOE_ERR_UNSUPPORTED = 2,   /* valid arguments this build has no kernel for (e.g. a path forced on the wrong dtype) */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_CHECK = 4,  /* a device-side range check failed (see moe_get_device_status) */
  MOE_ERR_DEVICE_TIMEOUT = 5 /* a bounded device-side wait gave up */
} moe_status;

typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

/* Kernel family for the expert FFN (a3, a4). AUTO picks, for bf16: STREAM with at most 256 routed
 * rows; otherwise TENSOR_T when the GEMM has at least three 256-row x 256-feature items per resident
 * CTA pair (rows assumed evenly spread over the experts), else TENSOR; SIMT for fp32. TENSOR_PAIR
 * is available on request (measured slower). */
typedef enum {
  MOE_PATH_AUTO = 0,
  MOE_PATH_TENSOR = 1,      /* tcgen05/TMEM grouped GEMM fed by TMA, 128x256 tiles per CTA (bf16 only) */
  MOE_PATH_STREAM = 2,      /* weight-streaming column-slab kernel for few rows per expert (bf16 only) */
  MOE_PATH_SIMT = 3,        /* CUDA-core tiled grouped GEMM (fp32 and bf16) */
  MOE_PATH_TENSOR_PAIR = 4, /* tcgen05 cta_group::2 on CTA pairs, 256x256 tiles (bf16 only) */
  MOE_PATH_TENSOR_T = 5     /* tcgen05 cta_group::2 with the product transposed: 256 output features x
                               up to 256 rows per pair tile, rows rounded up to 16 (bf16 only) */
} moe_path;
/* The family AUTO runs for an expert GEMM of T*k routed rows, E experts and N output columns
 * (N = d_ff for expert_up, d for expert_down); -1 on bad arguments. Host only. */
int moe_ffn_path(int T, int k, int E, int N, moe_dtype dt);
/* Kernel launches of one moe_forward_ex call with these arguments (router_stats: nonzero when a
 * statistics output is passed): 4 for at most 8 bf16 tokens with weight-streaming GEMMs (router
 * and dispatch in one launch, E % 8 == 0, no statistics), 5 with top-2 and the tensor-core router
 * (the router writes the dispatch histograms), 6 otherwise (router, dispatch count + scatter, two
 * expert GEMMs, combine); 0 for T = 0; -1 on bad arguments. moe_forward_q follows the same rules
 * with weight-streaming GEMMs. Host only: nothing is launched. */
int moe_forward_launches(int T, int d, int F, int E, int k, moe_dtype dt, moe_path path, int router_stats);

/* ---------------------------------------------------------------------------------------------
 * moe_router_topk — router GEMM, softmax and deterministic top-k, fused in one kernel: bf16 layers
 *   compute a 128-token tile's logits on the tensor cores and give each token to one epilogue
 *   thread for softmax and top-k; other layers use a CUDA-core kernel.
 *   csdn/6a919c0d §2.2 steps 1-4 (single linear router with one output per expert, softmax,
 *   keep the k most confident experts, weights = their confidences); aicoding/6a320eef §3.2
 *   (h x W_router, W_router is d x E; Softmax; top-2; weights = the p values); csdn/6a919c0d
 *   §4.2 (stabilise with the maximum logit).
 * In:  x [T, d] (dt), w_r [d, E] (dt), b_r [E] fp32 or NULL (added to the logits).
 * Out: topk_idx [T, k] int32, topk_gate [T, k] fp32. Slot j holds the (j+1)-th largest logit;
 *      equal logits go to the lower expert index. gate = softmax probability (fp32 logits,
 *      fp32 softmax), not renormalised over the k experts.
 * Kernels: bf16 with E <= 256 and E % 8 == 0 computes the logits on the tensor cores (tcgen05,
 *      fp32 accumulation in TMEM), one token per epilogue thread; other layers use a CUDA-core
 *      kernel (fp32 FMA). Both select on fp32 logits.
 * Errors: MOE_ERR_INVALID_ARG on bad sizes/pointers. This call keeps no status word (it has no
 *      workspace); within moe_forward a timed-out device wait is reported through the workspace.
 */
moe_status moe_router_topk(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                           moe_dtype dt, int32_t* topk_idx, float* topk_gate, void* stream);

/* Router flags (moe_router_topk_ex, moe_forward_ex; 0 = the layer as defined above).
 * MOE_GATES_RENORMALISE: gate[t, j] = softmax over the k chosen logits only, exp(l_j - m) /
 *   sum_i exp(l_i - m) over the chosen i (hotelren/2927663 §4.3, top-k on the logits, then a
 *   softmax of the selected values); the gates of a token sum to one. */
enum { MOE_GATES_RENORMALISE = 1 };
/* MOE_CAPACITY_REROUTE (moe_forward_ex, moe_forward_q only; needs capacity > 0, the raw gates and no
 *   router_stats): an assignment whose expert already holds `capacity` rows is rerouted as
 *   moe_dispatch_reroute does, within each token's min(E, 8) best experts, instead of dropped. The
 *   topk_idx / topk_gate outputs then hold the expert that took each slot (-1 when dropped) and its
 *   softmax probability; the layer launches the router (for the token's ranking), the rerouting
 *   kernel and the two-kernel dispatch in place of its usual routing launches. */
enum { MOE_CAPACITY_REROUTE = 2 };
moe_status moe_router_topk_ex(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                              moe_dtype dt, int flags, int32_t* topk_idx, float* topk_gate, void* stream);

/* moe_router_topk_stats — moe_router_topk_ex that also writes the batch's routing statistics,
 *   computed inside the router kernel beside the top-k. p is the full softmax over the E experts
 *   (whatever the gates are); `stats` is a device array of MOE_ROUTER_STATS_LEN(E) floats:
 *     stats[e]         (1/T) sum_t p[t, e]: soft load of expert e (csdn/6a462027 §4.2, the
 *                      probabilities summed over the batch divided by the token count);
 *     stats[E + e]     #{(t, j) : idx[t, j] = e} / (T k): expert e's share of the assignments;
 *     stats[2E]        sum_e (stats[E + e] - 1/E)^2: the load-balancing term before its weight
 *                      lambda (aicoding/6a320eef §3.2; csdn/6a462027 §3.1);
 *     stats[2E + 1]    (1/T) sum_t -sum_e p[t, e] ln p[t, e]: mean router entropy in nats
 *                      (aicoding/6a320eef §5.2).
 *   Partial sums per CTA go to the workspace (moe_workspace_bytes with any d, F covers them);
 *   the CTA that finishes last reduces them in a fixed order, so the values are reproducible.
 *   T = 0: nothing is written. A workspace that is too small or NULL: MOE_ERR_INVALID_ARG. */
#define MOE_ROUTER_STATS_LEN(E) (2 * (E) + 2)
moe_status moe_router_topk_stats(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                                 moe_dtype dt, int flags, int32_t* topk_idx, float* topk_gate, float* stats,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_dispatch — per-expert histogram, exclusive scan, stable permutation and row gather.
 *   csdn/6a462027 §4.2 steps 4-5 (find the selected experts, scatter each expert's tokens to it).
 * In:  x [T, d] (dt), topk_idx [T, k] int32, topk_gate [T, k] fp32.
 * Out: counts [E] int32 (assignments per expert), offsets [E+1] int32 (exclusive scan,
 *      offsets[E] = T*k), row_of [T, k] int32 (row of assignment (t, j)), perm_token [T*k] int32
 *      (token of each row), row_gate [T*k] fp32 (gate of each row), x_perm [T*k, d] (dt, row r is
 *      x[perm_token[r]]). Within an expert, rows follow row-major (t, j) order; every output is
 *      exact (bit-reproducible).
 * Workspace: status word and per-block count tables.
 * Errors: an index outside [0, E) records MOE_ERR_DEVICE_CHECK (detail = flat assignment index)
 *      and that assignment is dropped from every output (its row_of entry is -1).
 */
moe_status moe_dispatch(const void* x, const int32_t* topk_idx, const float* topk_gate, int T, int d, int E,
                        int k, moe_dtype dt, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                        int32_t* row_of, float* row_gate, void* x_perm, void* workspace, size_t ws_bytes,
                        void* stream);

/* moe_dispatch_ex — moe_dispatch with an expert capacity (aicoding/6a320eef §3.2: capacity =
 *   ceil(batch * k / num_experts * capacity_factor); an expert that is full diverts further tokens).
 *   capacity > 0: each expert keeps its first `capacity` assignments in row-major (t, j) order and the
 *   later ones are dropped (row_of = -1, no row, no contribution to the output); counts[e] is the
 *   number kept. capacity = 0: no limit (moe_dispatch). Negative: MOE_ERR_INVALID_ARG.
 * moe_capacity — ceil(T * k / E * cf) as an int, -1 on bad arguments. */
moe_status moe_dispatch_ex(const void* x, const int32_t* topk_idx, const float* topk_gate, int T, int d, int E,
                           int k, moe_dtype dt, int capacity, int32_t* counts, int32_t* offsets,
                           int32_t* perm_token, int32_t* row_of, float* row_gate, void* x_perm, void* workspace,
                           size_t ws_bytes, void* stream);
int moe_capacity(int T, int k, int E, double cf);

/* ---------------------------------------------------------------------------------------------
 * moe_dispatch_reroute — dispatch with an expert capacity that reroutes instead of dropping.
 *   aicoding/6a320eef §3.2: when the chosen expert's queue is already at capacity, the token is
 *   rerouted to the next-best expert; csdn/6a919c0d §3.2: a retry sends a dropped request to the
 *   next-best expert.
 * The T*k assignments queue in row-major (t, j) order. Slot j of token t asks for rank_idx[t, j];
 *   if that expert already holds `capacity` assignments, the slot takes the next entry of the token's
 *   ranking rank_idx[t, k], rank_idx[t, k+1], ... (each entry tried at most once per token) whose
 *   expert has room, and with none left it is dropped. The slot's gate is rank_gate at the rank that
 *   took it (the probability of that expert).
 * In:  x [T, d] (dt), rank_idx [T, R] int32 and rank_gate [T, R] fp32: each token's R best experts,
 *      best first, distinct (moe_router_topk with k = R gives them); k <= R <= E; capacity >= 1.
 * Out: final_idx [T, k] int32 (the expert that took each slot, -1 if dropped), final_gate [T, k]
 *      fp32 (0 if dropped), then counts, offsets, perm_token, row_of, row_gate, x_perm exactly as
 *      moe_dispatch does for final_idx / final_gate (a dropped slot has row_of -1 and no row; rows
 *      within an expert keep the (t, j) order; offsets[E] = the rows placed).
 * Workspace: status word, the dispatch ticket and the per-chunk count tables (moe_workspace_bytes).
 * One warp places the assignments (a single CTA); then two launches as moe_dispatch. An index outside
 *   [0, E) in the first k columns is recorded (MOE_ERR_DEVICE_CHECK, detail = assignment) and dropped.
 */
moe_status moe_dispatch_reroute(const void* x, const int32_t* rank_idx, const float* rank_gate, int T, int d, int E,
                                int k, int R, moe_dtype dt, int capacity, int32_t* final_idx, float* final_gate,
                                int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* row_of,
                                float* row_gate, void* x_perm, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_dispatch_noalloc — moe_dispatch without a workspace, for callers that cannot provide device
 *   scratch memory: a plugin that its host framework gives only input and output buffers (the
 *   framework owns all device memory through its own pool), or a latency-critical loop that must
 *   not call cudaMalloc, which can block and synchronise the device. The pages have no counterpart
 *   of this call; it exists for such callers only.
 * Same inputs, outputs and results as moe_dispatch (bit for bit), by the same two launches. The
 *   per-chunk count tables (and the count kernel's one-word ticket) live in a fixed array of
 *   1 MiB + 256 bytes inside the library's own device memory, one copy per GPU that loads the
 *   library, held until the process exits. Limit: ceil(T*k / 256) * E <= 131072 (for example
 *   T*k <= 262144 with E = 128, T*k <= 32768 with E = 1024); larger sizes return
 *   MOE_ERR_INVALID_ARG before anything is launched. Nothing is allocated and nothing is freed.
 * Every call looks up the array's device address on the current device (host code cannot use the
 *   array's name as a pointer); the first lookup on a device may load the library's device code,
 *   so make the first call on each device before any stream capture.
 * Every call on a device shares the array and leaves its contents behind. Each call clears the
 *   ticket (a 4-byte memset on `stream`) and rewrites the tables it reads, but calls whose kernels
 *   overlap on the GPU (e.g. on two streams at once) race on it: issue them in order on one stream.
 * An index outside [0, E) is dropped (row_of entry -1, offsets[E] < T*k); no status word is kept.
 */
moe_status moe_dispatch_noalloc(const void* x, const int32_t* topk_idx, const float* topk_gate, int T, int d,
                                int E, int k, moe_dtype dt, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                int32_t* row_of, float* row_gate, void* x_perm, void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_expert_up — grouped GEMM1 with the GeLU epilogue:  h[r, :] = GeLU(x_perm[r, :] W1[e])
 * for every row r in expert e's range [offsets[e], offsets[e+1]).
 *   csdn/6a462027 §3.2 (homogeneous d -> d_ff -> d GELU experts with their own W1, W2) and §4.2
 *   step 6 ("in practice a grouped GEMM"); GeLU is the erf form.
 * In:  x_perm [T*k, d] (dt), w1 [E, d, F] (dt, expert-major, row-major per expert), offsets [E+1].
 * Out: h [T*k, F] (dt). bf16: fp32 accumulation, GeLU in fp32, one round-to-nearest-even.
 * Workspace: status word.
 */
moe_status moe_expert_up(const void* x_perm, const void* w1, const int32_t* offsets, int T, int d, int F, int E,
                         int k, moe_dtype dt, void* h, void* workspace, size_t ws_bytes, void* stream);
moe_status moe_expert_up_ex(const void* x_perm, const void* w1, const int32_t* offsets, int T, int d, int F,
                            int E, int k, moe_dtype dt, moe_path path, void* h, void* workspace, size_t ws_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_expert_down — grouped GEMM2 with the gate epilogue:  y_perm[r, :] = row_gate[r] * (h[r, :] W2[e]).
 *   csdn/6a919c0d §2.2 step 4 (each expert's output weighted by its confidence).
 * In:  h [T*k, F] (dt), w2 [E, F, d] (dt), offsets [E+1], row_gate [T*k] fp32.
 * Out: y_perm [T*k, d] fp32 (fp32 accumulation, gate multiplied in fp32, no rounding to dt).
 * Workspace: status word.
 */
moe_status moe_expert_down(const void* h, const void* w2, const int32_t* offsets, const float* row_gate, int T,
                           int d, int F, int E, int k, moe_dtype dt, void* y_perm, void* workspace,
                           size_t ws_bytes, void* stream);
moe_status moe_expert_down_ex(const void* h, const void* w2, const int32_t* offsets, const float* row_gate,
                              int T, int d, int F, int E, int k, moe_dtype dt, moe_path path, void* y_perm,
                              void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_grouped_ffn — moe_expert_up then moe_expert_down, with h kept in the workspace.
 * In:  x_perm [T*k, d], w1 [E, d, F], w2 [E, F, d], offsets [E+1], row_gate [T*k].
 * Out: y_perm [T*k, d] fp32.
 */
moe_status moe_grouped_ffn(const void* x_perm, const void* w1, const void* w2, const int32_t* offsets,
                           const float* row_gate, int T, int d, int F, int E, int k, moe_dtype dt, void* y_perm,
                           void* workspace, size_t ws_bytes, void* stream);
moe_status moe_grouped_ffn_ex(const void* x_perm, const void* w1, const void* w2, const int32_t* offsets,
                              const float* row_gate, int T, int d, int F, int E, int k, moe_dtype dt,
                              moe_path path, void* y_perm, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_combine — out[t, :] = sum_{j = 0..k-1} y_perm[row_of[t, j], :], summed in fp32 in slot
 * order j = 0, 1, ..., then rounded once to `dt`, the element type of `out` (round-to-nearest-even
 * for bf16; fp32 keeps the sum as it is).
 *   csdn/6a462027 §4.2 step 7 (sum the expert outputs back per token, "scatter_add").
 * In:  y_perm [T*k, d] fp32, row_of [T, k] int32.  Out: out [T, d] (dt).
 * A row_of entry outside [0, T*k) contributes nothing (dispatch writes -1 for a dropped item).
 */
moe_status moe_combine(const void* y_perm, const int32_t* row_of, int T, int d, int k, moe_dtype dt, void* out,
                       void* stream);

/* ---------------------------------------------------------------------------------------------
 * moe_forward — the whole layer: router_topk, dispatch, expert_up, expert_down, combine.
 * In:  x [T, d], w_r [d, E], b_r [E] or NULL, w1 [E, d, F], w2 [E, F, d].
 * Out: out [T, d] (dt), and optional copies of the routing (NULL: kept in the workspace only):
 *      topk_idx [T, k], topk_gate [T, k], counts [E].
 * moe_forward_ex also takes: the output's element type `out_dt` (e.g. fp32 output of a bf16
 *      layer), the FFN kernel family `path`, `flags` (MOE_GATES_RENORMALISE, MOE_CAPACITY_REROUTE),
 *      an expert `capacity` (as in moe_dispatch_ex, dropping, or rerouting with
 *      MOE_CAPACITY_REROUTE; 0 = no limit) and `router_stats` (NULL, or MOE_ROUTER_STATS_LEN(E)
 *      floats as in moe_router_topk_stats).
 * Kernels (same results as the separate calls; moe_forward_launches gives the count): with top-2 and
 *      the tensor-core router, the router also writes each 128-token tile's expert histogram and the
 *      dispatch is one launch; for at most 8 bf16 tokens with weight-streaming GEMMs (E % 8 == 0, no
 *      statistics) one launch routes and dispatches, and the up-projection reads x through
 *      perm_token (the workspace's x_perm is then not written).
 */
moe_status moe_forward(const void* x, const void* w_r, const float* b_r, const void* w1, const void* w2, int T,
                       int d, int F, int E, int k, moe_dtype dt, void* out, int32_t* topk_idx, float* topk_gate,
                       int32_t* counts, void* workspace, size_t ws_bytes, void* stream);
moe_status moe_forward_ex(const void* x, const void* w_r, const float* b_r, const void* w1, const void* w2,
                          int T, int d, int F, int E, int k, moe_dtype dt, moe_dtype out_dt, moe_path path,
                          int flags, int capacity, void* out, int32_t* topk_idx, float* topk_gate,
                          int32_t* counts, float* router_stats, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Workspace and status.
 * moe_workspace_bytes: bytes of workspace every call with these sizes needs (0 on bad sizes).
 * moe_workspace_init:  clears the status word (async on `stream`); call once after allocating.
 * moe_get_device_status: synchronises `stream`, returns and clears the first device-side error
 *      recorded in the workspace (MOE_OK if none); *detail (nullable) receives its detail value.
 * moe_status_string: static text for a status code.
 */
size_t moe_workspace_bytes(int T, int d, int F, int E, int k, moe_dtype dt);
moe_status moe_workspace_init(void* workspace, size_t ws_bytes, void* stream);
moe_status moe_get_device_status(void* workspace, int32_t* detail, void* stream);
const char* moe_status_string(moe_status s);

/* Self-test of the bounded device wait every pipelined kernel uses: launches one CTA that waits
 * on a barrier nothing will complete, gives up after timeout_us microseconds, records
 * MOE_ERR_DEVICE_TIMEOUT in the workspace and returns; no fault, the context stays usable. */
moe_status moe_selftest_wait_timeout(void* workspace, size_t ws_bytes, int timeout_us, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Block-quantised expert weights (INT4 / INT8) for weight streaming.
 *   csdn/6a462500 §4.3 (64 x 64 blocks, per-block min and max, codes of 4 bits); csdn/6a919c0d
 *   §2.3 (INT4 expert weights halve the bytes moved again; INT8 as the middle tier).
 * Quantisation of each 64 x 64 block of each expert's [K, N] matrix: scale = (max - min) /
 *   (2^bits - 1), code = round((w - min) / scale) in fp32 (correctly rounded subtraction and
 *   division, ties to even), restored as w ~ min + code * scale (|error| <= scale / 2). A block of
 *   equal values has scale 0 and codes 0. bits is 4 or 8; K and N must be multiples of 64.
 * Layout of `codes` (moe_qweight_bytes(K, N, E, bits) bytes, 16-byte aligned), per expert:
 *   INT8: [N/64][K/16][2][32][16] bytes: for each 64-column slab and 16-deep k-block 2p + s (step s
 *   of the 32-deep range p), half h of lane l = 4g + t holds column tiles m = 2h and 2h + 1, 8 bytes
 *   each; byte q of tile m holds (k, column) = (kp, c0), (kp+1, c0), (kp, c1), (kp+1, c1), (kp+2, c0),
 *   (kp+3, c0), (kp+2, c1), (kp+3, c1) for q = 0..7, with kp = 32p + 8t + 4s, c0 = 16m + g,
 *   c1 = c0 + 8 (the order of an m16n8k16 fp16 A fragment, with k numbered within each 32-deep range
 *   so that one lane's activations for the range's two steps are 8 consecutive values).
 *   INT4: [N/64][K/16][32][4] 32-bit words: for each 64-column slab and 16-deep k-block 4b + j
 *   (step j of the 64-deep block b), lane l = 4g + t holds 4 words; word m covers columns
 *   c0 = 16m + g and c1 = c0 + 8 at k-rows kp .. kp+3, kp = 64b + 16t + 4j, its nibble i
 *   (bits 4i..4i+3) holding (k, column) = (kp, c0), (kp, c1), (kp+2, c0), (kp+2, c1), (kp+1, c0),
 *   (kp+1, c1), (kp+3, c0), (kp+3, c1) for i = 0..7 (the order of an m16n8k16 A fragment, decoded
 *   two values per instruction, with k numbered within each 64-deep block so that one lane's
 *   activations for the block's four steps are 16 consecutive values).
 * Layout of `scale_min` (moe_qscale_bytes(K, N, E) bytes, 8-byte aligned): fp32 pairs
 *   (scale, min), [E][K/64][N/64].
 * moe_quantize_weights: w [E, K, N] (bf16 or fp32) -> codes, scale_min on the device.
 * moe_expert_up_q / moe_expert_down_q: moe_expert_up / moe_expert_down (bf16 activations; h bf16,
 *   y_perm fp32) reading quantised W1 [E, d, F] / W2 [E, F, d]; weight-streaming kernel for any
 *   number of rows (built for decode batches). moe_forward_q: the whole layer with them (x, w_r
 *   bf16; out_dt, flags, capacity, router_stats and the workspace as in moe_forward_ex).
 *   Products: INT4 codes multiply bf16 activations; INT8 codes multiply the activations (x rows,
 *   h) converted to fp16, which is exact for bf16 values of magnitude 2^-14 .. 65504. Smaller values
 *   keep fp16's subnormal spacing (2^-24), and larger ones overflow, so INT8 layers need activations
 *   within fp16's range. Accumulation is fp32 for both.
 *   The streaming kernel's waits on its own copies are bounded: moe_forward_q records a wait that
 *   gave up as MOE_ERR_DEVICE_TIMEOUT in its workspace; moe_expert_up_q / moe_expert_down_q take
 *   no workspace, so there the kernel ends early without a record.
 * Sizes 0 / MOE_ERR_INVALID_ARG on bad sizes, NULL or misaligned pointers. */
size_t moe_qweight_bytes(int K, int N, int E, int bits);
size_t moe_qscale_bytes(int K, int N, int E);
moe_status moe_quantize_weights(const void* w, int K, int N, int E, moe_dtype dt, int bits, void* codes,
                                float* scale_min, void* stream);
moe_status moe_expert_up_q(const void* x_perm, const void* w1_codes, const float* w1_scale_min,
                           const int32_t* offsets, int T, int d, int F, int E, int k, int bits, void* h,
                           void* stream);
moe_status moe_expert_down_q(const void* h, const void* w2_codes, const float* w2_scale_min,
                             const int32_t* offsets, const float* row_gate, int T, int d, int F, int E, int k,
                             int bits, void* y_perm, void* stream);
moe_status moe_forward_q(const void* x, const void* w_r, const float* b_r, const void* w1_codes,
                         const float* w1_scale_min, const void* w2_codes, const float* w2_scale_min, int T, int d,
                         int F, int E, int k, int bits, moe_dtype out_dt, int flags, int capacity, void* out,
                         int32_t* topk_idx, float* topk_gate, int32_t* counts, float* router_stats, void* workspace,
                         size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * CUDA-graph replay of the whole layer.
 * moe_forward_graph_create: records the kernels of one moe_forward_ex call with these arguments
 *      (captured on a private stream; nothing runs) and instantiates them as a CUDA graph. Every
 *      pointer and size is fixed in the graph: each launch runs the full layer again on the
 *      current contents of the same buffers, with one host call instead of one per kernel.
 *      Argument errors are those of moe_forward_ex; *graph is NULL on any error.
 * moe_graph_launch: enqueues one replay on `stream`. The buffers must stay allocated and the
 *      usual stream ordering applies (write x before, read out after, on or after `stream`).
 * moe_graph_destroy: frees the graph (NULL is a no-op).
 * moe_graph_capture_begin / moe_graph_capture_end: the general form. begin returns a private
 *      stream in capture; every moe_* call given that stream is recorded, not run; end stops the
 *      capture, instantiates what was recorded into *graph and destroys the stream (always, also
 *      on error). Use it for moe_forward_q or for a sequence of the separate entry points. */
typedef struct moe_graph_s* moe_graph;
moe_status moe_graph_capture_begin(void** capture_stream);
moe_status moe_forward_graph_create(const void* x, const void* w_r, const float* b_r, const void* w1,
                                    const void* w2, int T, int d, int F, int E, int k, moe_dtype dt,
                                    moe_dtype out_dt, moe_path path, int flags, int capacity, void* out,
                                    int32_t* topk_idx, float* topk_gate, int32_t* counts, float* router_stats,
                                    void* workspace, size_t ws_bytes, moe_graph* graph);
moe_status moe_graph_capture_end(void* capture_stream, moe_graph* graph);
moe_status moe_graph_launch(moe_graph graph, void* stream);
moe_status moe_graph_destroy(moe_graph graph);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
