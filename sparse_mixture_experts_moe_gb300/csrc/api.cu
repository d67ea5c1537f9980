// C ABI of the layer (include/moe.h): host-side validation, workspace layout, path
// choice and step sequencing. Every entry point validates all arguments before it
// makes any CUDA call, so invalid calls fail the same way with or without a GPU.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  return sms;
}

size_t device_l2_bytes() {
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return (size_t)126 << 20;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) return (size_t)126 << 20;
  return (size_t)l2;
}

namespace {

constexpr int kStreamPathMaxRows = 256;
constexpr int kMaxRank = 8;  // the ranking entries the layer routes with when it reroutes at capacity

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline size_t elem_bytes(int dt) { return dt == MOE_DTYPE_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace regions, in this order; each starts on a 256-byte boundary.
struct Layout {
  size_t header, stats_part, blk_counts, blk_base, topk_idx, topk_gate, rank_idx, rank_gate, counts, offsets,
      perm_token, row_of, row_gate, h, x_perm, y_perm, end;
  size_t stats_end, dispatch_end, ffn_end, grouped_end;
  Layout(int T, int d, int F, int E, int k, int dt) {
    const size_t A = (size_t)T * k, eb = elem_bytes(dt);
    const size_t nb = (A + kDispatchChunk - 1) / kDispatchChunk;
    const size_t stat_rows = ((size_t)T + kRouterStatsTokensPerCta - 1) / kRouterStatsTokensPerCta;
    size_t o = 0;
    header = o; o += align256(kWsHeaderBytes);
    stats_part = o; o += align256(stat_rows * (2 * (size_t)E + 1) * 4);
    stats_end = o;
    blk_counts = o; o += align256(nb * E * 4);
    blk_base = o; o += align256(nb * E * 4);
    dispatch_end = o;
    topk_idx = o; o += align256(A * 4);
    topk_gate = o; o += align256(A * 4);
    rank_idx = o; o += align256((size_t)T * kMaxRank * 4);   // rerouting: each token's best experts
    rank_gate = o; o += align256((size_t)T * kMaxRank * 4);
    counts = o; o += align256((size_t)E * 4);
    offsets = o; o += align256((size_t)(E + 1) * 4);
    perm_token = o; o += align256(A * 4);
    row_of = o; o += align256(A * 4);
    row_gate = o; o += align256(A * 4);
    h = o; o += align256(A * F * eb);
    grouped_end = o;
    x_perm = o; o += align256(A * d * eb);
    y_perm = o; o += align256(A * d * 4);
    end = o;
    ffn_end = align256(kWsHeaderBytes);
  }
};

bool sizes_ok(int T, int d, int F, int E, int k, int dt) {
  if (dt != MOE_DTYPE_F32 && dt != MOE_DTYPE_BF16) return false;
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 8 || k > E) return false;
  if (d < 8 || d % 8 != 0 || F < 8 || F % 8 != 0) return false;
  const long long A = (long long)T * k;
  if (A >= (1ll << 31)) return false;
  const long long big = d > F ? d : F;
  if ((long long)T * big > (1ll << 40)) return false;
  return true;
}

uint64_t wait_timeout_ns() {
  const char* s = std::getenv("MOE_WAIT_TIMEOUT_MS");
  long long ms = s != nullptr ? std::atoll(s) : 2000;
  if (ms <= 0) ms = 2000;
  return (uint64_t)ms * 1000000ull;
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The TMA-fed kernels' tensor maps are built by the driver's cuTensorMapEncodeTiled, which needs a
// context current on the calling host thread. The runtime makes the device's primary context current
// on a thread only at the thread's first runtime call that needs one, so a thread whose first CUDA
// work is one of these entry points would encode without a context, and the encode fails. Called
// after validation and before the first launch of every entry point that may encode: when no
// context is current, it selects the thread's current device, which makes its primary context
// current. (cuCtxGetCurrent is a thread-local lookup; nothing else runs when a context is current.)
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
void bind_primary_context() {
  static const CtxGetCurrentFn get = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  CUcontext cur = nullptr;
  if (get != nullptr && get(&cur) == CUDA_SUCCESS && cur != nullptr) return;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) (void)cudaSetDevice(dev);
}

template <typename P>
inline P* at(void* ws, size_t off) { return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off); }

// AUTO: fp32 -> SIMT; bf16 with at most 256 routed rows -> STREAM (weight streaming); otherwise
// the transposed CTA-pair GEMM when it has at least three 256-row items per resident pair (its
// operand feed and ragged-row handling are the better ones, measured faster on e16 up, prefill and
// skew), else the one-CTA GEMM, which balances a few large items better (e16 down: 63 against
// 78 us). The item count assumes the rows spread evenly over the experts: the host does not read
// the device's counts.
moe_path resolve_path(moe_path path, int dt, int rows, int E, int N) {
  if (path != MOE_PATH_AUTO) return path;
  if (dt == MOE_DTYPE_F32) return MOE_PATH_SIMT;
  if (rows <= kStreamPathMaxRows) return MOE_PATH_STREAM;
  const long long active = rows < E ? rows : E;
  const long long rpe = (rows + active - 1) / active;
  const long long items = active * ((rpe + 255) / 256) * ((N + 255) / 256);
  const long long pairs = device_sm_count() / 2;
  return items >= 3 * pairs ? MOE_PATH_TENSOR_T : MOE_PATH_TENSOR;
}

// Layer flags: MOE_GATES_RENORMALISE, MOE_CAPACITY_REROUTE; rerouting needs a capacity, the raw gates
// and no routing statistics.
bool forward_flags_ok(int flags, int capacity, const float* router_stats) {
  if ((flags & ~(MOE_GATES_RENORMALISE | MOE_CAPACITY_REROUTE)) != 0) return false;
  if (flags & MOE_CAPACITY_REROUTE)
    return capacity > 0 && !(flags & MOE_GATES_RENORMALISE) && router_stats == nullptr;
  return true;
}

bool path_ok(moe_path path, int dt) {
  (void)dt;
  return path >= MOE_PATH_AUTO && path <= MOE_PATH_TENSOR_T;
}

moe_status run_ffn_half(moe_path path, FfnArgs& args, cudaStream_t s) {
  path = resolve_path(path, args.dt, args.rows, args.E, args.N);
  if ((path == MOE_PATH_TENSOR || path == MOE_PATH_STREAM || path == MOE_PATH_TENSOR_PAIR ||
       path == MOE_PATH_TENSOR_T) &&
      args.dt != MOE_DTYPE_BF16)
    return MOE_ERR_UNSUPPORTED;
  bind_primary_context();
  cudaError_t e;
  switch (path) {
    case MOE_PATH_TENSOR: e = launch_ffn_tensor(args, s); break;
    case MOE_PATH_TENSOR_PAIR: e = launch_ffn_tensor_pair(args, s); break;
    case MOE_PATH_TENSOR_T: e = launch_ffn_tensor_t(args, s); break;
    case MOE_PATH_STREAM: e = launch_ffn_stream(args, s); break;
    default: e = launch_ffn_simt(args, s); break;
  }
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: no kernel for this combination";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or launch failed";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: a device-side range check failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
  }
  return "unknown moe_status";
}

size_t moe_workspace_bytes(int T, int d, int F, int E, int k, moe_dtype dt) {
  if (!sizes_ok(T, d, F, E, k, dt)) return 0;
  return Layout(T, d, F, E, k, dt).end;
}

moe_status moe_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (workspace == nullptr || ws_bytes < kWsHeaderBytes || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, kWsHeaderBytes, (cudaStream_t)stream));
}

moe_status moe_get_device_status(void* workspace, int32_t* detail, void* stream) {
  if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t word[2] = {0, 0};
  if (cudaMemcpy(word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail != nullptr) *detail = word[1];
  return (moe_status)word[0];
}

moe_status moe_router_topk(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                           moe_dtype dt, int32_t* topk_idx, float* topk_gate, void* stream) {
  return moe_router_topk_ex(x, w_r, b_r, T, d, E, k, dt, 0, topk_idx, topk_gate, stream);
}

moe_status moe_router_topk_stats(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                                 moe_dtype dt, int flags, int32_t* topk_idx, float* topk_gate, float* stats,
                                 void* workspace, size_t ws_bytes, void* stream) {
  if (!sizes_ok(T, d, 8, E, k, dt) || (flags & ~MOE_GATES_RENORMALISE) != 0) return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || stats == nullptr) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < Layout(T, d, 8, E, k, dt).stats_end) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (x == nullptr || w_r == nullptr || topk_idx == nullptr || topk_gate == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
  // header words: [0] status, [1] detail, [3] the statistics ticket
  const RouterStats st{at<float>(workspace, Layout(T, d, 8, E, k, dt).stats_part), stats, at<int>(workspace, 0) + 3};
  bind_primary_context();
  return cuda_status(launch_router_topk(x, w_r, b_r, T, d, E, k, dt, flags, st, topk_idx, topk_gate,
                                        at<int>(workspace, 0), wait_timeout_ns(), (cudaStream_t)stream));
}

moe_status moe_router_topk_ex(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                              moe_dtype dt, int flags, int32_t* topk_idx, float* topk_gate, void* stream) {
  if (!sizes_ok(T, d, 8, E, k, dt) || (flags & ~MOE_GATES_RENORMALISE) != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (x == nullptr || w_r == nullptr || topk_idx == nullptr || topk_gate == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
  bind_primary_context();
  return cuda_status(launch_router_topk(x, w_r, b_r, T, d, E, k, dt, flags, RouterStats{nullptr, nullptr, nullptr},
                                        topk_idx, topk_gate, nullptr, wait_timeout_ns(), (cudaStream_t)stream));
}

moe_status moe_dispatch(const void* x, const int32_t* topk_idx, const float* topk_gate, int T, int d, int E,
                        int k, moe_dtype dt, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                        int32_t* row_of, float* row_gate, void* x_perm, void* workspace, size_t ws_bytes,
                        void* stream) {
  return moe_dispatch_ex(x, topk_idx, topk_gate, T, d, E, k, dt, 0, counts, offsets, perm_token, row_of, row_gate,
                         x_perm, workspace, ws_bytes, stream);
}

int moe_capacity(int T, int k, int E, double cf) {
  if (T < 0 || k < 1 || E < 1 || !(cf > 0.0)) return -1;
  const double c = std::ceil((double)T * k / E * cf);
  return c > 2147483647.0 ? -1 : (int)c;
}

moe_status moe_dispatch_ex(const void* x, const int32_t* topk_idx, const float* topk_gate, int T, int d, int E,
                           int k, moe_dtype dt, int capacity, int32_t* counts, int32_t* offsets,
                           int32_t* perm_token, int32_t* row_of, float* row_gate, void* x_perm, void* workspace,
                           size_t ws_bytes, void* stream) {
  if (!sizes_ok(T, d, 8, E, k, dt) || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr || workspace == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_idx == nullptr || topk_gate == nullptr || perm_token == nullptr ||
                row_of == nullptr || row_gate == nullptr || x_perm == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L(T, d, 8, E, k, dt);
  if (ws_bytes < L.dispatch_end) return MOE_ERR_INVALID_ARG;
  // header words: [0] status, [1] detail, [2] the count kernel's ticket, [3] the router statistics ticket
  return cuda_status(launch_dispatch_fast(x, topk_idx, topk_gate, T, d, E, k, dt, capacity, counts, offsets,
                                          perm_token, row_of, row_gate, x_perm, at<int32_t>(workspace, L.blk_counts),
                                          at<int32_t>(workspace, L.blk_base), at<int>(workspace, L.header),
                                          at<int>(workspace, L.header) + 2, (cudaStream_t)stream));
}

moe_status moe_dispatch_reroute(const void* x, const int32_t* rank_idx, const float* rank_gate, int T, int d, int E,
                                int k, int R, moe_dtype dt, int capacity, int32_t* final_idx, float* final_gate,
                                int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* row_of,
                                float* row_gate, void* x_perm, void* workspace, size_t ws_bytes, void* stream) {
  if (!sizes_ok(T, d, 8, E, k, dt) || R < k || R > E || capacity < 1) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr || workspace == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || rank_idx == nullptr || rank_gate == nullptr || final_idx == nullptr ||
                final_gate == nullptr || perm_token == nullptr || row_of == nullptr || row_gate == nullptr ||
                x_perm == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L(T, d, 8, E, k, dt);
  if (ws_bytes < L.dispatch_end) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch_reroute(x, rank_idx, rank_gate, T, d, E, k, R, dt, capacity, final_idx,
                                             final_gate, counts, offsets, perm_token, row_of, row_gate, x_perm,
                                             at<int32_t>(workspace, L.blk_counts), at<int32_t>(workspace, L.blk_base),
                                             at<int>(workspace, L.header), at<int>(workspace, L.header) + 2,
                                             (cudaStream_t)stream));
}

// a_rows (nullable): row r of `a` is a[a_rows[r]] (the weight-streaming path only).
static moe_status expert_half(int stage, const void* a, const void* w, const int32_t* offsets,
                              const float* row_gate, int T, int d, int F, int E, int k, moe_dtype dt, moe_path path,
                              void* out, void* workspace, size_t ws_bytes, void* stream,
                              const int32_t* a_rows = nullptr) {
  if (!sizes_ok(T, d, F, E, k, dt) || !path_ok(path, dt)) return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < kWsHeaderBytes || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (a == nullptr || w == nullptr || offsets == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (stage == 2 && row_gate == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  FfnArgs args;
  args.a = a; args.w = w; args.offsets = offsets; args.row_gate = row_gate; args.out = out;
  args.rows = T * k; args.E = E; args.dt = dt; args.stage = stage;
  args.K = stage == 1 ? d : F;
  args.N = stage == 1 ? F : d;
  args.status = at<int>(workspace, 0);
  args.timeout_ns = wait_timeout_ns();
  args.a_rows = a_rows;
  args.max_rows_per_expert = T;
  return run_ffn_half(path, args, (cudaStream_t)stream);
}

moe_status moe_expert_up_ex(const void* x_perm, const void* w1, const int32_t* offsets, int T, int d, int F,
                            int E, int k, moe_dtype dt, moe_path path, void* h, void* workspace, size_t ws_bytes,
                            void* stream) {
  return expert_half(1, x_perm, w1, offsets, nullptr, T, d, F, E, k, dt, path, h, workspace, ws_bytes, stream);
}
moe_status moe_expert_up(const void* x_perm, const void* w1, const int32_t* offsets, int T, int d, int F, int E,
                         int k, moe_dtype dt, void* h, void* workspace, size_t ws_bytes, void* stream) {
  return moe_expert_up_ex(x_perm, w1, offsets, T, d, F, E, k, dt, MOE_PATH_AUTO, h, workspace, ws_bytes, stream);
}
moe_status moe_expert_down_ex(const void* h, const void* w2, const int32_t* offsets, const float* row_gate,
                              int T, int d, int F, int E, int k, moe_dtype dt, moe_path path, void* y_perm,
                              void* workspace, size_t ws_bytes, void* stream) {
  return expert_half(2, h, w2, offsets, row_gate, T, d, F, E, k, dt, path, y_perm, workspace, ws_bytes, stream);
}
moe_status moe_expert_down(const void* h, const void* w2, const int32_t* offsets, const float* row_gate, int T,
                           int d, int F, int E, int k, moe_dtype dt, void* y_perm, void* workspace,
                           size_t ws_bytes, void* stream) {
  return moe_expert_down_ex(h, w2, offsets, row_gate, T, d, F, E, k, dt, MOE_PATH_AUTO, y_perm, workspace,
                            ws_bytes, stream);
}

moe_status moe_grouped_ffn_ex(const void* x_perm, const void* w1, const void* w2, const int32_t* offsets,
                              const float* row_gate, int T, int d, int F, int E, int k, moe_dtype dt,
                              moe_path path, void* y_perm, void* workspace, size_t ws_bytes, void* stream) {
  if (!sizes_ok(T, d, F, E, k, dt) || !path_ok(path, dt)) return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L(T, d, F, E, k, dt);
  if (ws_bytes < L.grouped_end) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  void* h = at<void>(workspace, L.h);
  moe_status st = moe_expert_up_ex(x_perm, w1, offsets, T, d, F, E, k, dt, path, h, workspace, ws_bytes, stream);
  if (st != MOE_OK) return st;
  return moe_expert_down_ex(h, w2, offsets, row_gate, T, d, F, E, k, dt, path, y_perm, workspace, ws_bytes, stream);
}
moe_status moe_grouped_ffn(const void* x_perm, const void* w1, const void* w2, const int32_t* offsets,
                           const float* row_gate, int T, int d, int F, int E, int k, moe_dtype dt, void* y_perm,
                           void* workspace, size_t ws_bytes, void* stream) {
  return moe_grouped_ffn_ex(x_perm, w1, w2, offsets, row_gate, T, d, F, E, k, dt, MOE_PATH_AUTO, y_perm,
                            workspace, ws_bytes, stream);
}

// ------------------------------------------------------------------ block-quantised weights
namespace {
bool qsizes_ok(int K, int N, int E, int bits) {
  return (bits == 4 || bits == 8) && K >= 64 && N >= 64 && K % 64 == 0 && N % 64 == 0 && E >= 1 && E <= 1024;
}
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

moe_status expert_half_q(int stage, const void* a, const void* codes, const float* scale_min,
                         const int32_t* offsets, const float* row_gate, int T, int d, int F, int E, int k, int bits,
                         void* out, void* stream, const int32_t* a_rows = nullptr, int* status = nullptr) {
  if (!sizes_ok(T, d, F, E, k, MOE_DTYPE_BF16)) return MOE_ERR_INVALID_ARG;
  const int K = stage == 1 ? d : F, N = stage == 1 ? F : d;
  if (!qsizes_ok(K, N, E, bits)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (a == nullptr || codes == nullptr || scale_min == nullptr || offsets == nullptr || out == nullptr ||
      (stage == 2 && row_gate == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(codes) || !aligned8(scale_min) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  QFfnArgs p{a, codes, scale_min, offsets, row_gate, out, T * k, K, N, E, bits, stage, a_rows, T, status,
             wait_timeout_ns()};
  bind_primary_context();
  return cuda_status(launch_ffn_stream_q(p, (cudaStream_t)stream));
}
}  // namespace

int moe_ffn_path(int T, int k, int E, int N, moe_dtype dt) {
  if (T < 0 || k < 1 || E < 1 || N < 1 || (dt != MOE_DTYPE_F32 && dt != MOE_DTYPE_BF16)) return -1;
  return (int)resolve_path(MOE_PATH_AUTO, dt, T * k, E, N);
}

int moe_forward_launches(int T, int d, int F, int E, int k, moe_dtype dt, moe_path path, int router_stats) {
  if (!sizes_ok(T, d, F, E, k, dt) || !path_ok(path, dt)) return -1;
  if (T == 0) return 0;
  // the decisions of moe_forward_ex and route_and_dispatch
  const Layout L(T, d, F, E, k, dt);
  const bool small_ok = resolve_path(path, dt, T * k, E, F) == MOE_PATH_STREAM &&
                        resolve_path(path, dt, T * k, E, d) == MOE_PATH_STREAM;
  if (small_ok && !router_stats && route_small_ok(T, d, E, k, dt, L.end - L.y_perm)) return 4;
  const bool tc_router = dt == MOE_DTYPE_BF16 && E <= 256 && E % 8 == 0;
  return tc_router && k * 128 == kDispatchChunk ? 5 : 6;
}

size_t moe_qweight_bytes(int K, int N, int E, int bits) {
  if (!qsizes_ok(K, N, E, bits)) return 0;
  return (size_t)E * K * N * bits / 8;
}
size_t moe_qscale_bytes(int K, int N, int E) {
  if (!qsizes_ok(K, N, E, 4)) return 0;
  return (size_t)E * (K / 64) * (N / 64) * 2 * sizeof(float);
}
moe_status moe_quantize_weights(const void* w, int K, int N, int E, moe_dtype dt, int bits, void* codes,
                                float* scale_min, void* stream) {
  if (!qsizes_ok(K, N, E, bits) || (dt != MOE_DTYPE_BF16 && dt != MOE_DTYPE_F32)) return MOE_ERR_INVALID_ARG;
  if (w == nullptr || codes == nullptr || scale_min == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || !aligned8(scale_min)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize(w, K, N, E, dt, bits, codes, scale_min, (cudaStream_t)stream));
}
moe_status moe_expert_up_q(const void* x_perm, const void* w1_codes, const float* w1_scale_min,
                           const int32_t* offsets, int T, int d, int F, int E, int k, int bits, void* h,
                           void* stream) {
  return expert_half_q(1, x_perm, w1_codes, w1_scale_min, offsets, nullptr, T, d, F, E, k, bits, h, stream);
}
moe_status moe_expert_down_q(const void* h, const void* w2_codes, const float* w2_scale_min,
                             const int32_t* offsets, const float* row_gate, int T, int d, int F, int E, int k,
                             int bits, void* y_perm, void* stream) {
  return expert_half_q(2, h, w2_codes, w2_scale_min, offsets, row_gate, T, d, F, E, k, bits, y_perm, stream);
}

moe_status moe_combine(const void* y_perm, const int32_t* row_of, int T, int d, int k, moe_dtype dt, void* out,
                       void* stream) {
  if (!sizes_ok(T, d, 8, k, k, dt)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (y_perm == nullptr || row_of == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(y_perm, row_of, T, d, k, dt, out, (cudaStream_t)stream));
}

namespace {
// Router, then dispatch. With k = 2 a tensor-core router tile (128 tokens) holds exactly one dispatch
// chunk (256 assignments), so the router also writes each chunk's expert histogram and the dispatch
// needs no count kernel; otherwise (or when the CUDA-core router ran) the two-kernel dispatch.
// small_ok: the expert GEMMs will stream weights; then a batch of at most 8 tokens (no statistics)
// takes the one-launch router + dispatch, which writes no x_perm: *rows_via_perm tells the caller
// to read x through perm_token instead.
moe_status route_and_dispatch(const void* x, const void* w_r, const float* b_r, int T, int d, int E, int k,
                              moe_dtype dt, int flags, int capacity, RouterStats rs, int32_t* idx, float* gate,
                              int32_t* cnt, int32_t* offs, int32_t* perm, int32_t* rowof, float* rgate, void* xp,
                              const Layout& L, void* workspace, size_t ws_bytes, void* stream, bool small_ok,
                              bool* rows_via_perm) {
  *rows_via_perm = false;
  bind_primary_context();
  if (flags & MOE_CAPACITY_REROUTE) {
    // each token's R best experts, then the rerouting dispatch into the caller's idx / gate
    const int R = E < kMaxRank ? E : kMaxRank;
    int32_t* ri = at<int32_t>(workspace, L.rank_idx);
    float* rg = at<float>(workspace, L.rank_gate);
    moe_status st = cuda_status(launch_router_topk(x, w_r, b_r, T, d, E, R, dt, 0, RouterStats{nullptr, nullptr, nullptr},
                                                   ri, rg, at<int>(workspace, 0), wait_timeout_ns(),
                                                   (cudaStream_t)stream));
    if (st != MOE_OK) return st;
    return cuda_status(launch_dispatch_reroute(x, ri, rg, T, d, E, k, R, dt, capacity, idx, gate, cnt, offs, perm,
                                               rowof, rgate, xp, at<int32_t>(workspace, L.blk_counts),
                                               at<int32_t>(workspace, L.blk_base), at<int>(workspace, 0),
                                               at<int>(workspace, 0) + 2, (cudaStream_t)stream));
  }
  if (small_ok && rs.part == nullptr && route_small_ok(T, d, E, k, dt, L.end - L.y_perm)) {
    *rows_via_perm = true;
    return cuda_status(launch_route_small(x, w_r, b_r, T, d, E, k, (flags & MOE_GATES_RENORMALISE) != 0, capacity,
                                          at<float>(workspace, L.y_perm), at<int>(workspace, 0) + 2, idx, gate, cnt,
                                          offs, perm, rowof, rgate, (cudaStream_t)stream));
  }
  rs.hist = k * 128 == kDispatchChunk ? at<int32_t>(workspace, L.blk_counts) : nullptr;
  bool wrote_hist = false;
  moe_status st = cuda_status(launch_router_topk(x, w_r, b_r, T, d, E, k, dt, flags, rs, idx, gate,
                                                 at<int>(workspace, 0), wait_timeout_ns(), (cudaStream_t)stream,
                                                 &wrote_hist));
  if (st != MOE_OK) return st;
  if (wrote_hist)
    return cuda_status(launch_dispatch_from_hist(x, idx, gate, T, d, E, k, dt, capacity,
                                                 at<int32_t>(workspace, L.blk_counts), cnt, offs, perm, rowof,
                                                 rgate, xp, (cudaStream_t)stream));
  return moe_dispatch_ex(x, idx, gate, T, d, E, k, dt, capacity, cnt, offs, perm, rowof, rgate, xp, workspace,
                         ws_bytes, stream);
}
}  // namespace

moe_status moe_forward_ex(const void* x, const void* w_r, const float* b_r, const void* w1, const void* w2,
                          int T, int d, int F, int E, int k, moe_dtype dt, moe_dtype out_dt, moe_path path,
                          int flags, int capacity, void* out, int32_t* topk_idx, float* topk_gate,
                          int32_t* counts, float* router_stats, void* workspace, size_t ws_bytes, void* stream) {
  if (!sizes_ok(T, d, F, E, k, dt) || !path_ok(path, dt) || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (!forward_flags_ok(flags, capacity, router_stats)) return MOE_ERR_INVALID_ARG;
  if (out_dt != MOE_DTYPE_F32 && out_dt != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L(T, d, F, E, k, dt);
  if (ws_bytes < L.end) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (x == nullptr || w_r == nullptr || w1 == nullptr || w2 == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r) || !aligned16(w1) || !aligned16(w2) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  int32_t* idx = topk_idx != nullptr ? topk_idx : at<int32_t>(workspace, L.topk_idx);
  float* gate = topk_gate != nullptr ? topk_gate : at<float>(workspace, L.topk_gate);
  int32_t* cnt = counts != nullptr ? counts : at<int32_t>(workspace, L.counts);
  int32_t* offs = at<int32_t>(workspace, L.offsets);
  int32_t* perm = at<int32_t>(workspace, L.perm_token);
  int32_t* rowof = at<int32_t>(workspace, L.row_of);
  float* rgate = at<float>(workspace, L.row_gate);
  void* xp = at<void>(workspace, L.x_perm);
  void* h = at<void>(workspace, L.h);
  void* yp = at<void>(workspace, L.y_perm);
  const RouterStats rs{router_stats != nullptr ? at<float>(workspace, L.stats_part) : nullptr, router_stats,
                       at<int>(workspace, 0) + 3};
  const bool small_ok = resolve_path(path, dt, T * k, E, F) == MOE_PATH_STREAM &&
                        resolve_path(path, dt, T * k, E, d) == MOE_PATH_STREAM;
  bool via_perm = false;
  moe_status st = route_and_dispatch(x, w_r, b_r, T, d, E, k, dt, flags, capacity, rs, idx, gate, cnt, offs, perm,
                                     rowof, rgate, xp, L, workspace, ws_bytes, stream, small_ok, &via_perm);
  if (st != MOE_OK) return st;
  st = via_perm ? expert_half(1, x, w1, offs, nullptr, T, d, F, E, k, dt, path, h, workspace, ws_bytes, stream, perm)
                : moe_expert_up_ex(xp, w1, offs, T, d, F, E, k, dt, path, h, workspace, ws_bytes, stream);
  if (st != MOE_OK) return st;
  st = moe_expert_down_ex(h, w2, offs, rgate, T, d, F, E, k, dt, path, yp, workspace, ws_bytes, stream);
  if (st != MOE_OK) return st;
  return moe_combine(yp, rowof, T, d, k, out_dt, out, stream);
}
moe_status moe_forward_q(const void* x, const void* w_r, const float* b_r, const void* w1_codes,
                         const float* w1_scale_min, const void* w2_codes, const float* w2_scale_min, int T, int d,
                         int F, int E, int k, int bits, moe_dtype out_dt, int flags, int capacity, void* out,
                         int32_t* topk_idx, float* topk_gate, int32_t* counts, float* router_stats, void* workspace,
                         size_t ws_bytes, void* stream) {
  const moe_dtype dt = MOE_DTYPE_BF16;
  if (!sizes_ok(T, d, F, E, k, dt) || !qsizes_ok(d, F, E, bits) || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (!forward_flags_ok(flags, capacity, router_stats)) return MOE_ERR_INVALID_ARG;
  if (out_dt != MOE_DTYPE_F32 && out_dt != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L(T, d, F, E, k, dt);
  if (ws_bytes < L.end) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (x == nullptr || w_r == nullptr || out == nullptr || !aligned16(x) || !aligned16(w_r) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  int32_t* idx = topk_idx != nullptr ? topk_idx : at<int32_t>(workspace, L.topk_idx);
  float* gate = topk_gate != nullptr ? topk_gate : at<float>(workspace, L.topk_gate);
  int32_t* cnt = counts != nullptr ? counts : at<int32_t>(workspace, L.counts);
  int32_t* offs = at<int32_t>(workspace, L.offsets);
  int32_t* rowof = at<int32_t>(workspace, L.row_of);
  float* rgate = at<float>(workspace, L.row_gate);
  void* xp = at<void>(workspace, L.x_perm);
  void* h = at<void>(workspace, L.h);
  void* yp = at<void>(workspace, L.y_perm);
  const RouterStats rs{router_stats != nullptr ? at<float>(workspace, L.stats_part) : nullptr, router_stats,
                       at<int>(workspace, 0) + 3};
  int32_t* perm = at<int32_t>(workspace, L.perm_token);
  bool via_perm = false;
  moe_status st = route_and_dispatch(x, w_r, b_r, T, d, E, k, dt, flags, capacity, rs, idx, gate, cnt, offs, perm,
                                     rowof, rgate, xp, L, workspace, ws_bytes, stream, true, &via_perm);
  if (st != MOE_OK) return st;
  int* status = at<int>(workspace, 0);
  st = expert_half_q(1, via_perm ? x : xp, w1_codes, w1_scale_min, offs, nullptr, T, d, F, E, k, bits, h, stream,
                     via_perm ? perm : nullptr, status);
  if (st != MOE_OK) return st;
  st = expert_half_q(2, h, w2_codes, w2_scale_min, offs, rgate, T, d, F, E, k, bits, yp, stream, nullptr, status);
  if (st != MOE_OK) return st;
  return moe_combine(yp, rowof, T, d, k, out_dt, out, stream);
}

moe_status moe_forward(const void* x, const void* w_r, const float* b_r, const void* w1, const void* w2, int T,
                       int d, int F, int E, int k, moe_dtype dt, void* out, int32_t* topk_idx, float* topk_gate,
                       int32_t* counts, void* workspace, size_t ws_bytes, void* stream) {
  return moe_forward_ex(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, dt, MOE_PATH_AUTO, 0, 0, out, topk_idx, topk_gate,
                        counts, nullptr, workspace, ws_bytes, stream);
}

moe_status moe_selftest_wait_timeout(void* workspace, size_t ws_bytes, int timeout_us, void* stream) {
  if (workspace == nullptr || ws_bytes < kWsHeaderBytes || !aligned16(workspace) || timeout_us <= 0 ||
      timeout_us > 10000000)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait(at<int>(workspace, 0), (uint64_t)timeout_us * 1000ull, (cudaStream_t)stream));
}

}  // extern "C"
