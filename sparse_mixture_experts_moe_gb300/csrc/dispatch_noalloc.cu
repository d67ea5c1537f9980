// moe_dispatch_noalloc: the dispatch step for callers that cannot hand the library any
// device scratch memory.
//
// moe_dispatch needs two small per-chunk count tables besides its inputs and outputs,
// and normally takes them from a caller-allocated workspace. Some callers cannot
// provide one: a plugin that a host framework hands only its input and output buffers
// (the framework owns all device memory through its own pool), or a latency-critical
// loop that must never call cudaMalloc, which can block and synchronise the device.
// This variant keeps the count tables in a fixed-size array that lives in the
// library's own device memory (one copy per GPU, held until the process exits).
//
// The array is shared by every call on a device and keeps what the last call left in
// it. Every call clears the one word that must start at zero (the count kernel's ticket)
// and rewrites the tables it reads, but two calls whose kernels overlap on the GPU (for
// example on two streams) race on it: issue them in order on one stream.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// 1 MiB of count tables, [ceil(T*k / 256) x E] int32 each, after a 256-byte slot whose first word
// is the count kernel's ticket (the CTA that finishes last scans and sets it back to zero).
constexpr size_t kNoAllocTicketBytes = 256;
constexpr size_t kNoAllocTableBytes = 1u << 20;
constexpr size_t kNoAllocMaxTableInts = kNoAllocTableBytes / (2 * sizeof(int32_t));

static __device__ __align__(256) int32_t g_dispatch_scratch[(kNoAllocTicketBytes + kNoAllocTableBytes) / sizeof(int32_t)];

}  // namespace
}  // namespace moe

extern "C" moe_status moe_dispatch_noalloc(const void* x, const int32_t* topk_idx, const float* topk_gate, int T,
                                           int d, int E, int k, moe_dtype dt, int32_t* counts, int32_t* offsets,
                                           int32_t* perm_token, int32_t* row_of, float* row_gate, void* x_perm,
                                           void* stream) {
  using namespace moe;
  if (dt != MOE_DTYPE_F32 && dt != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 8 || k > E || d < 8 || d % 8 != 0) return MOE_ERR_INVALID_ARG;
  if ((long long)T * k >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  const long long A = (long long)T * k;
  const long long nb = (A + kDispatchChunk - 1) / kDispatchChunk;
  if (nb * E > (long long)kNoAllocMaxTableInts) return MOE_ERR_INVALID_ARG;  // beyond the fixed scratch
  if (counts == nullptr || offsets == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_idx == nullptr || topk_gate == nullptr || perm_token == nullptr ||
                row_of == nullptr || row_gate == nullptr || x_perm == nullptr))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || (reinterpret_cast<uintptr_t>(x_perm) & 15u) != 0)
    return MOE_ERR_INVALID_ARG;
  // The array's device address on the current device, looked up on every call: host code cannot
  // use the array's name as a device pointer, and a cached address would go stale after a reset of
  // the device's context.
  void* base = nullptr;
  if (cudaGetSymbolAddress(&base, g_dispatch_scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* ticket = static_cast<int32_t*>(base);
  int32_t* blk_counts = ticket + kNoAllocTicketBytes / sizeof(int32_t);
  int32_t* blk_base = blk_counts + kNoAllocMaxTableInts;
  // The ticket must start at zero; the previous call's last CTA left it so, and it is cleared
  // again here so that no earlier call's state can matter.
  if (A > 0 && cudaMemsetAsync(ticket, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  // No status word: an index outside [0, E) is dropped (its row_of entry is -1, offsets[E] < T*k).
  const cudaError_t err = launch_dispatch_fast(x, topk_idx, topk_gate, T, d, E, k, dt, 0, counts, offsets,
                                               perm_token, row_of, row_gate, x_perm, blk_counts, blk_base, nullptr,
                                               ticket, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
