// moe_dispatch_noalloc: capacity-limited dispatch + gather for callers that
// cannot allocate device memory.
//
// moe_dispatch keeps the state of its cross-block scan (tile ticket, per-tile
// status flags, per-tile expert histograms and prefixes) in a workspace the
// caller allocates.  Some callers cannot provide one: a plug-in whose host
// framework owns all device memory and hands it only the operation's inputs
// and outputs, or a latency-critical serving loop whose device memory plan is
// fixed up front and where a cudaMalloc (which may synchronise the device) is
// not allowed on the request path.  This entry point keeps that scan state in
// a fixed-size array in device global memory that belongs to the library
// itself, so it needs no allocation at all.
//
// The array (g_dispatch_scratch) is sized for at most kNoAllocMaxAssignments
// = 1,048,576 assignments (T*k), i.e. 256 dispatch tiles, and E <= 128:
// about 257 KiB, held by every GPU that loads the library until the process
// exits.  Every call shares it: the tile ticket and status flags are cleared
// at the start of each call (they must start at zero; the histogram and
// prefix slots are always written before they are read), and calls whose
// kernels overlap on the GPU (different streams without ordering, or
// several host threads) race on it and must be serialised by the caller.
//
// Host code cannot use the array's name as a device address, so the first
// call in each CUDA context (with that context current) looks the address up
// with cudaGetSymbolAddress and caches it under the context's process-unique
// id (cuCtxGetId); later calls in the same context reuse it.  A context that
// is torn down and recreated (cudaDeviceReset, a new primary or non-primary
// context) has a new id, so its first call looks the address up again.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "moe_b300.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxTiles = 256;
constexpr long long kNoAllocMaxAssignments = static_cast<long long>(kNoAllocMaxTiles) * kDispatchItemsLarge * kDispatchThreads;
// layout in ints: [0] ticket, [1, 1+kNoAllocMaxTiles) tile status, then a done counter,
// then per-tile expert histograms [tiles][E], then inclusive prefixes [tiles][E]
constexpr size_t kCtrlInts = 2 + kNoAllocMaxTiles;
constexpr size_t kAggOffset = (kCtrlInts + 63) / 64 * 64;
constexpr size_t kInclOffset = kAggOffset + static_cast<size_t>(kNoAllocMaxTiles) * kMaxExperts;
constexpr size_t kScratchInts = kInclOffset + static_cast<size_t>(kNoAllocMaxTiles) * kMaxExperts;

static __device__ __align__(256) int g_dispatch_scratch[kScratchInts];

constexpr int kMaxCachedContexts = 64;
struct CachedAddress {
  unsigned long long ctx_id;
  int* ptr;
};
std::mutex g_scratch_mu;
CachedAddress g_scratch_cache[kMaxCachedContexts] = {};
int g_scratch_used = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

cudaError_t load_context_calls() {
  if (g_ctx_get_current != nullptr && g_ctx_get_id != nullptr) return cudaSuccess;
  void* f1 = nullptr;
  void* f2 = nullptr;
  cudaDriverEntryPointQueryResult q1, q2;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
  if (e != cudaSuccess || q1 != cudaDriverEntryPointSuccess || f1 == nullptr) return cudaErrorSymbolNotFound;
  e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
  if (e != cudaSuccess || q2 != cudaDriverEntryPointSuccess || f2 == nullptr) return cudaErrorSymbolNotFound;
  g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
  g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  return cudaSuccess;
}

// Device address of g_dispatch_scratch in the current context (looked up
// once per context, keyed by the context's process-unique id).
cudaError_t scratch_in_current_context(int** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  cudaError_t e = load_context_calls();
  if (e != cudaSuccess) return e;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  void* p = nullptr;
  if (ctx == nullptr) {
    // no context is current yet: the runtime creates the device's primary
    // context for this lookup and makes it current
    if ((e = cudaGetSymbolAddress(&p, g_dispatch_scratch)) != cudaSuccess) return e;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  for (int i = 0; i < g_scratch_used; ++i) {
    if (g_scratch_cache[i].ctx_id == id) {
      *out = g_scratch_cache[i].ptr;
      return cudaSuccess;
    }
  }
  if (p == nullptr && (e = cudaGetSymbolAddress(&p, g_dispatch_scratch)) != cudaSuccess) return e;
  // a full table overwrites an entry (that context, if used again, is looked up again)
  const int slot = g_scratch_used < kMaxCachedContexts ? g_scratch_used++ : static_cast<int>(id % kMaxCachedContexts);
  g_scratch_cache[slot] = CachedAddress{id, static_cast<int*>(p)};
  *out = static_cast<int*>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_noalloc(const moe_shape_t* shape, int32_t C, const int32_t* idx,
                                             const void* x, int32_t* pos, int32_t* counts, int32_t* offsets,
                                             int64_t* dropped, void* x_perm, int32_t* row_token,
                                             int32_t* error_out, void* stream) {
  // the same shapes as moe_dispatch (an invalid or unsupported one returns before anything is enqueued)
  const moe_status_t sst = check_shape(shape);
  if (sst != MOE_OK) return sst;
  if (C < 0) return MOE_ERR_INVALID_ARG;
  // the plain token-choice dispatch only: no expert choice, no re-routing pass
  if (shape->routing != MOE_ROUTE_TOKEN_CHOICE || shape->overflow != MOE_OVERFLOW_DROP) return MOE_ERR_INVALID_ARG;
  const long long Tk = shape->T * static_cast<long long>(shape->k);
  if (Tk > kNoAllocMaxAssignments) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  if (counts == nullptr || offsets == nullptr || dropped == nullptr) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (idx == nullptr || x == nullptr || pos == nullptr)) return MOE_ERR_INVALID_ARG;
  const long long EC = static_cast<long long>(shape->E) * C;
  const long long rows = Tk < EC ? Tk : EC;
  if (rows > 0 && x_perm == nullptr) return MOE_ERR_INVALID_ARG;
  // the gather moves rows in 16-byte units
  const auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if ((shape->T > 0 && misaligned(x)) || (rows > 0 && misaligned(x_perm))) return MOE_ERR_UNSUPPORTED;

  int* scratch = nullptr;
  if (scratch_in_current_context(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (error_out != nullptr && cudaMemsetAsync(error_out, 0, sizeof(int32_t), st) != cudaSuccess)
    return MOE_ERR_CUDA;

  DispatchParams dp{};
  dp.idx = idx;
  dp.T = static_cast<int>(shape->T);
  dp.k = shape->k;
  dp.E = shape->E;
  dp.C = C;
  dp.pos = pos;
  dp.counts = counts;
  dp.offsets = offsets;
  dp.dropped = reinterpret_cast<long long*>(dropped);
  dp.ctrl = scratch;
  dp.clear_ctrl = 1;  // launch_dispatch clears the ticket, the status flags and the done counter
  dp.agg = scratch + kAggOffset;
  dp.incl = scratch + kInclOffset;
  dp.nblk = dispatch_nblk(Tk);  // <= kNoAllocMaxTiles for Tk <= kNoAllocMaxAssignments
  dp.stall_block = -1;
  dp.err = error_out;
  if (launch_dispatch(dp, st) != cudaSuccess) return MOE_ERR_CUDA;

  GatherParams gp{};
  gp.x = x;
  gp.idx = idx;
  gp.pos = pos;
  gp.offsets = offsets;
  gp.T = static_cast<int>(shape->T);
  gp.k = shape->k;
  gp.d = shape->d;
  gp.E = shape->E;
  gp.x_perm = x_perm;
  gp.row_token = row_token;
  gp.elem_bytes = shape->dtype == MOE_BF16 ? 2 : 4;
  gp.rows_alloc = rows;
  gp.err = error_out;
  return launch_gather(gp, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
