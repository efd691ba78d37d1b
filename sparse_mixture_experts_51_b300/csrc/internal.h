// Host-side launchers of the MoE layer kernels, and the workspace layout.
// Nothing here is part of the public C ABI (see include/moe_b300.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_b300.h"

namespace moe {

constexpr int kMaxExperts = 128;  // largest E the kernels support
constexpr int kMaxTopK = 16;      // largest k the kernels support

// Workspace carve-up shared by moe_forward / moe_dispatch / moe_expert_ffn.
// Every region starts on a 256-byte boundary.
struct WsLayout {
  size_t err;        // int32 error word (+ padding)
  size_t disp_ctrl;  // int32 ticket + int32 status[nblk]   (cleared per dispatch)
  size_t disp_agg;   // int32 [nblk][E] per-block expert histograms
  size_t disp_incl;  // int32 [nblk][E] inclusive prefixes
  size_t idx, w, pos;        // [T,k] int32 / fp32 / int32
  size_t counts, offsets;    // [E], [E+1] int32
  size_t dropped;            // int64
  size_t x_perm;             // [R,d] dtype
  size_t h;                  // [R,F] dtype
  size_t y_perm;             // [R,d] fp32
  size_t total;
  int nblk_dispatch;
  int64_t rows;              // R = min(T*k, E*C)
};

// Dispatch tiles: 256 threads x `items` consecutive priority positions each.
// Short batches use 1024-assignment tiles (more CTAs, shorter per-tile
// work); batches above 262144 assignments use 4096-assignment tiles.  Either
// way at most 256 tiles cover up to 2^20 assignments.
constexpr int kDispatchThreads = 256;
constexpr int kDispatchItemsSmall = 4;
constexpr int kDispatchItemsLarge = 16;
constexpr long long kDispatchSmallMax = 256LL * kDispatchItemsSmall * kDispatchThreads;
inline int dispatch_items(long long Tk) { return Tk <= kDispatchSmallMax ? kDispatchItemsSmall : kDispatchItemsLarge; }
inline int dispatch_nblk(long long Tk) {
  const long long tile = static_cast<long long>(dispatch_items(Tk)) * kDispatchThreads;
  return static_cast<int>(Tk == 0 ? 1 : (Tk + tile - 1) / tile);
}

WsLayout ws_layout(const moe_shape_t& s, int32_t C);

struct RouterParams {
  const void* x;
  const float* W_g;
  const float* b_g;
  const float* W_n;
  const float* eps;
  int T, d, E, k;
  int32_t* idx;
  float* w;
  float* logits;
  long long* stats;
  int* err;
};
cudaError_t launch_router(const RouterParams& p, int dtype, cudaStream_t st);
// the cluster-tiled router kernel (router_tiled.cu), for wide logit tables
cudaError_t launch_router_tiled(const RouterParams& p, int dtype, cudaStream_t st, int sms);

struct DispatchParams {
  const int32_t* idx;
  int T, k, E, C;
  int32_t* pos;
  int32_t* counts;
  int32_t* offsets;
  long long* dropped;
  int* ctrl;       // ticket + status[nblk]
  int* agg;        // [nblk][E]
  int* incl;       // [nblk][E]
  int nblk;
  int stall_block;  // testing hook: this tile never publishes its status (-1 = none)
  int* err;
};
cudaError_t launch_dispatch(const DispatchParams& p, cudaStream_t st);

struct GatherParams {
  const void* x;
  const int32_t* idx;
  const int32_t* pos;
  const int32_t* offsets;
  int T, k, d, E;
  void* x_perm;
  int32_t* row_token;
  int elem_bytes;
  long long rows_alloc;  // rows of x_perm
  int* err;
};
cudaError_t launch_gather(const GatherParams& p, cudaStream_t st);

struct FfnParams {
  const void* x_perm;
  const int32_t* offsets;
  const void* W1;
  const void* W3;
  const void* W2;
  const float* b1;
  const float* b2;
  void* h;
  float* y_perm;
  int E, d, F, act;
  long long rows;  // allocated rows of x_perm / h / y_perm
  int* err;
};
// between_gemms (optional) is recorded on `st` after the first GEMM is enqueued
cudaError_t launch_ffn_bf16(const FfnParams& p, cudaStream_t st, cudaEvent_t between_gemms = nullptr);
cudaError_t launch_ffn_f32(const FfnParams& p, cudaStream_t st);

struct CombineParams {
  const float* y_perm;
  const int32_t* idx;
  const float* w;
  const int32_t* pos;
  const int32_t* offsets;
  const void* residual;
  void* out;
  float* moe_out;
  int T, k, d, E;
  long long rows;
  int dtype;
  int* err;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t st);

}  // namespace moe
