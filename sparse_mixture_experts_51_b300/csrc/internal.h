// Host-side launchers of the MoE layer kernels, and the workspace layout.
// Nothing here is part of the public C ABI (see include/moe_b300.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "moe_b300.h"

namespace moe {

// A named NVTX range around the host code that enqueues one stage of the
// layer (profilers attribute the stage's kernels to it; without a profiler
// attached the push and pop do nothing).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Kernels this library has enqueued (moe_kernel_launches).
inline std::atomic<unsigned long long>& launch_count() {
  static std::atomic<unsigned long long> n{0};
  return n;
}
inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) launch_count().fetch_add(1, std::memory_order_relaxed);
  return e;
}

// Launch `kern` on `st` with programmatic stream serialisation (it may start
// while the previous kernel on the stream finishes; the kernel calls
// pdl_wait() before reading that kernel's outputs).  cluster_y > 1 adds a
// (1, cluster_y, 1) thread-block cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_y, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned n = 1;
  if (cluster_y > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = cluster_y;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return counted(cudaLaunchKernelEx(&cfg, kern, args...));
}

constexpr int kMaxExperts = 128;  // largest E the kernels support
constexpr int kMaxTopK = 16;      // largest k the kernels support
constexpr int kStatsMaxBlocks = 148;  // blocks of the routing-stats kernel (one wave)

// Workspace carve-up shared by moe_forward / moe_dispatch / moe_expert_ffn.
// Every region starts on a 256-byte boundary.
struct WsLayout {
  size_t err;        // int32 error word (+ padding)
  size_t disp_ctrl;  // int32 ticket, status[nblk], done (self-resetting; zero at first use)
  size_t disp_agg;   // int32 [nblk][E] per-block expert histograms
  size_t disp_incl;  // int32 [nblk][E] inclusive prefixes
  size_t stats_ticket;  // int32 last-block ticket of moe_routing_stats (self-resetting)
  size_t stats_acc;     // uint64 [2E+1] fixed-point totals of p, entropy and routed loads
  size_t h_shared;      // [T,d_ff_shared] dtype: hidden activation of the shared experts
  size_t y_shared;      // [T,d] fp32: shared experts' output
  // expert-choice routing only (zero size otherwise)
  size_t ec_logits, ec_radius, ec_gate;  // [T,E] fp32
  size_t ec_lse;                         // [T] fp32
  size_t ec_row_of;                      // [T,E] int32
  size_t ec_flag;                        // [E,T] uint8
  size_t ec_band;                        // [E,T] int32
  size_t ec_h64;                         // [E,T] fp64
  size_t ec_sel;                         // [E*Cp] int32
  size_t rt_scratch;                     // tensor-core router filter (bf16 token choice)
  size_t rt_scratch_bytes;
  int32_t ec_cp;                         // min(C, T)
  size_t idx, w, pos;        // [T,k] int32 / fp32 / int32
  size_t row_of;             // [T,k] int32: expert-grouped row of each assignment, -1 if dropped
  size_t counts, offsets;    // [E], [E+1] int32
  size_t dropped;            // int64
  size_t rr_backup;          // [T] int32 (overflow re-routing only, else empty)
  size_t rr_req, rr_pos2;    // [T,k] int32
  size_t rr_counts1;         // [E] int32: counts after the first pass
  size_t rr_dropped2;        // int64
  size_t x_perm;             // [R,d] dtype
  size_t h;                  // [R,F] dtype
  size_t y_perm;             // [R,d] fp32
  size_t dec_h;              // decode-sized batches: [E*128, d_ff] bf16 hidden rows of every (expert, token)
  size_t dec_ctrl;           // and the fused FFN's tile ticket and per-expert counts
  bool dec;                  // the fused decode FFN applies (ffn_decode_applies)
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
// MOE_OK, or the status every entry point returns for an invalid or unsupported shape
moe_status_t check_shape(const moe_shape_t* s);

struct RouterParams {
  const void* x;
  const float* W_g;
  const float* b_g;
  const float* W_n;
  const float* eps;
  int T, d, E, k;
  int32_t* idx;     // [T,k] out; null: no top-k (expert-choice routing: logits, radius and lse only)
  float* w;
  float* logits;
  float* radius;    // [T,E] out or null: a rigorous bound on |logit - exact logit|
  float* lse;       // [T] out or null: log-sum-exp of the token's fp32 logits
  int32_t* backup;  // [T] out or null: the (k+1)-th ranked expert, exact like the top-k (-1 if k = E)
  int gate_raw;     // 1: gates are the full-softmax probabilities of the selected experts
  long long* stats;
  int* err;
  void* scratch;    // workspace room for the tensor-core filter path (null: CUDA cores only)
  size_t scratch_bytes;
  int early_trigger;  // 1: let the next kernel launch right after this one's own wait on its predecessor
};
cudaError_t launch_router(const RouterParams& p, int dtype, cudaStream_t st);
// the tensor-core filter router (router_tc.cu) for wide logit tables of bf16 layers
bool router_tc_applies(const RouterParams& p, int dtype);
size_t router_tc_scratch_bytes(long long T, int d, int E);
// its carve-up of that scratch: approximate logits [T][nc], the bf16 hi|lo
// split of the router-weight columns [nc][2d], the fp32 columns [nc][d] and
// their norms [nc] (nc = E, or 2E with the noise columns)
struct RouterTcScratch {
  float* approx;
  void* wsplit;
  float* wt;
  float* cn;
};
RouterTcScratch router_tc_scratch(void* scratch, long long T, int d, int E);
cudaError_t launch_router_tc(const RouterParams& p, void* scratch, cudaStream_t st);
// its weight split and filter GEMM alone: the approximate logits [T, nc] (a test hook)
cudaError_t launch_router_tc_filter(const RouterParams& p, void* scratch, float* approx, cudaStream_t st);
// the cluster-tiled router kernel (router_tiled.cu), for wide logit tables
cudaError_t launch_router_tiled(const RouterParams& p, int dtype, cudaStream_t st, int sms);

struct DispatchParams {
  const int32_t* idx;
  int T, k, E, C;
  int32_t* pos;
  int32_t* counts;
  int32_t* offsets;
  long long* dropped;
  int* ctrl;       // ticket, status[nblk], done counter
  int clear_ctrl;  // 1: zero ctrl before the kernel; 0: it is zero already (the last block resets it)
  int early_trigger;  // 1: let the next kernel launch at once (it waits for this one before reading its outputs)
  int* agg;        // [nblk][E]
  int* incl;       // [nblk][E]
  int nblk;
  int stall_block;  // testing hook: this tile never publishes its status (-1 = none)
  const int32_t* base;  // [E] or null: slots already taken in each expert (a second, re-routing pass)
  int allow_skip;       // 1: an expert id of -1 is no assignment (not an error)
  int* err;
};
cudaError_t launch_dispatch(const DispatchParams& p, cudaStream_t st);

// Overflow re-routing around a second dispatch pass: requests (the first
// dropped assignment of each token asks for its backup expert), then the
// merge of the second pass into the tables of the first.
struct RerouteParams {
  const int32_t* backup;  // [T]
  int32_t* idx;           // [T,k] in/out: expert of each assignment (rerouted ones replaced)
  int32_t* pos;           // [T,k] in/out: slot (rerouted ones filled in)
  int32_t* req;           // [T,k] out (requests pass) / in (merge pass): backup asked for, or -1
  const int32_t* pos2;    // [T,k] second-pass slots
  long long* dropped;     // out (merge): assignments left without an expert
  int T, k;
};
cudaError_t launch_reroute_requests(const RerouteParams& p, cudaStream_t st);
cudaError_t launch_reroute_merge(const RerouteParams& p, cudaStream_t st);

struct GatherParams {
  const void* x;
  const int32_t* idx;
  const int32_t* pos;
  const int32_t* offsets;
  int T, k, d, E;
  void* x_perm;
  int32_t* row_token;
  int32_t* row_of;  // [T,k] out (optional): grouped row of each assignment, -1 if dropped
  int elem_bytes;
  long long rows_alloc;  // rows of x_perm
  int* err;
};
cudaError_t launch_gather(const GatherParams& p, cudaStream_t st);

struct FfnParams {
  const void* x_perm;
  const int32_t* offsets;  // [E+1]; null: a dense FFN (E = 1) over all `rows` rows
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
// The expert FFN and combine of a decode-sized batch (ffn_decode.cu): one
// persistent kernel, phase 1 dense over all T <= 128 tokens (no routing
// needed), phase 2 scattered to the kept assignments' grouped rows of
// y_perm, then the weighted combine into the residual, block by block.
struct DecodeFfnParams {
  const void* x;  // [T, d] bf16 tokens
  int T, d, F, E, k, act;
  const void* W1;
  const void* W3;
  const void* W2;
  const float* b1;
  const float* b2;
  void* h;                 // [E*128, F] bf16 workspace
  // [T,k] routing tables: read after the routing kernels complete, or (self_route)
  // written by the kernel's own routing tiles before any tile reads them
  int32_t* idx;
  int32_t* pos;
  int32_t* offsets;
  float* y_perm;           // [rows, d]
  long long rows;
  int* ctrl;               // ffn_decode_ctrl_bytes, zero at first use (self-resetting)
  int* err;
  // the combine, done by the same kernel: out = x + sum over kept ranks of w * y (+ y_shared)
  float* w;                // [T,k] gates (written by the routing tiles when self_route)
  const float* y_shared;   // [T,d] fp32 or null
  void* out;               // [T,d] bf16
  float* moe_out;          // [T,d] fp32 or null
  // self_route = 1: the kernel also routes (exact top-k as in router.cu) and
  // dispatches (slots in priority order, capacity C, as in dispatch.cu)
  int self_route;
  const float* W_g;
  const float* b_g;
  const float* W_n;
  const float* eps;
  int gate_raw;
  int C;
  float* logits;           // [T,E] or null
  long long* stats;        // router counters or null
  int32_t* counts;         // [E]
  long long* dropped;      // [1]
  int32_t* row_of;         // [T,k] workspace: grouped row of each assignment, -1 if dropped
};
bool ffn_decode_applies(const moe_shape_t& s);
// the fused kernel can also route the batch: overflow drop, nc = E (2E with the
// noise projection) a power of two in [4, 256], router weights 16-byte aligned
bool ffn_decode_routes(const moe_shape_t& s, const float* W_g, const float* W_n);
size_t ffn_decode_h_bytes(const moe_shape_t& s);
size_t ffn_decode_ctrl_bytes(const moe_shape_t& s);
cudaError_t launch_ffn_decode(const DecodeFfnParams& p, cudaStream_t st);

// between_gemms (optional) is recorded on `st` after the first GEMM is enqueued
cudaError_t launch_ffn_bf16(const FfnParams& p, cudaStream_t st, cudaEvent_t between_gemms = nullptr);
cudaError_t launch_ffn_f32(const FfnParams& p, cudaStream_t st);
// out[r, n] = sum_k A[r, k mod Ka] * B[n, k] on the tensor cores (bf16 in, fp32 out)
cudaError_t launch_dense_wrapped_gemm(const void* A, long long rows, int Ka, const void* B, int N, int K, float* out,
                                      int* err, cudaStream_t st);

struct CombineParams {
  const float* y_perm;
  const float* y_shared;  // [T,d] fp32 or null: shared experts' output, added after the ranks
  const int32_t* row_of;  // [T,k] grouped rows (-1 dropped); when set, idx/pos/offsets are not read
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

// Expert-choice routing (expert_choice.cu): each expert takes its Cp = min(C, T)
// highest-scoring tokens; rows e*Cp .. e*Cp+Cp-1 of the grouped buffers are
// expert e's tokens in token order.
struct EcParams {
  const float* logits;  // [T,E] fp32 router logits
  const float* radius;  // [T,E] their error radii
  const float* lse;     // [T]
  const void* x;        // [T,d] tokens (fp64 re-evaluation of the band)
  const float* W_g;
  const float* b_g;
  const float* W_n;
  const float* eps;
  int T, d, E, Cp;
  int32_t* sel;      // [E*Cp] out: token of each grouped row
  int32_t* row_of;   // [T,E] out: grouped row of (t, e), -1 if e did not choose t
  float* gate_te;    // [T,E] out: p[t,e] where chosen
  uint8_t* flag;     // [E][T] scratch
  int32_t* band;     // [E][T] scratch
  double* h64;       // [E][T] scratch
  int* err;
};
cudaError_t launch_ec_select(const EcParams& p, int dtype, cudaStream_t st);
cudaError_t launch_ec_finalize(const EcParams& p, int32_t* counts, int32_t* offsets, long long* dropped,
                               cudaStream_t st);
cudaError_t launch_ec_gather(const EcParams& p, const void* x, void* x_perm, int elem_bytes, cudaStream_t st);

struct StatsParams {
  const float* logits;     // [T,E]
  const int32_t* idx;      // [T,k]
  const int32_t* counts;   // [E] kept per expert
  const long long* dropped;
  long long T;
  int E, k;
  double* f;        // [E] out
  double* P;        // [E] out
  double* summary;  // [6] out
  unsigned long long* acc;  // [2E+1] fixed-point totals (zero between calls)
  int* ticket;
  int* err;
};
int stats_blocks(long long T);
cudaError_t launch_routing_stats(const StatsParams& p, cudaStream_t st);

}  // namespace moe
