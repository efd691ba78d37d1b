// C ABI of the MoE layer library: argument checks, workspace carve-up and
// the launch sequence router -> dispatch -> gather -> expert GEMMs -> combine.
// Declarations and the full contract are in include/moe_b300.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "moe_b300.h"
#include "moe_b300_testing.h"

namespace moe {

namespace {
constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
size_t dtype_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

WsLayout ws_layout(const moe_shape_t& s, int32_t C) {
  WsLayout L{};
  const long long Tk = s.T * s.k;
  const long long EC = static_cast<long long>(s.E) * C;
  const bool ec = s.routing == MOE_ROUTE_EXPERT_CHOICE;
  L.ec_cp = static_cast<int32_t>(C < s.T ? C : s.T);
  L.rows = ec ? static_cast<long long>(s.E) * L.ec_cp : (Tk < EC ? Tk : EC);
  L.nblk_dispatch = dispatch_nblk(Tk);
  const size_t b = dtype_bytes(s.dtype);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.err = take(sizeof(int));
  L.disp_ctrl = take(sizeof(int) * (2 + L.nblk_dispatch));
  L.disp_agg = take(sizeof(int) * static_cast<size_t>(L.nblk_dispatch) * s.E);
  L.disp_incl = take(sizeof(int) * static_cast<size_t>(L.nblk_dispatch) * s.E);
  L.stats_ticket = take(sizeof(int));
  L.stats_acc = take(sizeof(unsigned long long) * (2 * static_cast<size_t>(s.E) + 1));
  // (the regions up to here do not depend on C: any C's workspace holds them)
  L.h_shared = take(b * static_cast<size_t>(s.T) * s.d_ff_shared);
  L.y_shared = take(s.d_ff_shared > 0 ? sizeof(float) * static_cast<size_t>(s.T) * s.d : 0);
  const size_t TE = ec ? static_cast<size_t>(s.T) * s.E : 0;
  L.ec_logits = take(sizeof(float) * TE);
  L.ec_radius = take(sizeof(float) * TE);
  L.ec_gate = take(sizeof(float) * TE);
  L.ec_lse = take(ec ? sizeof(float) * static_cast<size_t>(s.T) : 0);
  L.ec_row_of = take(sizeof(int32_t) * TE);
  L.ec_flag = take(TE);
  L.ec_band = take(sizeof(int32_t) * TE);
  L.ec_h64 = take(sizeof(double) * TE);
  L.ec_sel = take(ec ? sizeof(int32_t) * static_cast<size_t>(L.rows) : 0);
  L.rt_scratch_bytes = (s.dtype == MOE_BF16 && !ec) ? router_tc_scratch_bytes(s.T, s.d, s.E) : 0;
  L.rt_scratch = take(L.rt_scratch_bytes);
  L.idx = take(sizeof(int32_t) * Tk);
  L.w = take(sizeof(float) * Tk);
  L.pos = take(sizeof(int32_t) * Tk);
  L.row_of = take(sizeof(int32_t) * Tk);
  L.counts = take(sizeof(int32_t) * s.E);
  L.offsets = take(sizeof(int32_t) * (s.E + 1));
  L.dropped = take(sizeof(long long));
  const bool rr = s.overflow == MOE_OVERFLOW_REROUTE;
  L.rr_backup = take(rr ? sizeof(int32_t) * static_cast<size_t>(s.T) : 0);
  L.rr_req = take(rr ? sizeof(int32_t) * Tk : 0);
  L.rr_pos2 = take(rr ? sizeof(int32_t) * Tk : 0);
  L.rr_counts1 = take(rr ? sizeof(int32_t) * s.E : 0);
  L.rr_dropped2 = take(rr ? sizeof(long long) : 0);
  L.x_perm = take(b * static_cast<size_t>(L.rows) * s.d);
  L.h = take(b * static_cast<size_t>(L.rows) * s.d_ff);
  L.y_perm = take(sizeof(float) * static_cast<size_t>(L.rows) * s.d);
  L.dec = ffn_decode_applies(s);
  L.dec_h = take(L.dec ? ffn_decode_h_bytes(s) : 0);
  L.dec_ctrl = take(L.dec ? ffn_decode_ctrl_bytes(s) : 0);
  L.total = o;
  return L;
}

// Argument check shared by every entry point that takes a layer shape.
moe_status_t check_shape(const moe_shape_t* s) {
  if (s == nullptr) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->d < 1 || s->E < 1 || s->k < 1 || s->d_ff < 1) return MOE_ERR_INVALID_ARG;
  if (s->k > s->E) return MOE_ERR_INVALID_ARG;
  if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (s->act != MOE_ACT_GELU && s->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (s->T * static_cast<long long>(s->k) >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (s->E > kMaxExperts || s->k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (s->dtype == MOE_BF16 && (s->d % 64 != 0 || s->d_ff % 64 != 0)) return MOE_ERR_UNSUPPORTED;
  if (s->dtype == MOE_F32 && s->d % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (s->d_ff_shared < 0) return MOE_ERR_INVALID_ARG;
  if (s->dtype == MOE_BF16 && s->d_ff_shared % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (s->routing != MOE_ROUTE_TOKEN_CHOICE && s->routing != MOE_ROUTE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  if (s->routing == MOE_ROUTE_EXPERT_CHOICE && s->T * static_cast<long long>(s->E) >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED;
  if (s->gates != MOE_GATES_RENORM && s->gates != MOE_GATES_RAW) return MOE_ERR_INVALID_ARG;
  if (s->overflow != MOE_OVERFLOW_DROP && s->overflow != MOE_OVERFLOW_REROUTE) return MOE_ERR_INVALID_ARG;
  if (s->routing == MOE_ROUTE_EXPERT_CHOICE && (s->gates != MOE_GATES_RENORM || s->overflow != MOE_OVERFLOW_DROP))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

namespace {

moe_status_t check_ws(const moe_shape_t* s, int32_t C, const void* ws, size_t ws_bytes) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(*s, C).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_capacity(int64_t T, int32_t k, int32_t E, double capacity_factor) {
  if (T < 0 || k < 1 || E < 1 || !std::isfinite(capacity_factor) || capacity_factor <= 0.0) return -1;
  const double v = std::ceil(capacity_factor * static_cast<double>(T) * static_cast<double>(k) / static_cast<double>(E));
  if (!(v <= 2147483647.0)) return -1;
  return static_cast<int32_t>(v);
}

int64_t moe_max_rows(const moe_shape_t* shape, int32_t C) {
  if (check_shape(shape) == MOE_ERR_INVALID_ARG || C < 0) return -1;
  return ws_layout(*shape, C).rows;
}

moe_status_t moe_workspace_size(const moe_shape_t* shape, int32_t C, size_t* bytes) {
  if (bytes == nullptr || C < 0) return MOE_ERR_INVALID_ARG;
  const moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  *bytes = ws_layout(*shape, C).total;
  return MOE_OK;
}

moe_status_t moe_route(const moe_shape_t* shape, const void* x, const float* W_g, const float* b_g,
                       const float* W_noise, const float* eps, int32_t* idx, float* w, float* logits,
                       int64_t* stats, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0 && (x == nullptr || idx == nullptr || w == nullptr)) return MOE_ERR_INVALID_ARG;
  if (W_g == nullptr) return MOE_ERR_INVALID_ARG;
  if ((W_noise == nullptr) != (eps == nullptr)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && !aligned16(x)) return MOE_ERR_UNSUPPORTED;
  RouterParams p{};
  p.x = x;
  p.W_g = W_g;
  p.b_g = b_g;
  p.W_n = W_noise;
  p.eps = eps;
  p.T = static_cast<int>(shape->T);
  p.d = shape->d;
  p.E = shape->E;
  p.k = shape->k;
  p.idx = idx;
  p.w = w;
  p.logits = logits;
  p.gate_raw = shape->gates == MOE_GATES_RAW ? 1 : 0;
  p.stats = reinterpret_cast<long long*>(stats);
  p.err = nullptr;
  return cuda_status(launch_router(p, shape->dtype, static_cast<cudaStream_t>(stream)));
}

// The token-choice router of the whole layer: moe_route, plus the backup
// expert of each token when overflow re-routing is on.
static moe_status_t route_impl(const moe_shape_t* shape, const void* x, const float* W_g, const float* b_g,
                               const float* W_noise, const float* eps, int32_t* idx, float* w, float* logits,
                               int64_t* stats, int32_t* backup, int* err, cudaStream_t st, void* scratch = nullptr,
                               size_t scratch_bytes = 0, bool early_trigger = false) {
  if (shape->T == 0) return MOE_OK;
  RouterParams p{};
  p.x = x;
  p.W_g = W_g;
  p.b_g = b_g;
  p.W_n = W_noise;
  p.eps = eps;
  p.T = static_cast<int>(shape->T);
  p.d = shape->d;
  p.E = shape->E;
  p.k = shape->k;
  p.idx = idx;
  p.w = w;
  p.logits = logits;
  p.backup = backup;
  p.gate_raw = shape->gates == MOE_GATES_RAW ? 1 : 0;
  p.stats = reinterpret_cast<long long*>(stats);
  p.err = err;
  p.scratch = scratch;
  p.scratch_bytes = scratch_bytes;
  p.early_trigger = early_trigger ? 1 : 0;
  return cuda_status(launch_router(p, shape->dtype, st));
}

// Expert-choice routing: the router in its no-top-k mode (logits, radii,
// log-sum-exp), then every expert's exact top-C' selection.
static moe_status_t ec_route_impl(const moe_shape_t* shape, const void* x, const float* W_g, const float* b_g,
                                  const float* W_noise, const float* eps, float* logits, void* ws, const WsLayout& L,
                                  cudaStream_t st, EcParams& ep) {
  if (logits == nullptr) logits = at<float>(ws, L.ec_logits);
  RouterParams p{};
  p.x = x;
  p.W_g = W_g;
  p.b_g = b_g;
  p.W_n = W_noise;
  p.eps = eps;
  p.T = static_cast<int>(shape->T);
  p.d = shape->d;
  p.E = shape->E;
  p.k = shape->k;
  p.idx = nullptr;
  p.w = nullptr;
  p.logits = logits;
  p.radius = at<float>(ws, L.ec_radius);
  p.lse = at<float>(ws, L.ec_lse);
  p.stats = nullptr;
  p.err = at<int>(ws, L.err);
  if (shape->T > 0) {
    cudaError_t e = launch_router(p, shape->dtype, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  ep = EcParams{};
  ep.logits = logits;
  ep.radius = p.radius;
  ep.lse = p.lse;
  ep.x = x;
  ep.W_g = W_g;
  ep.b_g = b_g;
  ep.W_n = W_noise;
  ep.eps = eps;
  ep.T = static_cast<int>(shape->T);
  ep.d = shape->d;
  ep.E = shape->E;
  ep.Cp = L.ec_cp;
  ep.sel = at<int32_t>(ws, L.ec_sel);
  ep.row_of = at<int32_t>(ws, L.ec_row_of);
  ep.gate_te = at<float>(ws, L.ec_gate);
  ep.flag = at<uint8_t>(ws, L.ec_flag);
  ep.band = at<int32_t>(ws, L.ec_band);
  ep.h64 = at<double>(ws, L.ec_h64);
  ep.err = at<int>(ws, L.err);
  return cuda_status(launch_ec_select(ep, shape->dtype, st));
}

// gates of the chosen pairs in [E, C'] order: gates[row] = gate_te[sel[row], e]
__global__ void ec_gates_kernel(const int32_t* sel, const float* gate_te, int E, int Cp, float* gates) {
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= static_cast<long long>(E) * Cp) return;
  const int e = static_cast<int>(row / Cp);
  gates[row] = gate_te[static_cast<long long>(sel[row]) * E + e];
}

static moe_status_t dispatch_impl(const moe_shape_t* shape, int32_t C, int32_t* idx, const void* x,
                                  int32_t* pos, int32_t* counts, int32_t* offsets, int64_t* dropped,
                                  void* x_perm, int32_t* row_token, void* ws, const WsLayout& L,
                                  cudaStream_t st, int stall_block = -1, int32_t* row_of = nullptr,
                                  const int32_t* backup = nullptr, bool early_trigger = false,
                                  bool gather = true) {
  const bool rr = backup != nullptr;
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
  dp.ctrl = at<int>(ws, L.disp_ctrl);
  dp.clear_ctrl = 0;
  dp.agg = at<int>(ws, L.disp_agg);
  dp.incl = at<int>(ws, L.disp_incl);
  dp.nblk = L.nblk_dispatch;
  dp.stall_block = stall_block;
  dp.early_trigger = early_trigger ? 1 : 0;
  dp.err = at<int>(ws, L.err);
  if (rr) {
    // first pass into scratch counts / drop count; the second pass writes the real ones
    dp.counts = at<int32_t>(ws, L.rr_counts1);
    dp.dropped = at<long long>(ws, L.rr_dropped2);
  }
  cudaError_t e = launch_dispatch(dp, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (rr) {
    RerouteParams rp{};
    rp.backup = backup;
    rp.idx = idx;
    rp.pos = pos;
    rp.req = at<int32_t>(ws, L.rr_req);
    rp.pos2 = at<int32_t>(ws, L.rr_pos2);
    rp.dropped = reinterpret_cast<long long*>(dropped);
    rp.T = static_cast<int>(shape->T);
    rp.k = shape->k;
    if (launch_reroute_requests(rp, st) != cudaSuccess) return MOE_ERR_CUDA;
    DispatchParams d2 = dp;
    d2.idx = rp.req;
    d2.pos = at<int32_t>(ws, L.rr_pos2);
    d2.counts = counts;
    d2.dropped = at<long long>(ws, L.rr_dropped2);
    d2.base = at<int32_t>(ws, L.rr_counts1);
    d2.allow_skip = 1;
    if (launch_dispatch(d2, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_reroute_merge(rp, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!gather) return MOE_OK;
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
  gp.row_of = row_of;
  gp.elem_bytes = static_cast<int>(dtype_bytes(shape->dtype));
  gp.rows_alloc = L.rows;
  gp.err = at<int>(ws, L.err);
  return cuda_status(launch_gather(gp, st));
}

moe_status_t moe_route_expert_choice(const moe_shape_t* shape, int32_t C, const void* x, const float* W_g,
                                     const float* b_g, const float* W_noise, const float* eps, int32_t* sel,
                                     float* gates, float* logits, int64_t* dropped, void* ws, size_t ws_bytes,
                                     void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->routing != MOE_ROUTE_EXPERT_CHOICE || C < 0) return MOE_ERR_INVALID_ARG;
  if (W_g == nullptr) return MOE_ERR_INVALID_ARG;
  if ((W_noise == nullptr) != (eps == nullptr)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, C);
  if (shape->T > 0 && x == nullptr) return MOE_ERR_INVALID_ARG;
  if (L.rows > 0 && (sel == nullptr || gates == nullptr)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && !aligned16(x)) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, C, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EcParams ep{};
  if ((st = ec_route_impl(shape, x, W_g, b_g, W_noise, eps, logits, ws, L, s, ep)) != MOE_OK) return st;
  if (L.rows > 0) {
    if (cudaMemcpyAsync(sel, ep.sel, sizeof(int32_t) * static_cast<size_t>(L.rows), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    ec_gates_kernel<<<static_cast<unsigned>((L.rows + 255) / 256), 256, 0, s>>>(ep.sel, ep.gate_te, shape->E,
                                                                                 L.ec_cp, gates);
    if (counted(cudaGetLastError()) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (dropped != nullptr) {
    // counts / offsets are implied (C' each): the workspace copies take them
    if (shape->T == 0) return cuda_status(cudaMemsetAsync(dropped, 0, sizeof(int64_t), s));
    return cuda_status(launch_ec_finalize(ep, at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                                          reinterpret_cast<long long*>(dropped), s));
  }
  return MOE_OK;
}

moe_status_t moe_dispatch(const moe_shape_t* shape, int32_t C, const int32_t* idx, const void* x, int32_t* pos,
                          int32_t* counts, int32_t* offsets, int64_t* dropped, void* x_perm, int32_t* row_token,
                          void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;  // token-choice tables
  if (shape->overflow != MOE_OVERFLOW_DROP) return MOE_ERR_INVALID_ARG;     // re-routing: moe_forward only
  if (C < 0) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr || dropped == nullptr) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (idx == nullptr || x == nullptr || pos == nullptr)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, C);
  if (L.rows > 0 && x_perm == nullptr) return MOE_ERR_INVALID_ARG;
  // the gather moves rows in 16-byte units
  if ((shape->T > 0 && !aligned16(x)) || (L.rows > 0 && !aligned16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, C, ws, ws_bytes)) != MOE_OK) return st;
  return dispatch_impl(shape, C, const_cast<int32_t*>(idx), x, pos, counts, offsets, dropped, x_perm, row_token,
                       ws, L, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_testing_dispatch_stalled(const moe_shape_t* shape, int32_t C, const int32_t* idx,
                                          const void* x, int32_t* pos, int32_t* counts, int32_t* offsets,
                                          int64_t* dropped, void* x_perm, int32_t stalled_tile, void* ws,
                                          size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;  // token-choice tables
  if (shape->overflow != MOE_OVERFLOW_DROP) return MOE_ERR_INVALID_ARG;     // re-routing: moe_forward only
  if (C < 0 || counts == nullptr || offsets == nullptr || dropped == nullptr) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (idx == nullptr || x == nullptr || pos == nullptr)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, C);
  if (L.rows > 0 && x_perm == nullptr) return MOE_ERR_INVALID_ARG;
  if (stalled_tile < 0 || stalled_tile >= L.nblk_dispatch) return MOE_ERR_INVALID_ARG;
  if ((shape->T > 0 && !aligned16(x)) || (L.rows > 0 && !aligned16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, C, ws, ws_bytes)) != MOE_OK) return st;
  return dispatch_impl(shape, C, const_cast<int32_t*>(idx), x, pos, counts, offsets, dropped, x_perm, nullptr, ws,
                       L, static_cast<cudaStream_t>(stream), stalled_tile);
}

static moe_status_t ffn_impl(const moe_shape_t* shape, const void* x_perm, const int32_t* offsets, const void* W1,
                             const void* W3, const void* W2, const float* b1, const float* b2, float* y_perm,
                             void* ws, const WsLayout& L, cudaStream_t st) {
  FfnParams fp{};
  fp.x_perm = x_perm;
  fp.offsets = offsets;
  fp.W1 = W1;
  fp.W3 = W3;
  fp.W2 = W2;
  fp.b1 = b1;
  fp.b2 = b2;
  fp.h = at<void>(ws, L.h);
  fp.y_perm = y_perm;
  fp.E = shape->E;
  fp.d = shape->d;
  fp.F = shape->d_ff;
  fp.act = shape->act;
  fp.rows = L.rows;
  fp.err = at<int>(ws, L.err);
  return cuda_status(shape->dtype == MOE_BF16 ? launch_ffn_bf16(fp, st) : launch_ffn_f32(fp, st));
}

static moe_status_t check_experts(const moe_shape_t* shape, const void* W1, const void* W3, const void* W2,
                                  const float* b1) {
  if (W1 == nullptr || W2 == nullptr) return MOE_ERR_INVALID_ARG;
  if (shape->act == MOE_ACT_SWIGLU && (W3 == nullptr || b1 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (shape->act == MOE_ACT_GELU && W3 != nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || (W3 && !aligned16(W3))) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static moe_status_t check_shared(const moe_shape_t* shape, const moe_shared_t* sh) {
  if (shape->d_ff_shared == 0) return sh == nullptr ? MOE_OK : MOE_ERR_INVALID_ARG;
  if (sh == nullptr || sh->W1s == nullptr || sh->W2s == nullptr) return MOE_ERR_INVALID_ARG;
  if (shape->act == MOE_ACT_SWIGLU && (sh->W3s == nullptr || sh->b1s != nullptr)) return MOE_ERR_INVALID_ARG;
  if (shape->act == MOE_ACT_GELU && sh->W3s != nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(sh->W1s) || !aligned16(sh->W2s) || (sh->W3s && !aligned16(sh->W3s))) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// the shared experts as one dense FFN over every token (no offsets: one group of T rows)
static moe_status_t shared_impl(const moe_shape_t* shape, const void* x, const moe_shared_t* sh, float* y_shared,
                                void* ws, const WsLayout& L, cudaStream_t st) {
  if (shape->T == 0) return MOE_OK;
  FfnParams fp{};
  fp.x_perm = x;
  fp.offsets = nullptr;
  fp.W1 = sh->W1s;
  fp.W3 = sh->W3s;
  fp.W2 = sh->W2s;
  fp.b1 = sh->b1s;
  fp.b2 = sh->b2s;
  fp.h = at<void>(ws, L.h_shared);
  fp.y_perm = y_shared;
  fp.E = 1;
  fp.d = shape->d;
  fp.F = shape->d_ff_shared;
  fp.act = shape->act;
  fp.rows = shape->T;
  fp.err = at<int>(ws, L.err);
  return cuda_status(shape->dtype == MOE_BF16 ? launch_ffn_bf16(fp, st) : launch_ffn_f32(fp, st));
}

moe_status_t moe_shared_ffn(const moe_shape_t* shape, const void* x, const moe_shared_t* shared, float* y_shared,
                            void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->d_ff_shared == 0) return MOE_ERR_INVALID_ARG;
  if ((st = check_shared(shape, shared)) != MOE_OK) return st;
  if (shape->T > 0 && (x == nullptr || y_shared == nullptr)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!aligned16(x) || !aligned16(y_shared))) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, 0, ws, ws_bytes)) != MOE_OK) return st;
  return shared_impl(shape, x, shared, y_shared, ws, ws_layout(*shape, 0), static_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn(const moe_shape_t* shape, int32_t C, const void* x_perm, const int32_t* offsets,
                            const void* W1, const void* W3, const void* W2, const float* b1, const float* b2,
                            float* y_perm, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (C < 0 || offsets == nullptr) return MOE_ERR_INVALID_ARG;
  if ((st = check_experts(shape, W1, W3, W2, b1)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*shape, C);
  if (L.rows > 0 && (x_perm == nullptr || y_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (L.rows > 0 && (!aligned16(x_perm) || !aligned16(y_perm))) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, C, ws, ws_bytes)) != MOE_OK) return st;
  return ffn_impl(shape, x_perm, offsets, W1, W3, W2, b1, b2, y_perm, ws, L, static_cast<cudaStream_t>(stream));
}

static moe_status_t combine_impl(const moe_shape_t* shape, long long rows, const float* y_perm, const int32_t* idx,
                                 const float* w, const int32_t* pos, const int32_t* offsets, const void* residual,
                                 const float* y_shared, void* out, float* moe_out, int* err, cudaStream_t st,
                                 const int32_t* row_of = nullptr) {
  CombineParams cp{};
  cp.y_perm = y_perm;
  cp.y_shared = y_shared;
  cp.row_of = row_of;
  cp.idx = idx;
  cp.w = w;
  cp.pos = pos;
  cp.offsets = offsets;
  cp.residual = residual;
  cp.out = out;
  cp.moe_out = moe_out;
  cp.T = static_cast<int>(shape->T);
  cp.k = shape->k;
  cp.d = shape->d;
  cp.E = shape->E;
  cp.rows = rows;
  cp.dtype = shape->dtype;
  cp.err = err;
  return cuda_status(launch_combine(cp, st));
}

moe_status_t moe_combine(const moe_shape_t* shape, int32_t C, const float* y_perm, const int32_t* idx,
                         const float* w, const int32_t* pos, const int32_t* offsets, const void* residual,
                         const float* y_shared, void* out, float* moe_out, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;  // token-choice tables
  if (C < 0) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (idx == nullptr || w == nullptr || pos == nullptr || offsets == nullptr || out == nullptr))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*shape, C);
  if (L.rows > 0 && y_perm == nullptr) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!aligned16(out) || (residual && !aligned16(residual)) || (moe_out && !aligned16(moe_out)) ||
                       (y_perm && !aligned16(y_perm)) || (y_shared && !aligned16(y_shared))))
    return MOE_ERR_UNSUPPORTED;
  return combine_impl(shape, L.rows, y_perm, idx, w, pos, offsets, residual, y_shared, out, moe_out, nullptr,
                      static_cast<cudaStream_t>(stream));
}

static moe_status_t forward_impl(const moe_shape_t* shape, double capacity_factor, int32_t C_override,
                                 const void* x, const float* W_g, const float* b_g, const float* W_noise,
                                 const float* eps, const void* W1, const void* W3, const void* W2, const float* b1,
                                 const float* b2, const moe_shared_t* shared, void* out, float* moe_out,
                                 int32_t* idx, float* w, int32_t* pos,
                                 int32_t* counts, int32_t* offsets, int64_t* dropped, int64_t* stats,
                                 float* logits, void* ws, size_t ws_bytes, void* stream,
                                 void* const* stage_events) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  int32_t C = C_override;
  if (C < 0) {
    C = moe_capacity(shape->T, shape->k, shape->E, capacity_factor);
    if (C < 0) return MOE_ERR_INVALID_ARG;
  }
  if (W_g == nullptr) return MOE_ERR_INVALID_ARG;
  if ((W_noise == nullptr) != (eps == nullptr)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (x == nullptr || out == nullptr)) return MOE_ERR_INVALID_ARG;
  if ((st = check_experts(shape, W1, W3, W2, b1)) != MOE_OK) return st;
  if ((st = check_shared(shape, shared)) != MOE_OK) return st;
  if (shape->T > 0 && (!aligned16(x) || !aligned16(out) || (moe_out && !aligned16(moe_out))))
    return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, C, ws, ws_bytes)) != MOE_OK) return st;

  const WsLayout L = ws_layout(*shape, C);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  NvtxRange whole("moe_forward");
  // Inside a stream capture the stage events become external event-record
  // nodes, which record (and time) on every graph launch.
  unsigned int rec_flags = cudaEventRecordDefault;
  if (stage_events != nullptr) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return MOE_ERR_CUDA;
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
  auto mark = [&](int i) -> moe_status_t {
    if (stage_events == nullptr || stage_events[i] == nullptr) return MOE_OK;
    return cuda_status(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(stage_events[i]), s, rec_flags));
  };
  const bool ec = shape->routing == MOE_ROUTE_EXPERT_CHOICE;
  if (ec && (idx != nullptr || w != nullptr || pos != nullptr)) return MOE_ERR_INVALID_ARG;
  // decode-sized batches whose router fits the fused kernel: one launch for the whole layer
  const bool self_route = L.dec && !ec && ffn_decode_routes(*shape, W_g, W_noise);
  if (idx == nullptr) idx = at<int32_t>(ws, L.idx);
  if (w == nullptr) w = at<float>(ws, L.w);
  if (pos == nullptr) pos = at<int32_t>(ws, L.pos);
  if (counts == nullptr) counts = at<int32_t>(ws, L.counts);
  if (offsets == nullptr) offsets = at<int32_t>(ws, L.offsets);
  if (dropped == nullptr) dropped = at<int64_t>(ws, L.dropped);

  if ((st = mark(0)) != MOE_OK) return st;
  // the shared experts need no routing: their FFN runs first
  float* y_sh = nullptr;
  if (shape->d_ff_shared > 0) {
    NvtxRange r("shared_ffn");
    y_sh = at<float>(ws, L.y_shared);
    if ((st = shared_impl(shape, x, shared, y_sh, ws, L, s)) != MOE_OK) return st;
  }
  int32_t* row_of = at<int32_t>(ws, L.row_of);
  const float* gate = w;
  moe_shape_t cshape = *shape;  // the combine's view: k ranks per token
  if (ec) {
    EcParams ep{};
    {
      NvtxRange r("router_expert_choice");
      if ((st = ec_route_impl(shape, x, W_g, b_g, W_noise, eps, logits, ws, L, s, ep)) != MOE_OK) return st;
    }
    if ((st = mark(1)) != MOE_OK) return st;
    NvtxRange r("dispatch_gather");
    if (shape->T == 0) {
      if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * shape->E, s) != cudaSuccess ||
          cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (shape->E + 1), s) != cudaSuccess ||
          cudaMemsetAsync(dropped, 0, sizeof(int64_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else {
      if ((st = cuda_status(launch_ec_finalize(ep, counts, offsets, reinterpret_cast<long long*>(dropped), s))) !=
          MOE_OK)
        return st;
      if ((st = cuda_status(launch_ec_gather(ep, x, at<void>(ws, L.x_perm),
                                             static_cast<int>(dtype_bytes(shape->dtype)), s))) != MOE_OK)
        return st;
    }
    // the combine sees every expert as a "rank" of each token: row_of [T,E], gates [T,E]
    row_of = ep.row_of;
    gate = ep.gate_te;
    cshape.k = shape->E;
  } else if (self_route) {
    // the fused decode kernel routes and dispatches the batch itself (its first tiles)
    if ((st = mark(1)) != MOE_OK) return st;
  } else {
    int32_t* backup = shape->overflow == MOE_OVERFLOW_REROUTE ? at<int32_t>(ws, L.rr_backup) : nullptr;
    // decode-sized batches: the router and the dispatch let the fused expert
    // FFN launch at once (its first phase needs no routing), and there is no
    // gather (the FFN reads the tokens themselves)
    {
      NvtxRange r("router");
      if ((st = route_impl(shape, x, W_g, b_g, W_noise, eps, idx, w, logits, stats, backup, nullptr, s,
                           at<void>(ws, L.rt_scratch), L.rt_scratch_bytes, L.dec)) != MOE_OK)
        return st;
    }
    if ((st = mark(1)) != MOE_OK) return st;
    NvtxRange r("dispatch_gather");
    if ((st = dispatch_impl(shape, C, idx, x, pos, counts, offsets, dropped, at<void>(ws, L.x_perm), nullptr, ws, L,
                            s, -1, row_of, backup, L.dec, !L.dec)) != MOE_OK)
      return st;
  }
  if ((st = mark(2)) != MOE_OK) return st;
  float* y_perm = at<float>(ws, L.y_perm);
  FfnParams fp{};
  fp.x_perm = at<void>(ws, L.x_perm);
  fp.offsets = offsets;
  fp.W1 = W1;
  fp.W3 = W3;
  fp.W2 = W2;
  fp.b1 = b1;
  fp.b2 = b2;
  fp.h = at<void>(ws, L.h);
  fp.y_perm = y_perm;
  fp.E = shape->E;
  fp.d = shape->d;
  fp.F = shape->d_ff;
  fp.act = shape->act;
  fp.rows = L.rows;
  fp.err = at<int>(ws, L.err);
  if (L.dec && !ec) {
    // one kernel for both expert GEMMs (stage event 3 follows both)
    DecodeFfnParams dp{};
    dp.x = x;
    dp.T = static_cast<int>(shape->T);
    dp.d = shape->d;
    dp.F = shape->d_ff;
    dp.E = shape->E;
    dp.k = shape->k;
    dp.act = shape->act;
    dp.W1 = W1;
    dp.W3 = W3;
    dp.W2 = W2;
    dp.b1 = b1;
    dp.b2 = b2;
    dp.h = at<void>(ws, L.dec_h);
    dp.idx = idx;
    dp.pos = pos;
    dp.offsets = offsets;
    dp.y_perm = y_perm;
    dp.rows = L.rows;
    dp.ctrl = at<int>(ws, L.dec_ctrl);
    dp.err = at<int>(ws, L.err);
    dp.w = w;
    dp.y_shared = y_sh;
    dp.out = out;
    dp.moe_out = moe_out;
    if (self_route) {
      dp.self_route = 1;
      dp.W_g = W_g;
      dp.b_g = b_g;
      dp.W_n = W_noise;
      dp.eps = eps;
      dp.gate_raw = shape->gates == MOE_GATES_RAW ? 1 : 0;
      dp.C = C;
      dp.logits = logits;
      dp.stats = reinterpret_cast<long long*>(stats);
      dp.counts = counts;
      dp.dropped = reinterpret_cast<long long*>(dropped);
      dp.row_of = at<int32_t>(ws, L.row_of);
    }
    if ((st = cuda_status(launch_ffn_decode(dp, s))) != MOE_OK) return st;
    // the same kernel did the combine: stage events 3, 4 and 5 all follow it
    if ((st = mark(3)) != MOE_OK) return st;
    if ((st = mark(4)) != MOE_OK) return st;
    return mark(5);
  } else if (shape->dtype == MOE_BF16) {
    // launch_ffn_bf16 names its two GEMMs (expert_gemm1, expert_gemm2) itself
    if ((st = cuda_status(launch_ffn_bf16(fp, s, stage_events ? static_cast<cudaEvent_t>(stage_events[3]) : nullptr))) != MOE_OK)
      return st;
  } else {
    NvtxRange r("expert_ffn_f32");
    if ((st = cuda_status(launch_ffn_f32(fp, s))) != MOE_OK) return st;
    if ((st = mark(3)) != MOE_OK) return st;
  }
  if ((st = mark(4)) != MOE_OK) return st;
  NvtxRange rc("combine");
  if ((st = combine_impl(&cshape, L.rows, y_perm, idx, gate, pos, offsets, x, y_sh, out, moe_out, at<int>(ws, L.err), s,
                        row_of)) != MOE_OK)
    return st;
  return mark(5);
}

moe_status_t moe_forward(const moe_shape_t* shape, double capacity_factor, int32_t C_override, const void* x,
                         const float* W_g, const float* b_g, const float* W_noise, const float* eps, const void* W1,
                         const void* W3, const void* W2, const float* b1, const float* b2, const moe_shared_t* shared,
                         void* out, float* moe_out, int32_t* idx, float* w, int32_t* pos, int32_t* counts,
                         int32_t* offsets, int64_t* dropped, int64_t* stats, float* logits, void* ws, size_t ws_bytes,
                         void* stream) {
  return forward_impl(shape, capacity_factor, C_override, x, W_g, b_g, W_noise, eps, W1, W3, W2, b1, b2, shared, out,
                      moe_out, idx, w, pos, counts, offsets, dropped, stats, logits, ws, ws_bytes, stream, nullptr);
}

moe_status_t moe_forward_timed(const moe_shape_t* shape, double capacity_factor, int32_t C_override, const void* x,
                               const float* W_g, const float* b_g, const float* W_noise, const float* eps,
                               const void* W1, const void* W3, const void* W2, const float* b1, const float* b2,
                               const moe_shared_t* shared, void* out, float* moe_out, int32_t* idx, float* w,
                               int32_t* pos, int32_t* counts, int32_t* offsets, int64_t* dropped, int64_t* stats,
                               float* logits, void* ws, size_t ws_bytes, void* stream, void* const* stage_events) {
  if (stage_events == nullptr) return MOE_ERR_INVALID_ARG;
  return forward_impl(shape, capacity_factor, C_override, x, W_g, b_g, W_noise, eps, W1, W3, W2, b1, b2, shared, out,
                      moe_out, idx, w, pos, counts, offsets, dropped, stats, logits, ws, ws_bytes, stream,
                      stage_events);
}

moe_status_t moe_routing_stats(const moe_shape_t* shape, const float* logits, const int32_t* idx,
                               const int32_t* counts, const int64_t* dropped, double* f, double* P, double* summary,
                               void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (counts == nullptr || dropped == nullptr || f == nullptr || P == nullptr || summary == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (logits == nullptr || idx == nullptr)) return MOE_ERR_INVALID_ARG;
  // the stats regions precede every capacity-dependent region, so any C's workspace holds them
  if ((st = check_ws(shape, 0, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*shape, 0);
  StatsParams p{};
  p.logits = logits;
  p.idx = idx;
  p.counts = counts;
  p.dropped = reinterpret_cast<const long long*>(dropped);
  p.T = shape->T;
  p.E = shape->E;
  p.k = shape->k;
  p.f = f;
  p.P = P;
  p.summary = summary;
  p.acc = at<unsigned long long>(ws, L.stats_acc);
  p.ticket = at<int>(ws, L.stats_ticket);
  p.err = at<int>(ws, L.err);
  return cuda_status(launch_routing_stats(p, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_testing_router_filter(const moe_shape_t* shape, const void* x, const float* W_g,
                                       const float* W_noise, float* approx, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  if (x == nullptr || W_g == nullptr || approx == nullptr) return MOE_ERR_INVALID_ARG;
  const int nc = W_noise ? 2 * shape->E : shape->E;
  if (shape->dtype != MOE_BF16 || nc % 32 != 0 || nc > 256 || shape->T < 1) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(approx)) return MOE_ERR_UNSUPPORTED;
  if ((st = check_ws(shape, 0, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*shape, 0);
  RouterParams p{};
  p.x = x;
  p.W_g = W_g;
  p.W_n = W_noise;
  p.T = static_cast<int>(shape->T);
  p.d = shape->d;
  p.E = shape->E;
  p.k = shape->k;
  p.err = at<int>(ws, L.err);
  return cuda_status(launch_router_tc_filter(p, at<void>(ws, L.rt_scratch), approx, static_cast<cudaStream_t>(stream)));
}

unsigned long long moe_kernel_launches(void) { return launch_count().load(std::memory_order_relaxed); }

moe_status_t moe_get_device_error(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (code != 0) {
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return static_cast<moe_status_t>(code);
}

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: valid but outside the supported set";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
    case MOE_ERR_BOUNDS: return "MOE_ERR_BOUNDS: a device-side index check failed";
  }
  return "unknown moe_status_t";
}

}  // extern "C"
