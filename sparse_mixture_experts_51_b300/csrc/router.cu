// Router: logits, exact top-k selection and renormalised gates.
//
// Logits H = x W_g + b_g (+ eps * softplus(x W_noise)) follow the noisy top-k
// gating of "LLM part 09: Sparse Mixture-of-Experts (MoE)", s2; the gates are
// the softmax over the k selected logits (same section, and the renormalised
// top-k of "Mixture-of-experts Models", Level 2).
//
// The logits are a skinny fp32 contraction [T,d] x [d,nc], nc = E (or 2E
// with the noise projection).  Two kernels cover the shapes:
//
//  * router_warp_kernel (nc <= 16, the router weights fit in shared memory):
//    HBM-bound.  Persistent CTAs stage W^T once; a warp takes TW tokens at a
//    time, lanes stride over d with 8- or 16-byte loads, every lane keeps a
//    TW x NC accumulator, and a butterfly reduce-scatter leaves one logit per
//    lane.
//  * router_tiled_kernel (router_tiled.cu; wider nc, or weights too large
//    for shared memory): FMA-bound.  A thread-block cluster of KS CTAs owns
//    a tile of TB tokens and every column; CTA r reduces over its own slice
//    of d through a 4-stage cp.async ring, every thread keeps a TM x 4
//    register tile, and the KS partial tiles are summed in rank order
//    through distributed shared memory.
//
// Exactness.  Both kernels sum in short chunks with a known summation depth
// n_eff, so the rounding error of a logit is at most
// gamma(n_eff) * ||x_t|| * ||W_col|| (Cauchy-Schwarz).  The ranking step
// evaluates this bound per token and expert together with the error of the
// bias add and of the softplus noise term.  When the bound separates the k
// selected logits from each other and from every other expert, the fp32
// order is the exact order.  Otherwise the warp re-evaluates every expert
// that could still be in the top k in fp64 and ranks those values (ties ->
// lower expert index).  Either way the selected experts and their order are
// those of the exactly computed logits.  Only the ranks that the bound does
// not settle are re-evaluated: the leading ranks whose lower ends lie above
// every expert ranked below them keep their fp32 order.
#include <mutex>

#include "router_rank.cuh"

namespace moe {
namespace {

using namespace router_detail;

constexpr int WT = 384;   // threads per CTA, warp kernel

// ================================================================ warp kernel
// Shared memory: Wt [NC][ldw] fp32 (column c of [W_g | W_noise] as a row,
// zero rows for c >= nc), red [WT/32][40] per-warp reduced logits and token
// norms, cn2 [NC] (column norms of the combined weight),
// cnt [2].  ldw = d rounded up to 128, plus 4 (conflict-free transposed store).
struct WarpPlan {
  int nc;       // logit columns
  int ldw;      // row stride of Wt (floats), multiple of 4
  int groups;   // 128-element groups of d per token row (4 elements per lane)
  int n_eff;    // summation depth for the error bound
  long long ngroups_tok;  // token groups of TW tokens
};

template <typename TX, int NC, int TW>
__global__ void __launch_bounds__(WT, 1) router_warp_kernel(RouterParams p, WarpPlan q) {
  extern __shared__ __align__(16) float smem[];
  constexpr int NVAL = TW * NC;            // accumulators per lane (power of two <= 32)
  constexpr int LV = NVAL >= 32 ? 5 : NVAL >= 16 ? 4 : NVAL >= 8 ? 3 : NVAL >= 4 ? 2 : NVAL >= 2 ? 1 : 0;
  constexpr int CH = (sizeof(TX) == 2 ? 8 : 4) / TW;  // 128-element groups per load batch (64 B per lane)
  using V = Vec4<TX>;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, d = p.d, nc = q.nc, ldw = q.ldw;
  float* Wt = smem;                               // [NC][ldw]
  float* red = smem + NC * ldw;                   // [WT/32][40]: 32 reduced logits + TW norms
  float* cn2 = red + (WT / 32) * 40;              // [NC]
  int* cnt = reinterpret_cast<int*>(cn2 + NC);    // [2]
  const TX* x = static_cast<const TX*>(p.x);

  pdl_wait();  // tokens (and weights) may be the predecessor's output
  if (p.early_trigger) pdl_trigger();
  // ---- stage the router weights, transposed, with 4-byte asynchronous
  // copies (all in flight at once); zero rows and tail padding
  for (int i = tid; i < d * NC; i += WT) {
    const int j = i / NC, c = i - j * NC;
    const float* src = p.W_g;
    if (c < nc) src = c < E ? p.W_g + static_cast<size_t>(j) * E + c : p.W_n + static_cast<size_t>(j) * E + (c - E);
    cp_async4(Wt + c * ldw + j, src, c < nc);
  }
  cp_async_commit();
  const int pad = ldw - d;
  for (int i = tid; i < NC * pad; i += WT) {
    const int c = i / pad, j = d + (i - c * pad);
    Wt[c * ldw + j] = 0.f;
  }
  if (tid < 2) cnt[tid] = 0;
  cp_async_wait_all();
  __syncthreads();
  for (int c = warp; c < NC; c += WT / 32) {
    float s2 = 0.f;
    for (int j = lane; j < d; j += 32) s2 = fmaf(Wt[c * ldw + j], Wt[c * ldw + j], s2);
    s2 = warp_sum(s2);
    if (lane == 0) cn2[c] = sqrtf(s2);  // the column norm itself: every token's bound uses it
  }
  __syncthreads();

  const float gam = (q.n_eff * kU) / (1.0f - q.n_eff * kU);
  int n_recomputed = 0, n_near = 0;
  float* myred = red + warp * 40;
  const long long wstride = static_cast<long long>(gridDim.x) * (WT / 32);

  for (long long grp = static_cast<long long>(blockIdx.x) * (WT / 32) + warp; grp < q.ngroups_tok; grp += wstride) {
    const long long tbase = grp * TW;
    // the noise of this batch's tokens, requested before the contraction so
    // its memory latency is hidden behind it
    float ep[TW][1];
#pragma unroll
    for (int u = 0; u < TW; ++u) load_eps<1>(p, tbase + u, lane, ep[u]);
    float acc[TW][NC], sq[TW];
#pragma unroll
    for (int u = 0; u < TW; ++u) {
      sq[u] = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[u][c] = 0.f;
    }
    // ---- batches of CH groups x TW tokens (4 elements per lane each), two
    // batches in flight: the next batch is loaded before this one is multiplied
    auto load_batch = [&](typename V::raw (&xr)[TW][CH], int g0) {
#pragma unroll
      for (int u = 0; u < TW; ++u) {
        const long long t = tbase + u;
#pragma unroll
        for (int gi = 0; gi < CH; ++gi) {
          const int j = (g0 + gi) * 128 + lane * 4;
          xr[u][gi] = (t < p.T && j < d) ? V::load(x + t * d + j) : V::zero();
        }
      }
    };
    auto mul_batch = [&](const typename V::raw (&xr)[TW][CH], int g0) {
      float cacc[TW][NC];
#pragma unroll
      for (int u = 0; u < TW; ++u)
#pragma unroll
        for (int c = 0; c < NC; ++c) cacc[u][c] = 0.f;
#pragma unroll
      for (int gi = 0; gi < CH; ++gi) {
        if (g0 + gi >= q.groups) break;  // past the row: nothing left in this batch
        const int j = (g0 + gi) * 128 + lane * 4;
        float xv[TW][4];
#pragma unroll
        for (int u = 0; u < TW; ++u) {
          V::unpack(xr[u][gi], xv[u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) sq[u] = fmaf(xv[u][i], xv[u][i], sq[u]);
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float4 w4 = *reinterpret_cast<const float4*>(&Wt[c * ldw + j]);
#pragma unroll
          for (int u = 0; u < TW; ++u) {
            cacc[u][c] = fmaf(xv[u][0], w4.x, cacc[u][c]);
            cacc[u][c] = fmaf(xv[u][1], w4.y, cacc[u][c]);
            cacc[u][c] = fmaf(xv[u][2], w4.z, cacc[u][c]);
            cacc[u][c] = fmaf(xv[u][3], w4.w, cacc[u][c]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < TW; ++u)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[u][c] += cacc[u][c];
    };
    typename V::raw xa[TW][CH], xb[TW][CH];
    load_batch(xa, 0);
    for (int g0 = 0; g0 < q.groups; g0 += 2 * CH) {
      if (g0 + CH < q.groups) load_batch(xb, g0 + CH);
      mul_batch(xa, g0);
      if (g0 + CH >= q.groups) break;
      if (g0 + 2 * CH < q.groups) load_batch(xa, g0 + 2 * CH);
      mul_batch(xb, g0 + CH);
    }

    // ---- butterfly reduce-scatter: lane l ends with value l >> (5 - LV), value v = u*NC + c
    float vals[NVAL];
#pragma unroll
    for (int u = 0; u < TW; ++u)
#pragma unroll
      for (int c = 0; c < NC; ++c) vals[u * NC + c] = acc[u][c];
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
      const int o = 16 >> lvl;
      if (lvl < LV) {
        const int half = NVAL >> (lvl + 1);  // values kept after this step
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < NVAL / 2; ++i) {
          if (i < half) {
            const float send = upper ? vals[i] : vals[i + half];
            const float keep = upper ? vals[i + half] : vals[i];
            vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
      } else {
        vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], o);
      }
    }
#pragma unroll
    for (int u = 0; u < TW; ++u) {
      sq[u] = warp_sum(sq[u]);
      if (lane == 0) myred[32 + u] = sq[u];
    }
    if ((lane & ((1 << (5 - LV)) - 1)) == 0) myred[lane >> (5 - LV)] = vals[0];
    __syncwarp();

#pragma unroll 1
    for (int u = 0; u < TW; ++u) {
      const long long t = tbase + u;
      if (t >= p.T) break;
      float g[1], z[1];
      g[0] = lane < E ? myred[u * NC + lane] : 0.f;
      z[0] = (p.W_n != nullptr && lane < E) ? myred[u * NC + E + lane] : 0.f;
      auto wcol = [&](int c, int j) { return *reinterpret_cast<const float4*>(&Wt[c * ldw + j]); };
      const float xb[1] = {0.f};
      rank_token<TX, 1>(p, t, lane, g, z, ep[u], sqrtf(myred[32 + u]), cn2, gam, wcol, n_recomputed, n_near, xb);
    }
    __syncwarp();
  }

  pdl_trigger();
  if (p.stats) flush_stats(p, cnt, lane, n_recomputed, n_near);
}

// ---------------------------------------------------------------- host side
// Device facts cached per device: SM count and opt-in shared memory.
struct DevInfo {
  int sms = 0;
  int max_smem_optin = 0;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

template <typename TX, int NC, int TW>
cudaError_t launch_warp(const RouterParams& p, const WarpPlan& q, int smem_bytes, int grid, cudaStream_t st) {
  auto kern = router_warp_kernel<TX, NC, TW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(WT), static_cast<size_t>(smem_bytes), st, 1, p, q);
}

// The warp kernel, for nc <= 16 when the transposed weights fit in shared
// memory.  Returns cudaErrorNotSupported when the shape is not for it.
template <typename TX>
cudaError_t try_warp_kernel(const RouterParams& p, cudaStream_t st, const DevInfo& di) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  if (nc > 16) return cudaErrorNotSupported;
  const int NC = nc <= 4 ? 4 : nc <= 8 ? 8 : 16;
  const int groups = (p.d + 127) / 128;
  const int ldw = groups * 128 + 4;  // every lane's 4-element group stays inside the row
  const size_t smem = sizeof(float) * (static_cast<size_t>(NC) * ldw + (WT / 32) * 40 + NC) + 2 * sizeof(int);
  if (smem > static_cast<size_t>(di.max_smem_optin)) return cudaErrorNotSupported;
  // tokens per warp group: the most that still gives every warp one group
  const long long warps_total = static_cast<long long>(di.sms) * (WT / 32);
  int TW = 1;
  for (int cand : {4, 2}) {
    if (cand * NC > 32) continue;  // at most 32 accumulators per lane
    if ((static_cast<long long>(p.T) + cand - 1) / cand >= warps_total) { TW = cand; break; }
  }
  WarpPlan q{};
  q.nc = nc;
  q.ldw = ldw;
  q.groups = groups;
  const int CH = (sizeof(TX) == 2 ? 8 : 4) / TW;
  // per lane: 4*CH products per batch, then one add per batch, then 5 tree levels
  q.n_eff = 4 * CH + (groups + CH - 1) / CH + 5;
  q.ngroups_tok = (static_cast<long long>(p.T) + TW - 1) / TW;
  const long long want = (q.ngroups_tok + (WT / 32) - 1) / (WT / 32);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(di.sms, want)));
  const int sb = static_cast<int>(smem);
  if (NC == 4) {
    if (TW == 4) return launch_warp<TX, 4, 4>(p, q, sb, grid, st);
    if (TW == 2) return launch_warp<TX, 4, 2>(p, q, sb, grid, st);
    return launch_warp<TX, 4, 1>(p, q, sb, grid, st);
  }
  if (NC == 8) {
    if (TW == 4) return launch_warp<TX, 8, 4>(p, q, sb, grid, st);
    if (TW == 2) return launch_warp<TX, 8, 2>(p, q, sb, grid, st);
    return launch_warp<TX, 8, 1>(p, q, sb, grid, st);
  }
  if (TW == 2) return launch_warp<TX, 16, 2>(p, q, sb, grid, st);
  return launch_warp<TX, 16, 1>(p, q, sb, grid, st);
}

template <typename TX>
cudaError_t launch_typed(const RouterParams& p, int dtype, cudaStream_t st, const DevInfo& di) {
  const cudaError_t e = try_warp_kernel<TX>(p, st, di);
  if (e != cudaErrorNotSupported) return e;
  return launch_router_tiled(p, dtype, st, di.sms);
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, int dtype, cudaStream_t st) {
  // wide logit tables of long bf16 batches: the tensor-core filter path
  if (p.T > 0 && p.scratch != nullptr && router_tc_applies(p, dtype) &&
      p.scratch_bytes >= router_tc_scratch_bytes(p.T, p.d, p.E))
    return launch_router_tc(p, p.scratch, st);
  if (p.T == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_dev_once[dev], [dev] {
    DevInfo di;
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) di.sms = 148;
    if (cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      di.max_smem_optin = 227 * 1024;
    g_dev[dev] = di;
  });
  const DevInfo& di = g_dev[dev];
  return dtype == MOE_BF16 ? launch_typed<__nv_bfloat16>(p, dtype, st, di) : launch_typed<float>(p, dtype, st, di);
}

}  // namespace moe
