// Router for wide logit tables (nc = E or 2E > 16 columns), or weights too
// large to stage whole in shared memory: an FMA-bound skinny contraction.
//
// Logits H = x W_g + b_g (+ eps * softplus(x W_noise)) ("LLM part 09:
// Sparse Mixture-of-Experts (MoE)", s2), exact top-k and gates as in
// router.cu.
//
// A thread-block cluster of KS CTAs owns a tile of TB tokens and all nc
// columns; CTA r of the cluster reduces over its own run of 32-wide slices
// of d.  Per slice, a 4-stage ring of cp.async copies brings the raw token
// slice and the weight slice into shared memory three slices ahead; the
// token slice is widened to fp32 and transposed into one of two buffers;
// every thread multiplies a TM-token x 4-column register tile.  The KS
// partial tiles (and the partial norms the error bound needs) are summed in
// rank order through distributed shared memory, and the CTAs of the cluster
// share the per-token ranking.  Short batches (the decode-like layer) get
// enough CTAs from the cluster split alone and need a single memory round
// trip for their whole slice run.
//
// Summation depth for the error bound: 32 products per slice, the slices of
// one CTA in order, then the KS partials: n_eff = 32 + slices per CTA + KS.
#include <cooperative_groups.h>

#include <mutex>

#include "router_rank.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

using namespace router_detail;

constexpr int RT = 256;          // threads per CTA
constexpr int DK = 32;           // d-slice per pipeline step (and summation chunk)
constexpr int STAGES = 4;        // cp.async ring depth
constexpr int kMaxCluster = 16;  // CTAs per cluster (16 needs the non-portable opt-in)

struct TiledPlan {
  int KS;        // CTAs per cluster (d split)
  int nch;       // 32-wide slices of d
  int nch_per;   // slices per CTA
  int nc;        // logit columns (E, or 2E with noise)
  int vec_w;     // 1 if router weight rows are read 16 bytes at a time (E % 4 == 0, aligned)
};

template <typename TX, int CQ, int TM>
struct Tile {
  static constexpr int NCP = 4 * CQ;                   // padded columns
  static constexpr int TG = RT / CQ;                   // token groups
  static constexpr int TB = TG * TM;                   // tokens per tile
  static constexpr int XS_LD = TB + 4;                 // transposed-x row stride (floats)
  static constexpr int VEC = 16 / static_cast<int>(sizeof(TX));  // elements per 16-byte chunk
  static constexpr int VPT = DK / VEC;                 // chunks per token per slice
  static constexpr int RS = DK * static_cast<int>(sizeof(TX)) + 16;  // raw row stride (bytes, conflict-free)
  static constexpr int NV = (TB * VPT + RT - 1) / RT;  // chunks per thread per slice
  static constexpr int LT_LD = NCP + 1;
  // byte offsets in dynamic shared memory
  static constexpr int XT_BYTES = 2 * DK * XS_LD * 4;
  static constexpr int WR_BYTES = STAGES * DK * NCP * 4;
  static constexpr int XR_BYTES = STAGES * TB * RS;
  static constexpr int OFF_WR = XT_BYTES;
  static constexpr int OFF_XR = OFF_WR + WR_BYTES;
  static constexpr int STAGE_END = OFF_XR + XR_BYTES;
  static constexpr int LT_BYTES = TB * LT_LD * 4;
  static constexpr int OFF_XSQ = ((STAGE_END > LT_BYTES ? STAGE_END : LT_BYTES) + 15) / 16 * 16;
  static constexpr int OFF_CN2P = OFF_XSQ + (TB * 4 + 15) / 16 * 16;
  static constexpr int OFF_CN2F = OFF_CN2P + NCP * 4;
  static constexpr int OFF_WQ = OFF_CN2F + NCP * 4;
  static constexpr int OFF_VSQ = OFF_WQ + RT * 4;
  static constexpr int OFF_CNT = OFF_VSQ + (NV * RT * 4 + 15) / 16 * 16;
  static constexpr int SMEM = OFF_CNT + 16;
};

__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// SL: 32-expert slots a lane holds while ranking (E <= 32 * SL).
template <typename TX, int CQ, int TM, int SL>
__global__ void __launch_bounds__(RT, 2) router_tiled_kernel(RouterParams p, TiledPlan q) {
  using G = Tile<TX, CQ, TM>;
  constexpr int NCP = G::NCP, TB = G::TB, XS_LD = G::XS_LD, VEC = G::VEC, VPT = G::VPT, RS = G::RS;
  constexpr int NV = G::NV;
  constexpr int SLOTS = SL;
  extern __shared__ __align__(16) uint8_t smem[];
  float* xt = reinterpret_cast<float*>(smem);                  // [2][DK][XS_LD]
  float* wr = reinterpret_cast<float*>(smem + G::OFF_WR);      // [STAGES][DK][NCP]
  uint8_t* xr = smem + G::OFF_XR;                              // [STAGES][TB][RS] raw token slices

  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % CQ, tg = tid / CQ;
  const int KS = q.KS;
  const int E = p.E, d = p.d, nc = q.nc;
  const bool noisy = p.W_n != nullptr;
  const int rank = static_cast<int>(blockIdx.y);  // == cluster.block_rank(): the cluster spans y
  const long long t0 = static_cast<long long>(blockIdx.x) * TB;
  const TX* x = static_cast<const TX*>(p.x);
  const int ch0 = rank * q.nch_per;
  const int nloc = max(0, min(q.nch, ch0 + q.nch_per) - ch0);

  pdl_wait();  // tokens (and weights) may be the predecessor's output
  if (p.early_trigger) pdl_trigger();
  float sq[NV];
  float wsq = 0.f;  // sum of W^2 of column (tid mod NCP) over this CTA's rows
#pragma unroll
  for (int s = 0; s < NV; ++s) sq[s] = 0.f;

  // -------- slice `ch` (token chunks and weight rows) -> ring slot, asynchronously
  auto issue = [&](int ch, int slot) {
    const int j0 = ch * DK;
    uint8_t* xs = xr + slot * TB * RS;
    for (int v = tid; v < TB * VPT; v += RT) {
      const int jv = v / TB, tl = v - jv * TB;
      const long long t = t0 + tl;
      const int j = j0 + jv * VEC;
      const bool ok = t < p.T && j < d;
      const TX* src = ok ? x + t * d + j : x;
      cp_async16(reinterpret_cast<float*>(xs + tl * RS + jv * 16), reinterpret_cast<const float*>(src), ok);
    }
    float* wb = wr + slot * DK * NCP;
    if (q.vec_w) {
      for (int i = tid; i < DK * CQ; i += RT) {
        const int jj = i / CQ, c0 = (i - jj * CQ) * 4, j = j0 + jj;
        const bool ok = j < d && c0 < nc;
        const float* src = p.W_g;
        if (ok) src = c0 < E ? p.W_g + static_cast<size_t>(j) * E + c0 : p.W_n + static_cast<size_t>(j) * E + (c0 - E);
        cp_async16(wb + i * 4, src, ok);
      }
    } else {
      for (int i = tid; i < DK * NCP; i += RT) {
        const int jj = i / NCP, c = i - jj * NCP, j = j0 + jj;
        const bool ok = j < d && c < nc;
        const float* src = p.W_g;
        if (ok) src = c < E ? p.W_g + static_cast<size_t>(j) * E + c : p.W_n + static_cast<size_t>(j) * E + (c - E);
        cp_async4(wb + i, src, ok);
      }
    }
  };
  // -------- raw slice in ring slot -> transposed fp32 buffer b; squared norms
  auto convert = [&](int slot, int b) {
    const uint8_t* xs = xr + slot * TB * RS;
    float* xb = xt + b * DK * XS_LD;
#pragma unroll
    for (int s = 0; s < NV; ++s) {
      const int v = tid + s * RT;
      if (v < TB * VPT) {
        const int jv = v / TB, tl = v - jv * TB;
        const uint4 raw = *reinterpret_cast<const uint4*>(xs + tl * RS + jv * 16);
        float vals[8];
        Vec16<TX>::unpack(raw, vals);
#pragma unroll
        for (int e2 = 0; e2 < VEC; ++e2) {
          xb[(jv * VEC + e2) * XS_LD + tl] = vals[e2];
          sq[s] = fmaf(vals[e2], vals[e2], sq[s]);
        }
      }
    }
    const float* wb = wr + slot * DK * NCP;
    for (int e2 = tid; e2 < DK * NCP; e2 += RT) wsq = fmaf(wb[e2], wb[e2], wsq);
  };

  float acc[TM][4];
#pragma unroll
  for (int m = 0; m < TM; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = 0.f;

  // -------- pipeline: slices 0..STAGES-2 in flight, then one slice per step
#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) {
    if (i < nloc) issue(ch0 + i, i);
    cp_async_commit();  // possibly empty: keeps the group count uniform
  }
  cp_async_wait_2();  // slice 0 of this thread landed
  __syncthreads();
  if (nloc > 0) convert(0, 0);
  for (int i = 0; i < nloc; ++i) {
    cp_async_wait_1();  // slice i+1 of this thread landed
    __syncthreads();    // every copy of slice i+1, every convert of slice i visible; slice i-1 fully used
    if (i + STAGES - 1 < nloc) issue(ch0 + i + STAGES - 1, (i + STAGES - 1) % STAGES);
    cp_async_commit();
    if (i + 1 < nloc) convert((i + 1) % STAGES, (i + 1) & 1);
    const float* xb = xt + (i & 1) * DK * XS_LD;
    const float* wb = wr + (i % STAGES) * DK * NCP;
    float cacc[TM][4];
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) cacc[m][c] = 0.f;
#pragma unroll 8
    for (int jj = 0; jj < DK; ++jj) {
      const float4 wv = *reinterpret_cast<const float4*>(&wb[jj * NCP + 4 * cq]);
      float xv[TM];
      const float* xp = &xb[jj * XS_LD + tg * TM];
      if constexpr (TM % 4 == 0) {
#pragma unroll
        for (int m = 0; m < TM; m += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(xp + m);
          xv[m] = t4.x; xv[m + 1] = t4.y; xv[m + 2] = t4.z; xv[m + 3] = t4.w;
        }
      } else if constexpr (TM == 2) {
        const float2 t2 = *reinterpret_cast<const float2*>(xp);
        xv[0] = t2.x; xv[1] = t2.y;
      } else {
        xv[0] = xp[0];
      }
#pragma unroll
      for (int m = 0; m < TM; ++m) {
        cacc[m][0] = fmaf(xv[m], wv.x, cacc[m][0]);
        cacc[m][1] = fmaf(xv[m], wv.y, cacc[m][1]);
        cacc[m][2] = fmaf(xv[m], wv.z, cacc[m][2]);
        cacc[m][3] = fmaf(xv[m], wv.w, cacc[m][3]);
      }
    }
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][c] += cacc[m][c];
  }
  cp_async_wait_all();
  pdl_trigger();
  // the noise of this warp's first token to rank: requested now, used after
  // the cluster-wide reduction below
  const int tl_first = rank * (RT / 32) + warp, tl_step = KS * (RT / 32);
  float ep_cur[SLOTS];
  load_eps<SLOTS>(p, t0 + tl_first, lane, ep_cur);
  __syncthreads();  // the slice buffers are dead: the partial-logit tile may alias them

  // -------- park this CTA's partial logits and norms in shared memory
  float* Lt = reinterpret_cast<float*>(smem);                   // [TB][LT_LD]
  float* xsq = reinterpret_cast<float*>(smem + G::OFF_XSQ);     // [TB]   partial ||x_t||^2
  float* cn2p = reinterpret_cast<float*>(smem + G::OFF_CN2P);   // [NCP]  partial column sums of W^2
  float* cn2f = reinterpret_cast<float*>(smem + G::OFF_CN2F);   // [NCP]  full column norms (not squared)
  float* wq = reinterpret_cast<float*>(smem + G::OFF_WQ);       // [RT]   per-thread W^2 partials
  float* vsq = reinterpret_cast<float*>(smem + G::OFF_VSQ);     // [NV*RT] per-chunk x^2 partials
  int* cnt = reinterpret_cast<int*>(smem + G::OFF_CNT);
  if (tid < 2) cnt[tid] = 0;
#pragma unroll
  for (int m = 0; m < TM; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) Lt[(tg * TM + m) * G::LT_LD + 4 * cq + c] = acc[m][c];
#pragma unroll
  for (int s = 0; s < NV; ++s) vsq[tid + s * RT] = sq[s];
  wq[tid] = wsq;
  __syncthreads();
  for (int tl = tid; tl < TB; tl += RT) {
    float s2 = 0.f;
    for (int jv = 0; jv < VPT; ++jv) s2 += vsq[jv * TB + tl];
    xsq[tl] = s2;
  }
  // thread t2 accumulated column t2 mod NCP (RT is a multiple of NCP)
  for (int c = tid; c < NCP; c += RT) {
    float s2 = 0.f;
    for (int t2 = c; t2 < RT; t2 += NCP) s2 += wq[t2];
    cn2p[c] = s2;
  }
  cluster.sync();  // partials of every CTA of the cluster are visible

  for (int c = tid; c < NCP; c += RT) {
    float part[kMaxCluster];
#pragma unroll
    for (int r2 = 0; r2 < kMaxCluster; ++r2) part[r2] = r2 < KS ? *cluster.map_shared_rank(cn2p + c, r2) : 0.f;
    float s2 = 0.f;
#pragma unroll
    for (int r2 = 0; r2 < kMaxCluster; ++r2)
      if (r2 < KS) s2 += part[r2];
    cn2f[c] = sqrtf(s2);  // the column norm itself: every token's bound uses it
  }
  __syncthreads();

  // -------- per-token ranking, one warp per token, tokens spread over the cluster
  const int n_eff = DK + q.nch_per + KS;
  const float gam = (n_eff * kU) / (1.0f - n_eff * kU);
  int n_recomputed = 0, n_near = 0;
  auto wcol = [&](int c, int j) {
    const float* W = c < E ? p.W_g + c : p.W_n + (c - E);
    const size_t r0 = static_cast<size_t>(j) * E;
    return make_float4(__ldg(W + r0), __ldg(W + r0 + E), __ldg(W + r0 + 2 * E), __ldg(W + r0 + 3 * E));
  };

  for (int tl = tl_first; tl < TB; tl += tl_step) {
    const long long t = t0 + tl;
    if (t >= p.T) break;
    // the next token's noise, in flight while this token is ranked
    float ep_next[SLOTS];
    load_eps<SLOTS>(p, tl + tl_step < TB ? t + tl_step : p.T, lane, ep_next);
    // the KS partial tiles summed in rank order (KS = 1: this CTA's own tile)
    float g[SLOTS], z[SLOTS];
    float nx2 = 0.f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) { g[s] = 0.f; z[s] = 0.f; }
    if (KS == 1) {
      nx2 = xsq[tl];
      const float* Lr = Lt + tl * G::LT_LD;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        if (e < E) {
          g[s] = Lr[e];
          if (noisy) z[s] = Lr[E + e];
        }
      }
    } else {
#pragma unroll 4
      for (int r2 = 0; r2 < KS; ++r2) {
        nx2 += *cluster.map_shared_rank(xsq + tl, r2);
        const float* Lr = cluster.map_shared_rank(Lt + tl * G::LT_LD, r2);
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
          const int e = lane + 32 * s;
          if (e < E) {
            g[s] += Lr[e];
            if (noisy) z[s] += Lr[E + e];
          }
        }
      }
    }
    float xb[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) xb[s] = 0.f;
    rank_token<TX, SLOTS>(p, t, lane, g, z, ep_cur, sqrtf(nx2), cn2f, gam, wcol, n_recomputed, n_near, xb);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) ep_cur[s] = ep_next[s];
  }

  if (p.stats) flush_stats(p, cnt, lane, n_recomputed, n_near);
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

// ---------------------------------------------------------------- host side
int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

// expert slots per lane: the logit columns bound E (nc = E, or 2E with noise)
template <int CQ>
constexpr int slots_for(bool noisy) {
  return CQ <= 8 ? 1 : (CQ == 16 ? 2 : (CQ == 32 ? (noisy ? 2 : 4) : 4));
}

template <typename TX, int CQ, int TM, int SL>
cudaError_t launch_one_sl(const RouterParams& p, const TiledPlan& q, long long tiles, cudaStream_t st) {
  using G = Tile<TX, CQ, TM>;
  auto kern = router_tiled_kernel<TX, CQ, TM, SL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
  if (e != cudaSuccess) return e;
  if (q.KS > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  // a cluster of KS CTAs along y (also for KS = 1, so the cluster API sees a cluster)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(q.KS), 1);
  cfg.blockDim = dim3(RT, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(G::SMEM);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(q.KS);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return counted(cudaLaunchKernelEx(&cfg, kern, p, q));
}

template <typename TX, int CQ, int TM>
cudaError_t launch_one(const RouterParams& p, const TiledPlan& q, long long tiles, cudaStream_t st) {
  const bool noisy = p.W_n != nullptr;
  if (CQ == 32 && noisy) return launch_one_sl<TX, CQ, TM, slots_for<CQ>(true)>(p, q, tiles, st);
  return launch_one_sl<TX, CQ, TM, slots_for<CQ>(false)>(p, q, tiles, st);
}

// Whether a 16-CTA cluster of the largest-footprint 16-CTA plan (TM = 1) can
// be resident; probed once per device.  Otherwise clusters stay within 8.
constexpr int kMaxDevices = 64;
int g_max_cluster[kMaxDevices];
std::once_flag g_cluster_once[kMaxDevices];

template <typename TX, int CQ>
int probe_cluster16() {
  using G = Tile<TX, CQ, 1>;
  auto kern = router_tiled_kernel<TX, CQ, 1, slots_for<CQ>(false)>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM) != cudaSuccess) {
    cudaGetLastError();
    return 8;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, kMaxCluster, 1);
  cfg.blockDim = dim3(RT, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(G::SMEM);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kMaxCluster;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 8;
  }
  return n > 0 ? kMaxCluster : 8;
}

template <typename TX, int CQ>
cudaError_t launch_cq(const RouterParams& p, TiledPlan& q, int TM, long long tiles, cudaStream_t st) {
  if constexpr (CQ <= 4) {
    return launch_one<TX, CQ, 1>(p, q, tiles, st);
  } else {
    switch (TM) {
      case 8:
        if constexpr (sizeof(TX) == 2) return launch_one<TX, CQ, 8>(p, q, tiles, st);
        return cudaErrorInvalidConfiguration;
      case 4: return launch_one<TX, CQ, 4>(p, q, tiles, st);
      case 2:
        if constexpr (sizeof(TX) == 2) return launch_one<TX, CQ, 2>(p, q, tiles, st);
        return cudaErrorInvalidConfiguration;
      default: return launch_one<TX, CQ, 1>(p, q, tiles, st);
    }
  }
}

template <typename TX>
cudaError_t launch_typed(const RouterParams& p, cudaStream_t st, int sms, int max_cluster) {
  TiledPlan q{};
  q.nc = p.W_n ? 2 * p.E : p.E;
  const int CQ = pow2_at_least((q.nc + 3) / 4);
  q.vec_w = (p.E % 4 == 0 && reinterpret_cast<uintptr_t>(p.W_g) % 16 == 0 &&
             (p.W_n == nullptr || reinterpret_cast<uintptr_t>(p.W_n) % 16 == 0)) ? 1 : 0;
  const int TG = RT / CQ;
  q.nch = (p.d + DK - 1) / DK;
  // narrow tables (CQ <= 4) have the largest token tiles: keep them within portable clusters
  const int ks_max = std::min(CQ <= 4 ? 8 : max_cluster, q.nch);
  // CTAs to aim for: two per SM, or (when the next kernel is meant to run
  // beside this one: the decode-sized layer's expert FFN streams weights
  // while the routing runs) a single cluster's worth, leaving the other SMs free
  const long long target = p.early_trigger ? kMaxCluster : 2LL * sms;

  // the largest register tile (tokens per thread) that still fills the GPU
  // with at most ks_max CTAs per tile; at most 256 tokens per tile
  int TM = 1;
  if (CQ >= 8) {
    const int cands_bf16[3] = {8, 4, 2};
    const int cands_f32[1] = {4};
    const int* cands = sizeof(TX) == 2 ? cands_bf16 : cands_f32;
    const int ncand = sizeof(TX) == 2 ? 3 : 1;
    for (int i = 0; i < ncand; ++i) {
      const int cand = cands[i];
      if (TG * cand > 256) continue;
      const long long tl = (static_cast<long long>(p.T) + TG * cand - 1) / (TG * cand);
      if (tl * ks_max >= target) { TM = cand; break; }
    }
  }
  const int TB = TG * TM;
  const long long tiles = (static_cast<long long>(p.T) + TB - 1) / TB;
  const int ks = static_cast<int>(std::min<long long>(ks_max, std::max<long long>(1, (target + tiles - 1) / tiles)));
  q.nch_per = (q.nch + ks - 1) / ks;
  q.KS = (q.nch + q.nch_per - 1) / q.nch_per;  // no CTA without a slice
  if (q.KS > kMaxCluster || tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  switch (CQ) {
    case 1: return launch_cq<TX, 1>(p, q, TM, tiles, st);
    case 2: return launch_cq<TX, 2>(p, q, TM, tiles, st);
    case 4: return launch_cq<TX, 4>(p, q, TM, tiles, st);
    case 8: return launch_cq<TX, 8>(p, q, TM, tiles, st);
    case 16: return launch_cq<TX, 16>(p, q, TM, tiles, st);
    case 32: return launch_cq<TX, 32>(p, q, TM, tiles, st);
    case 64: return launch_cq<TX, 64>(p, q, TM, tiles, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace

cudaError_t launch_router_tiled(const RouterParams& p, int dtype, cudaStream_t st, int sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_cluster_once[dev], [dev] {
    // the 16-CTA plans use TM = 1; the widest of them (64 column quads) has the largest footprint
    g_max_cluster[dev] = std::min(probe_cluster16<__nv_bfloat16, 64>(), probe_cluster16<float, 64>());
  });
  return dtype == MOE_BF16 ? launch_typed<__nv_bfloat16>(p, st, sms, g_max_cluster[dev])
                           : launch_typed<float>(p, st, sms, g_max_cluster[dev]);
}

}  // namespace moe
