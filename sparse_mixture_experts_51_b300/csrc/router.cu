// Router: logits, exact top-k selection and renormalised gates.
//
// Logits H = x W_g + b_g (+ eps * softplus(x W_noise)) follow the noisy top-k
// gating of "LLM part 09: Sparse Mixture-of-Experts (MoE)", s2; the gates are
// the softmax over the k selected logits (same section, and the renormalised
// top-k of "Mixture-of-experts Models", Level 2).
//
// Design.  The logits are a skinny fp32 contraction [T,d] x [d,E(+E)]: each
// 256-thread block owns a tile of TB tokens and all columns, stages 32-wide
// slices of x (transposed) and of the router weights in shared memory, and
// every thread keeps a TM x 4 register tile.  The dot products are summed in
// 32-term chunks, so the rounding error of a logit is at most
// gamma(32 + ceil(d/32)) * ||x_t|| * ||W_col|| (Cauchy-Schwarz), which the
// kernel evaluates per token and expert together with the error of the bias
// add and of the softplus noise term.  A warp per token then ranks the
// experts.  When the bound separates the k selected logits from each other
// and from every other expert, the fp32 order is the exact order.  Otherwise
// the warp re-evaluates every expert that could still be in the top k in
// fp64 and ranks those values (ties -> lower expert index).  Either way the
// selected experts and their order are those of the exactly computed logits.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int RT = 256;  // threads per block
constexpr int DK = 32;   // d-slice staged per step
constexpr float kU = 5.9604644775390625e-8f;  // unit roundoff of fp32, 2^-24

template <typename TX>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[8]) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};

__device__ __forceinline__ float softplus_f32(float z) {
  return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z)));
}
__device__ __forceinline__ double softplus_f64(double z) {
  return fmax(z, 0.0) + log1p(exp(-fabs(z)));
}

// (value, expert) ordering: larger value first, then lower expert index.
__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}
__device__ __forceinline__ bool better_d(double v1, int e1, double v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

template <typename TX>
__device__ double dot_f64(const TX* xrow, const float* W, int d, int E, int col, int lane) {
  double acc = 0.0;
  for (int j = lane; j < d; j += 32)
    acc = fma(static_cast<double>(to_f32(xrow[j])), static_cast<double>(W[static_cast<size_t>(j) * E + col]), acc);
  return warp_sum_d(acc);
}

template <typename TX, int TM>
__global__ void __launch_bounds__(RT) router_kernel(RouterParams p, int ncq_pad) {
  extern __shared__ __align__(16) float smem[];
  constexpr int VEC = Vec16<TX>::N;    // elements per 16-byte vector
  constexpr int VPT = DK / VEC;        // vectors per token per slice
  constexpr int SLOTS = kMaxExperts / 32;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nc_pad = ncq_pad * 4;
  const int TG = RT / ncq_pad;
  const int TB = TG * TM;
  const int cq = tid % ncq_pad, tg = tid / ncq_pad;
  const int E = p.E, d = p.d, k = p.k;
  const bool noisy = p.W_n != nullptr;
  const int nc = noisy ? 2 * E : E;
  const long long t0 = static_cast<long long>(blockIdx.x) * TB;
  const TX* x = static_cast<const TX*>(p.x);

  const int xs_ld = TB + 4;
  const int stage_floats = DK * xs_ld + DK * nc_pad;
  const int lt_ld = nc_pad + 1;
  const int regionA = max(stage_floats, TB * lt_ld);
  float* xs = smem;                   // [DK][xs_ld]   x slice, transposed
  float* wsm = smem + DK * xs_ld;     // [DK][nc_pad]  router weight slice
  float* Lt = smem;                   // [TB][lt_ld]   fp32 logits (after the loop)
  float* xsq = smem + regionA;        // [TB*VPT]      partial sums of x^2
  float* cn2 = xsq + TB * VPT;        // [nc_pad]      column sums of W^2
  int* cnt = reinterpret_cast<int*>(cn2 + nc_pad);  // [2] block counters

  if (tid < 2) cnt[tid] = 0;

  float acc[TM][4], cacc[TM][4], colsq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int m = 0; m < TM; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = 0.f;
  constexpr int NVMAX = 8;  // TB*VPT/RT <= VPT <= 8 because TM <= ncq_pad
  float sq[NVMAX];
#pragma unroll
  for (int s = 0; s < NVMAX; ++s) sq[s] = 0.f;
  const int nvec = TB * VPT;

  const int nchunks = (d + DK - 1) / DK;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int j0 = ch * DK;
    // ---- stage x slice (16-byte vectors; d % VEC == 0 is checked on the host)
#pragma unroll
    for (int s = 0; s < NVMAX; ++s) {
      const int v = tid + s * RT;
      if (v < nvec) {
        const int tl = v / VPT, jv = v % VPT;
        const long long t = t0 + tl;
        const int j = j0 + jv * VEC;
        float vals[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) vals[q] = 0.f;
        if (t < p.T && j < d) Vec16<TX>::load(x + t * d + j, vals);
#pragma unroll
        for (int q = 0; q < VEC; ++q) {
          xs[(jv * VEC + q) * xs_ld + tl] = vals[q];
          sq[s] = fmaf(vals[q], vals[q], sq[s]);
        }
      }
    }
    // ---- stage router weight slice: columns [0,E) from W_g, [E,2E) from W_noise
    for (int i = tid; i < DK * nc_pad; i += RT) {
      const int jj = i / nc_pad, c = i % nc_pad;
      const int j = j0 + jj;
      float v = 0.f;
      if (j < d && c < nc) v = c < E ? p.W_g[static_cast<size_t>(j) * E + c] : p.W_n[static_cast<size_t>(j) * E + (c - E)];
      wsm[jj * nc_pad + c] = v;
    }
    __syncthreads();
    // ---- register-tiled partial dot products for this slice
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) cacc[m][c] = 0.f;
#pragma unroll 8
    for (int jj = 0; jj < DK; ++jj) {
      const float4 wv = *reinterpret_cast<const float4*>(&wsm[jj * nc_pad + 4 * cq]);
      float xv[TM];
      if constexpr (TM % 4 == 0) {
#pragma unroll
        for (int m = 0; m < TM; m += 4) {
          const float4 q = *reinterpret_cast<const float4*>(&xs[jj * xs_ld + tg * TM + m]);
          xv[m] = q.x; xv[m + 1] = q.y; xv[m + 2] = q.z; xv[m + 3] = q.w;
        }
      } else {
#pragma unroll
        for (int m = 0; m < TM; ++m) xv[m] = xs[jj * xs_ld + tg * TM + m];
      }
#pragma unroll
      for (int m = 0; m < TM; ++m) {
        cacc[m][0] = fmaf(xv[m], wv.x, cacc[m][0]);
        cacc[m][1] = fmaf(xv[m], wv.y, cacc[m][1]);
        cacc[m][2] = fmaf(xv[m], wv.z, cacc[m][2]);
        cacc[m][3] = fmaf(xv[m], wv.w, cacc[m][3]);
      }
      if (tg == 0) {
        colsq[0] = fmaf(wv.x, wv.x, colsq[0]);
        colsq[1] = fmaf(wv.y, wv.y, colsq[1]);
        colsq[2] = fmaf(wv.z, wv.z, colsq[2]);
        colsq[3] = fmaf(wv.w, wv.w, colsq[3]);
      }
    }
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][c] += cacc[m][c];
    __syncthreads();
  }

  // ---- park logits, column norms and token norm partials in shared memory
#pragma unroll
  for (int m = 0; m < TM; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) Lt[(tg * TM + m) * lt_ld + 4 * cq + c] = acc[m][c];
  if (tg == 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c) cn2[4 * cq + c] = colsq[c];
  }
#pragma unroll
  for (int s = 0; s < NVMAX; ++s) {
    const int v = tid + s * RT;
    if (v < nvec) xsq[v] = sq[s];
  }
  __syncthreads();

  // ---- per-token ranking, one warp per token
  const int n_eff = DK + nchunks;
  const float gam = (n_eff * kU) / (1.0f - n_eff * kU);
  int n_recomputed = 0, n_near = 0;

  for (int tl = warp; tl < TB; tl += RT / 32) {
    const long long t = t0 + tl;
    if (t >= p.T) break;
    float nx2 = 0.f;
    for (int jv = 0; jv < VPT; ++jv) nx2 += xsq[tl * VPT + jv];
    const float nx = sqrtf(nx2);

    float H[SLOTS], B[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      H[s] = -INFINITY;
      B[s] = 0.f;
      if (e < E) {
        const float g = Lt[tl * lt_ld + e];
        const float b = p.b_g ? p.b_g[e] : 0.f;
        const float gb = g + b;
        float h = gb, bound;
        const float cg = sqrtf(cn2[e]);
        if (noisy) {
          const float z = Lt[tl * lt_ld + E + e];
          const float ep = p.eps[t * E + e];
          const float sp = softplus_f32(z);
          const float ns = ep * sp;
          h = gb + ns;
          const float cn = sqrtf(cn2[E + e]);
          bound = gam * nx * (cg + fabsf(ep) * cn) + fabsf(ep) * (4e-7f + 3e-7f * sp) +
                  4.f * kU * (fabsf(g) + fabsf(b) + fabsf(ns) + fabsf(h));
        } else {
          bound = gam * nx * cg + 4.f * kU * (fabsf(g) + fabsf(b) + fabsf(h));
        }
        if (p.logits) p.logits[t * E + e] = h;
        if (h != h) h = -INFINITY;  // NaN ranks last
        H[s] = h;
        B[s] = bound * 1.25f + 1e-30f;
      }
    }

    // top-k by fp32 value (ties -> lower index), carrying the bounds
    float oh[kMaxTopK], ob[kMaxTopK];
    int oe[kMaxTopK];
    unsigned taken = 0u;  // bit s: slot s of this lane selected
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
      oh[r] = -INFINITY; ob[r] = 0.f; oe[r] = 0x7fffffff;
      if (r < k) {
        float bv = -INFINITY, bb = 0.f;
        int be = 0x7fffffff;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
          const int e = lane + 32 * s;
          if (e < E && !(taken >> s & 1u) && better(H[s], e, bv, be)) { bv = H[s]; bb = B[s]; be = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
          const float b2 = __shfl_xor_sync(0xffffffffu, bb, o);
          const int e2 = __shfl_xor_sync(0xffffffffu, be, o);
          if (better(v2, e2, bv, be)) { bv = v2; bb = b2; be = e2; }
        }
        oh[r] = bv; ob[r] = bb; oe[r] = be;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
      }
    }
    // best value and best upper bound among the experts left out
    float restH = -INFINITY, restU = -INFINITY;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      if (e < E && !(taken >> s & 1u)) {
        restH = fmaxf(restH, H[s]);
        restU = fmaxf(restU, H[s] + B[s]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      restH = fmaxf(restH, __shfl_xor_sync(0xffffffffu, restH, o));
      restU = fmaxf(restU, __shfl_xor_sync(0xffffffffu, restU, o));
    }
    bool cert = true;
    float lowest = INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
      if (r < k) {
        const float lo = oh[r] - ob[r];
        lowest = fminf(lowest, lo);
        if (r + 1 < k && !(lo > oh[r + 1] + ob[r + 1])) cert = false;
        if (!(lo > -INFINITY) || !(ob[r] < INFINITY)) cert = false;
      }
    }
    if (k < E) {
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r) {
        if (r == k - 1) {
          if (!(oh[r] - ob[r] > restU)) cert = false;
          if (oh[r] - restH < 1e-4f) ++n_near;
        }
      }
    }

    if (!cert) {
      // re-evaluate every expert that may still rank in the top k, in fp64
      ++n_recomputed;
      const TX* xrow = x + t * d;
      double h64[SLOTS];
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        const bool cand = e < E && ((taken >> s & 1u) || !(H[s] + B[s] < lowest));
        h64[s] = -INFINITY;
        unsigned m = __ballot_sync(0xffffffffu, cand);
        while (m) {
          const int l = __ffs(m) - 1;
          m &= m - 1;
          const int ce = l + 32 * s;
          double v = dot_f64(xrow, p.W_g, d, E, ce, lane);
          if (p.b_g) v += static_cast<double>(p.b_g[ce]);
          if (noisy) {
            const double z = dot_f64(xrow, p.W_n, d, E, ce, lane);
            v += static_cast<double>(p.eps[t * E + ce]) * softplus_f64(z);
          }
          if (v != v) v = -INFINITY;
          if (lane == l) h64[s] = v;
        }
      }
      unsigned taken64 = 0u;
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r) {
        if (r < k) {
          double bv = -INFINITY;
          int be = 0x7fffffff;
#pragma unroll
          for (int s = 0; s < SLOTS; ++s) {
            const int e = lane + 32 * s;
            if (e < E && !(taken64 >> s & 1u) && better_d(h64[s], e, bv, be)) { bv = h64[s]; be = e; }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const double v2 = __shfl_xor_sync(0xffffffffu, bv, o);
            const int e2 = __shfl_xor_sync(0xffffffffu, be, o);
            if (better_d(v2, e2, bv, be)) { bv = v2; be = e2; }
          }
          oh[r] = static_cast<float>(bv);
          oe[r] = be;
          if ((be & 31) == lane) taken64 |= 1u << (be >> 5);
        }
      }
    }

    // gates: softmax over the selected logits, shifted by the largest
    float den = 0.f, mine_w = 0.f;
    int mine_e = 0;
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
      if (r < k) {
        const float ex = expf(oh[r] - oh[0]);
        den += ex;
        if (r == lane) { mine_w = ex; mine_e = oe[r]; }
      }
    }
    if (lane < k) {
      p.idx[t * k + lane] = mine_e;
      p.w[t * k + lane] = mine_w / den;
    }
  }

  if (p.stats) {
    if (lane == 0 && (n_recomputed | n_near)) {
      atomicAdd(&cnt[0], n_recomputed);
      atomicAdd(&cnt[1], n_near);
    }
    __syncthreads();
    if (tid == 0) {
      if (cnt[0]) atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats[0]), static_cast<unsigned long long>(cnt[0]));
      if (cnt[1]) atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats[1]), static_cast<unsigned long long>(cnt[1]));
    }
  }
}

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <typename TX, int TM>
cudaError_t launch_tm(const RouterParams& p, int ncq_pad, cudaStream_t st) {
  constexpr int VEC = Vec16<TX>::N;
  constexpr int VPT = DK / VEC;
  const int TB = (RT / ncq_pad) * TM;
  const int nc_pad = ncq_pad * 4;
  const int xs_ld = TB + 4;
  const int stage = DK * xs_ld + DK * nc_pad;
  const int regionA = std::max(stage, TB * (nc_pad + 1));
  const size_t smem = sizeof(float) * (regionA + TB * VPT + nc_pad) + 2 * sizeof(int);
  auto kern = router_kernel<TX, TM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long blocks = (static_cast<long long>(p.T) + TB - 1) / TB;
  kern<<<static_cast<unsigned>(blocks), RT, smem, st>>>(p, ncq_pad);
  return cudaGetLastError();
}

template <typename TX>
cudaError_t launch_typed(const RouterParams& p, cudaStream_t st, int num_sms) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  const int ncq_pad = pow2_at_least((nc + 3) / 4);
  const int TG = RT / ncq_pad;
  // largest register tile that still leaves about two blocks per SM
  int TM = 1;
  const long long target = 2LL * num_sms;
  for (int cand : {8, 4, 2}) {
    if (cand <= ncq_pad && (static_cast<long long>(p.T) + TG * cand - 1) / (TG * cand) >= target) { TM = cand; break; }
  }
  switch (TM) {
    case 8: return launch_tm<TX, 8>(p, ncq_pad, st);
    case 4: return launch_tm<TX, 4>(p, ncq_pad, st);
    case 2: return launch_tm<TX, 2>(p, ncq_pad, st);
    default: return launch_tm<TX, 1>(p, ncq_pad, st);
  }
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, int dtype, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  return dtype == MOE_BF16 ? launch_typed<__nv_bfloat16>(p, st, sms) : launch_typed<float>(p, st, sms);
}

}  // namespace moe
