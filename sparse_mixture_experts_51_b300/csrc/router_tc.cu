// Router for wide logit tables on bf16 layers: a tensor-core filter, then
// exact ranking of the few experts it leaves.
//
// Logits H = x W_g + b_g (+ eps * softplus(x W_noise)) and their top-k
// ("LLM part 09: Sparse Mixture-of-Experts (MoE)", s2), with the selection
// exact as in router.cu.  The contraction with nc = E or 2E columns is
// dense: for long token batches the CUDA-core kernels spend most of the
// layer's time on it.  Here:
//   1. the fp32 router weights are split into two bf16 parts, w = hi + lo
//      + r with |r| <= 2^-16 |w| (router_tc_prep_kernel, once per call), and
//      the tensor cores compute g~ = x (hi + lo) in fp32 for every column
//      (one dense GEMM with K = 2d whose A operand reads x twice);
//   2. a warp per token bounds every approximate logit with a wide margin
//      delta = 2^-10 ||x|| ||w_col|| -- it covers the dropped part r and
//      the tensor core's fp32 accumulation of the exact bf16 products (its
//      rounding is not specified; any accumulation that loses fewer than
//      ~10 of fp32's 24 bits per step stays inside the margin); L = the
//      kr-th largest lower end; an expert whose upper end is below L cannot
//      be in the top kr, every other expert is a candidate;
//   3. the candidates' logits are recomputed on CUDA cores in fp32 (lanes
//      stride d, then a butterfly: summation depth d/32 + 5) with the
//      rigorous bound of router.cu, the other experts keep g~ with bound
//      delta, and the token is ranked by rank_token (fp64 re-evaluation of
//      any rank the bounds leave open).
// The top-k, their order, the backup rank and the gates (softmax over the
// selected exact logits) are those of the CUDA-core kernels.  Used only when
// no exact full logit table is asked for (no logits output, no raw-p gates,
// no expert-choice radii).
#include "router_rank.cuh"

namespace moe {
namespace {

using namespace router_detail;

constexpr float kFilterMargin = 1.0f / 1024.0f;  // delta = margin * ||x|| * ||w_col||

// Column c of [W_g | W_noise]: bf16 hi / lo parts as row c of wsplit [nc][2d]
// (hi in k < d, lo in k >= d), the fp32 column as row c of wt [nc][d], and
// its norm.  One block per column.
__global__ void __launch_bounds__(256) router_tc_prep_kernel(const float* W_g, const float* W_n, int d, int E,
                                                             __nv_bfloat16* wsplit, float* wt, float* cn) {
  __shared__ float s_red[8];
  const int c = blockIdx.x;
  pdl_wait();
  float ss = 0.f;
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const float w = c < E ? __ldg(W_g + static_cast<long long>(j) * E + c)
                          : __ldg(W_n + static_cast<long long>(j) * E + (c - E));
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
    wsplit[static_cast<long long>(c) * 2 * d + j] = hi;
    wsplit[static_cast<long long>(c) * 2 * d + d + j] = lo;
    wt[static_cast<long long>(c) * d + j] = w;
    ss = fmaf(w, w, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += s_red[w];
    cn[c] = sqrtf(t);
  }
  pdl_trigger();
}

template <int SLOTS>
__global__ void __launch_bounds__(256, 3) router_tc_rank_kernel(RouterParams p, const float* approx, const float* wt,
                                                             const float* cn_g) {
  __shared__ float s_cn[2 * kMaxExperts];
  const int lane = threadIdx.x & 31;
  const int E = p.E, d = p.d, k = p.k;
  const bool noisy = p.W_n != nullptr;
  const int nc = noisy ? 2 * E : E;
  const int kr = (p.backup != nullptr && k < E) ? k + 1 : k;
  pdl_wait();  // approximate logits from the GEMM, weights from the prep kernel
  for (int c = threadIdx.x; c < nc; c += blockDim.x) s_cn[c] = cn_g[c];
  __syncthreads();
  // the candidates' fp32 dot products: d/32 sequential terms per lane, then 5 butterfly levels
  const int n_eff = (d + 31) / 32 + 5;
  const float gam = (n_eff * kU) / (1.0f - n_eff * kU);
  int n_recomputed = 0, n_near = 0;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x);
  auto wcol = [&](int c, int j) { return __ldg(reinterpret_cast<const float4*>(wt + static_cast<long long>(c) * d + j)); };

  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  // the approximate logits and the noise of a token, requested one token ahead
  auto load_tok = [&](long long t, float (&ga)[SLOTS], float (&za)[SLOTS], float (&ep)[SLOTS]) {
    load_eps<SLOTS>(p, t, lane, ep);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      const bool ok = t < p.T && e < E;
      ga[s] = ok ? __ldg(approx + t * nc + e) : 0.f;
      za[s] = (ok && noisy) ? __ldg(approx + t * nc + E + e) : 0.f;
    }
  };
  long long t = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  float ga_n[SLOTS], za_n[SLOTS], ep_n[SLOTS];
  load_tok(t, ga_n, za_n, ep_n);
  // the token row two tokens ahead is pulled into L2 (its norm and the
  // candidates' dot products read it; most of the load latency is DRAM)
  auto prefetch_row = [&](long long tt) {
    if (tt < p.T)
      for (int j = lane * 64; j < d; j += 32 * 64)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(x + tt * d + j));
  };
  prefetch_row(t);
  prefetch_row(t + nwarps);
  for (; t < p.T; t += nwarps) {
    prefetch_row(t + 2 * nwarps);
    const __nv_bfloat16* xrow = x + t * d;
    float ga[SLOTS], za[SLOTS], ep[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) { ga[s] = ga_n[s]; za[s] = za_n[s]; ep[s] = ep_n[s]; }
    load_tok(t + nwarps, ga_n, za_n, ep_n);
    // ---- token norm
    float sq = 0.f;
    for (int j = lane * 4; j < d; j += 128) {
      float xv[4];
      Vec4<__nv_bfloat16>::unpack(Vec4<__nv_bfloat16>::load(xrow + j), xv);
      sq = fmaf(xv[0], xv[0], fmaf(xv[1], xv[1], fmaf(xv[2], xv[2], fmaf(xv[3], xv[3], sq))));
    }
    const float nx = sqrtf(warp_sum(sq));
    // ---- approximate logits and their margins
    float g[SLOTS], z[SLOTS], xb[SLOTS], lo[SLOTS], up[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      g[s] = z[s] = xb[s] = 0.f;
      lo[s] = up[s] = -INFINITY;
      if (e < E) {
        g[s] = ga[s];
        float h = g[s] + (p.b_g ? __ldg(p.b_g + e) : 0.f);
        float dl = kFilterMargin * nx * s_cn[e];
        if (noisy) {
          z[s] = za[s];
          h += ep[s] * softplus_f32(z[s]);
          dl += fabsf(ep[s]) * kFilterMargin * nx * s_cn[E + e];  // softplus is 1-Lipschitz
        }
        dl = dl * 1.25f + 4.f * kU * fabsf(h) + 1e-30f;
        xb[s] = dl;
        if (h != h) {  // not a number: let the exact path decide
          lo[s] = -INFINITY;
          up[s] = INFINITY;
        } else {
          lo[s] = h - dl;
          up[s] = h + dl;
        }
      }
    }
    // ---- L = the kr-th largest lower end; candidates reach L with their upper end
    bool taken[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) taken[s] = false;
    float L = -INFINITY;
    for (int r = 0; r < kr; ++r) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        if (e < E && !taken[s] && better(lo[s], e, bv, be)) { bv = lo[s]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int e2 = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(v2, e2, bv, be)) { bv = v2; be = e2; }
      }
#pragma unroll
      for (int s = 0; s < SLOTS; ++s)
        if ((be & 31) == lane && (be >> 5) == s) taken[s] = true;
      L = bv;
    }
    // ---- exact fp32 logits of the candidates, four at a time (warp-uniform)
    unsigned cm[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) cm[s] = __ballot_sync(0xffffffffu, lane + 32 * s < E && !(up[s] < L));
    while (true) {
      int ce[4];
      int n = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ce[q] = 0;
        bool got = false;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
          if (!got && cm[s] != 0u) {
            ce[q] = (__ffs(cm[s]) - 1) + 32 * s;
            cm[s] &= cm[s] - 1u;
            got = true;
          }
        }
        n += got ? 1 : 0;
      }
      if (n == 0) break;
      float ag[4] = {0.f, 0.f, 0.f, 0.f}, az[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = lane * 4; j < d; j += 128) {
        float xv[4];
        Vec4<__nv_bfloat16>::unpack(Vec4<__nv_bfloat16>::load(xrow + j), xv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < n) {
            const float4 w = wcol(ce[q], j);
            ag[q] = fmaf(xv[0], w.x, ag[q]);
            ag[q] = fmaf(xv[1], w.y, ag[q]);
            ag[q] = fmaf(xv[2], w.z, ag[q]);
            ag[q] = fmaf(xv[3], w.w, ag[q]);
            if (noisy) {
              const float4 u = wcol(E + ce[q], j);
              az[q] = fmaf(xv[0], u.x, az[q]);
              az[q] = fmaf(xv[1], u.y, az[q]);
              az[q] = fmaf(xv[2], u.z, az[q]);
              az[q] = fmaf(xv[3], u.w, az[q]);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < n) {  // warp-uniform
          ag[q] = warp_sum(ag[q]);
          if (noisy) az[q] = warp_sum(az[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < n) {
#pragma unroll
          for (int s = 0; s < SLOTS; ++s) {
            if (lane == (ce[q] & 31) && s == (ce[q] >> 5)) {
              g[s] = ag[q];
              z[s] = az[q];
              xb[s] = 0.f;  // an exact fp32 contraction: rank_token's own bound covers it
            }
          }
        }
      }
    }
    rank_token<__nv_bfloat16, SLOTS>(p, t, lane, g, z, ep, nx, s_cn, gam, wcol, n_recomputed, n_near, xb);
  }
  pdl_trigger();
  if (p.stats != nullptr) {
    __shared__ int cnt[2];
    if (threadIdx.x < 2) cnt[threadIdx.x] = 0;
    __syncthreads();
    flush_stats(p, cnt, lane, n_recomputed, n_near);
  }
}

}  // namespace

bool router_tc_applies(const RouterParams& p, int dtype) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  // long batches only: the filter GEMM has one tile column, so it needs T / 256
  // row tiles to spread over the SMs (measured on B300: the Switch-style
  // layer, T = 32768, gains 90 us a step; a 4096-token batch loses 70 us)
  return dtype == MOE_BF16 && p.idx != nullptr && p.logits == nullptr && p.radius == nullptr && p.lse == nullptr &&
         !p.gate_raw && nc % 32 == 0 && nc <= 256 && p.d % 64 == 0 && p.T >= 16384;
}

size_t router_tc_scratch_bytes(long long T, int d, int E) {
  const size_t nc = 2 * static_cast<size_t>(E);  // room for the noise columns
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  return up(sizeof(float) * static_cast<size_t>(T) * nc) + up(2 * nc * 2 * static_cast<size_t>(d)) +
         up(sizeof(float) * nc * d) + up(sizeof(float) * nc);
}

cudaError_t launch_router_tc(const RouterParams& p, void* scratch, cudaStream_t st) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  char* base = static_cast<char*>(scratch);
  float* approx = reinterpret_cast<float*>(base);
  base += up(sizeof(float) * static_cast<size_t>(p.T) * 2 * p.E);
  __nv_bfloat16* wsplit = reinterpret_cast<__nv_bfloat16*>(base);
  base += up(2 * static_cast<size_t>(2 * p.E) * 2 * p.d);
  float* wt = reinterpret_cast<float*>(base);
  base += up(sizeof(float) * static_cast<size_t>(2 * p.E) * p.d);
  float* cn = reinterpret_cast<float*>(base);
  cudaError_t e = launch_pdl(router_tc_prep_kernel, dim3(static_cast<unsigned>(nc)), dim3(256), 0, st, 1, p.W_g,
                             p.W_n, p.d, p.E, wsplit, wt, cn);
  if (e != cudaSuccess) return e;
  if ((e = launch_dense_wrapped_gemm(p.x, p.T, p.d, wsplit, nc, 2 * p.d, approx, p.err, st)) != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // persistent: three 8-warp blocks per SM (80 registers a thread), warps stride the tokens
  const long long want = (static_cast<long long>(p.T) + 7) / 8;
  const unsigned grid = static_cast<unsigned>(want < 3LL * sms ? want : 3LL * sms);
  if (p.E <= 32) return launch_pdl(router_tc_rank_kernel<1>, dim3(grid), dim3(256), 0, st, 1, p, approx, wt, cn);
  if (p.E <= 64) return launch_pdl(router_tc_rank_kernel<2>, dim3(grid), dim3(256), 0, st, 1, p, approx, wt, cn);
  return launch_pdl(router_tc_rank_kernel<4>, dim3(grid), dim3(256), 0, st, 1, p, approx, wt, cn);
}

// The filter alone (for tests): the weight split and the filter GEMM, the
// approximate logits g~ [T, nc] written to `approx`.
cudaError_t launch_router_tc_filter(const RouterParams& p, void* scratch, float* approx, cudaStream_t st) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  char* base = static_cast<char*>(scratch);
  base += up(sizeof(float) * static_cast<size_t>(p.T) * 2 * p.E);
  __nv_bfloat16* wsplit = reinterpret_cast<__nv_bfloat16*>(base);
  base += up(2 * static_cast<size_t>(2 * p.E) * 2 * p.d);
  float* wt = reinterpret_cast<float*>(base);
  base += up(sizeof(float) * static_cast<size_t>(2 * p.E) * p.d);
  float* cn = reinterpret_cast<float*>(base);
  cudaError_t e = launch_pdl(router_tc_prep_kernel, dim3(static_cast<unsigned>(nc)), dim3(256), 0, st, 1, p.W_g,
                             p.W_n, p.d, p.E, wsplit, wt, cn);
  if (e != cudaSuccess) return e;
  return launch_dense_wrapped_gemm(p.x, p.T, p.d, wsplit, nc, 2 * p.d, approx, p.err, st);
}

}  // namespace moe
