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
#include "router_tc.cuh"

namespace moe {
namespace {

using namespace router_detail;


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
__global__ void __launch_bounds__(256, 2) router_tc_rank_kernel(RouterParams p, const float* approx, const float* wt,
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
  // d <= 1024: the next token's row is held in registers (8 loads a lane) so
  // its norm never waits on memory; longer rows are read in the step itself
  constexpr int XR = 8;
  const bool xreg = d <= XR * 128;
  typename Vec4<__nv_bfloat16>::raw xr_n[XR];
  auto load_row = [&](long long tt) {
#pragma unroll
    for (int i = 0; i < XR; ++i) {
      const int j = i * 128 + lane * 4;
      xr_n[i] = (xreg && tt < p.T && j < d) ? Vec4<__nv_bfloat16>::load(x + tt * d + j) : Vec4<__nv_bfloat16>::zero();
    }
  };
  load_row(t);
  for (; t < p.T; t += nwarps) {
    prefetch_row(t + 2 * nwarps);
    float ga[SLOTS], za[SLOTS], ep[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) { ga[s] = ga_n[s]; za[s] = za_n[s]; ep[s] = ep_n[s]; }
    load_tok(t + nwarps, ga_n, za_n, ep_n);
    float nx = -1.f;
    if (xreg) {
      float sq = 0.f;
#pragma unroll
      for (int i = 0; i < XR; ++i) {
        float xv[4];
        Vec4<__nv_bfloat16>::unpack(xr_n[i], xv);
        sq = fmaf(xv[0], xv[0], fmaf(xv[1], xv[1], fmaf(xv[2], xv[2], fmaf(xv[3], xv[3], sq))));
      }
      nx = sqrtf(warp_sum(sq));
      load_row(t + nwarps);
    }
    rank_token_filtered<SLOTS>(p, t, lane, ga, za, ep, wt, s_cn, gam, n_recomputed, n_near, nx);
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

RouterTcScratch router_tc_scratch(void* scratch, long long T, int d, int E) {
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  char* base = static_cast<char*>(scratch);
  RouterTcScratch r{};
  r.approx = reinterpret_cast<float*>(base);
  base += up(sizeof(float) * static_cast<size_t>(T) * 2 * E);
  r.wsplit = base;
  base += up(2 * static_cast<size_t>(2 * E) * 2 * d);
  r.wt = reinterpret_cast<float*>(base);
  base += up(sizeof(float) * static_cast<size_t>(2 * E) * d);
  r.cn = reinterpret_cast<float*>(base);
  return r;
}

cudaError_t launch_router_tc(const RouterParams& p, void* scratch, cudaStream_t st) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  const RouterTcScratch sc = router_tc_scratch(scratch, p.T, p.d, p.E);
  float* approx = sc.approx;
  __nv_bfloat16* wsplit = static_cast<__nv_bfloat16*>(sc.wsplit);
  float* wt = sc.wt;
  float* cn = sc.cn;
  cudaError_t e = launch_pdl(router_tc_prep_kernel, dim3(static_cast<unsigned>(nc)), dim3(256), 0, st, 1, p.W_g,
                             p.W_n, p.d, p.E, wsplit, wt, cn);
  if (e != cudaSuccess) return e;
  if ((e = launch_dense_wrapped_gemm(p.x, p.T, p.d, wsplit, nc, 2 * p.d, approx, p.err, st)) != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // persistent: two 8-warp blocks per SM (up to 128 registers a thread: each
  // warp holds its next token's row), warps stride the tokens
  const long long want = (static_cast<long long>(p.T) + 7) / 8;
  const unsigned grid = static_cast<unsigned>(want < 2LL * sms ? want : 2LL * sms);
  if (p.E <= 32) return launch_pdl(router_tc_rank_kernel<1>, dim3(grid), dim3(256), 0, st, 1, p, approx, wt, cn);
  if (p.E <= 64) return launch_pdl(router_tc_rank_kernel<2>, dim3(grid), dim3(256), 0, st, 1, p, approx, wt, cn);
  return launch_pdl(router_tc_rank_kernel<4>, dim3(grid), dim3(256), 0, st, 1, p, approx, wt, cn);
}

// The filter alone (for tests): the weight split and the filter GEMM, the
// approximate logits g~ [T, nc] written to `approx`.
cudaError_t launch_router_tc_filter(const RouterParams& p, void* scratch, float* approx, cudaStream_t st) {
  const int nc = p.W_n ? 2 * p.E : p.E;
  const RouterTcScratch sc = router_tc_scratch(scratch, p.T, p.d, p.E);
  __nv_bfloat16* wsplit = static_cast<__nv_bfloat16*>(sc.wsplit);
  float* wt = sc.wt;
  float* cn = sc.cn;
  cudaError_t e = launch_pdl(router_tc_prep_kernel, dim3(static_cast<unsigned>(nc)), dim3(256), 0, st, 1, p.W_g,
                             p.W_n, p.d, p.E, wsplit, wt, cn);
  if (e != cudaSuccess) return e;
  return launch_dense_wrapped_gemm(p.x, p.T, p.d, wsplit, nc, 2 * p.d, approx, p.err, st);
}

}  // namespace moe
