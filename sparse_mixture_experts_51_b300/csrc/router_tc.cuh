// The per-token step of the tensor-core router filter (router_tc.cu): one
// warp takes token t's
// approximate logits g~ (from the filter GEMM of x against the bf16 hi + lo
// split of the router weights), bounds each one by the filter margin, finds
// the experts that may still hold one of the top ranks, recomputes those
// exactly in fp32 and ranks the token with rank_token (exact selection, fp64
// re-evaluation of any rank the bounds leave open).  Router logits
// H = x W_g + b_g (+ eps * softplus(x W_noise)) and top-k gates as in
// "LLM part 09: Sparse Mixture-of-Experts (MoE)", s2.
#pragma once

#include "router_rank.cuh"

namespace moe {
namespace router_detail {

// delta = margin * ||x|| * ||w_col||: the trust radius of an approximate logit
constexpr float kFilterMargin = 1.0f / 1024.0f;

// Ranks token t.  approx [T, nc] (nc = E, or 2E with the noise columns), wt
// [nc][d] the fp32 router-weight columns, cn [nc] their norms, gam the fp32
// error factor of the exact recomputation (summation depth d/32 + 5).
// ga/za/ep: this token's approximate gate and noise logits and its noise
// draws (lane e + 32 s holds expert e), loaded by the caller.
// nx_in: the token's norm when the caller has it (< 0: computed here).
template <int SLOTS>
__device__ __forceinline__ void rank_token_filtered(const RouterParams& p, long long t, int lane,
                                                    const float (&ga)[SLOTS], const float (&za)[SLOTS],
                                                    const float (&ep)[SLOTS], const float* wt, const float* cn,
                                                    float gam, int& n_recomputed, int& n_near, float nx_in = -1.f) {
  const int E = p.E, d = p.d, k = p.k;
  const bool noisy = p.W_n != nullptr;
  const int kr = (p.backup != nullptr && k < E) ? k + 1 : k;
  const __nv_bfloat16* xrow = static_cast<const __nv_bfloat16*>(p.x) + t * d;
  auto wcol = [&](int c, int j) { return __ldg(reinterpret_cast<const float4*>(wt + static_cast<long long>(c) * d + j)); };
  // ---- token norm
  float nx = nx_in;
  if (nx < 0.f) {
    float sq = 0.f;
    for (int j = lane * 4; j < d; j += 128) {
      float xv[4];
      Vec4<__nv_bfloat16>::unpack(Vec4<__nv_bfloat16>::load(xrow + j), xv);
      sq = fmaf(xv[0], xv[0], fmaf(xv[1], xv[1], fmaf(xv[2], xv[2], fmaf(xv[3], xv[3], sq))));
    }
    nx = sqrtf(warp_sum(sq));
  }
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
      float dl = kFilterMargin * nx * cn[e];
      if (noisy) {
        z[s] = za[s];
        h += ep[s] * softplus_f32(z[s]);
        dl += fabsf(ep[s]) * kFilterMargin * nx * cn[E + e];  // softplus is 1-Lipschitz
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
  unsigned cm[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) cm[s] = __ballot_sync(0xffffffffu, lane + 32 * s < E && !(up[s] < L));
  // ---- top-1 without a backup rank, a single candidate: the bounds alone
  // prove it is the top expert (its lower end L is above every other upper
  // end), and its gate, the softmax over the one selected logit, is exactly
  // 1 -- what rank_token writes after the recomputation below.  The token is
  // written at once, unless the bounds leave room for a near tie (top minus
  // the best other fp32 logit below kNearTie: that counter needs the values).
  if (k == 1 && kr == 1) {
    int ncand = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) ncand += __popc(cm[s]);
    if (ncand == 1) {
      float other_up = -INFINITY;
      int win = -1;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        if (e < E) {
          if ((cm[s] >> lane) & 1u) win = e;
          else other_up = fmaxf(other_up, up[s]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        other_up = fmaxf(other_up, __shfl_xor_sync(0xffffffffu, other_up, o));
        win = max(win, __shfl_xor_sync(0xffffffffu, win, o));
      }
      if (L - other_up >= 2.0f * kNearTie) {  // false for any NaN or infinity
        if (lane == 0) {
          p.idx[t] = win;
          p.w[t] = 1.0f;
        }
        return;
      }
    }
  }
  // ---- exact fp32 logits of the candidates, four at a time (warp-uniform)
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
  rank_token<__nv_bfloat16, SLOTS>(p, t, lane, g, z, ep, nx, cn, gam, wcol, n_recomputed, n_near, xb);
}

}  // namespace router_detail
}  // namespace moe
