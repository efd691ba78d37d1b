// Shared pieces of the two router kernels (router.cu, router_tiled.cu):
// 16- and 8-byte token loads widened to fp32, cp.async helpers, the fp64
// re-evaluation of candidate experts, and the per-token ranking with its
// rigorous fp32 error bound (see router.cu for the method).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace router_detail {

constexpr float kU = 5.9604644775390625e-8f;  // unit roundoff of fp32, 2^-24
// a token is counted as a near tie when its k-th and (k+1)-th fp32 logits
// are closer than this (a diagnostic; the selection is exact either way)
constexpr float kNearTie = 1e-4f;

template <typename TX>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& q, float (&v)[8]) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& q, float (&v)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// Four consecutive elements of a token row, widened to fp32, from one aligned load.
template <typename TX>
struct Vec4;
template <>
struct Vec4<float> {
  using raw = uint4;
  __device__ static raw load(const float* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ static void unpack(const raw& q, float (&v)[4]) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
  __device__ static raw zero() { return make_uint4(0u, 0u, 0u, 0u); }
};
template <>
struct Vec4<__nv_bfloat16> {
  using raw = uint2;
  __device__ static raw load(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
  __device__ static void unpack(const raw& q, float (&v)[4]) {
    v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
  }
  __device__ static raw zero() { return make_uint2(0u, 0u); }
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

// fp64 dot products of token row xrow (length d, d % 4 == 0) with the
// router-weight columns of up to four experts ce[0..n): column e of W_g and,
// with the noise projection, column e of W_noise.  wcol(c, j) returns rows
// j..j+3 of column c of the combined [W_g | W_noise].  Lanes stride d four
// elements at a time; the partial sums are then added across the warp.
template <typename TX, typename WCol>
__device__ __forceinline__ void dots_f64(const TX* xrow, int d, int E, bool noisy, int lane, int n,
                                         const int (&ce)[4], WCol wcol, double (&hg)[4], double (&hz)[4]) {
  using V = Vec4<TX>;
#pragma unroll
  for (int q = 0; q < 4; ++q) { hg[q] = 0.0; hz[q] = 0.0; }
#pragma unroll 4
  for (int j = lane * 4; j < d; j += 128) {
    float xv[4];
    V::unpack(V::load(xrow + j), xv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < n) {
        const float4 w = wcol(ce[q], j);
        hg[q] = fma(static_cast<double>(xv[0]), static_cast<double>(w.x), hg[q]);
        hg[q] = fma(static_cast<double>(xv[1]), static_cast<double>(w.y), hg[q]);
        hg[q] = fma(static_cast<double>(xv[2]), static_cast<double>(w.z), hg[q]);
        hg[q] = fma(static_cast<double>(xv[3]), static_cast<double>(w.w), hg[q]);
        if (noisy) {
          const float4 u = wcol(E + ce[q], j);
          hz[q] = fma(static_cast<double>(xv[0]), static_cast<double>(u.x), hz[q]);
          hz[q] = fma(static_cast<double>(xv[1]), static_cast<double>(u.y), hz[q]);
          hz[q] = fma(static_cast<double>(xv[2]), static_cast<double>(u.z), hz[q]);
          hz[q] = fma(static_cast<double>(xv[3]), static_cast<double>(u.w), hz[q]);
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    hg[q] = warp_sum_d(hg[q]);
    hz[q] = warp_sum_d(hz[q]);
  }
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const uint32_t d = smem_u32(dst);
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool valid) {
  const uint32_t d = smem_u32(dst);
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// eps[t, lane + 32 s] for the noisy logits (0 without noise or past the end).
template <int SLOTS>
__device__ __forceinline__ void load_eps(const RouterParams& p, long long t, int lane, float (&ep)[SLOTS]) {
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int e = lane + 32 * s;
    ep[s] = (p.eps != nullptr && p.W_n != nullptr && t < p.T && e < p.E) ? __ldg(p.eps + t * p.E + e) : 0.f;
  }
}

// ---------------------------------------------------------------- ranking
// One warp ranks token t.  Lane e + 32 s holds, in g[s] (and z[s] with the
// noise projection), the fp32 contraction of expert e = lane + 32 s, whose
// rounding error is at most gam * nx * ||W column|| (cn: column norms of the
// combined [W_g | W_noise], nc entries).  Writes idx/w (and the
// logits when asked); n_recomputed / n_near count settled-in-fp64 tokens and
// near ties (warp-uniform).
// ep[s] is eps[t, lane + 32 s] (loaded early by the caller; unused without noise).
// xb[s] is added to that expert's error bound (a caller whose value for the
// expert came from elsewhere states its error there; 0 otherwise).
template <typename TX, int SLOTS, typename WCol>
__device__ __forceinline__ void rank_token(const RouterParams& p, long long t, int lane, const float (&g)[SLOTS],
                                           const float (&z)[SLOTS], const float (&ep_in)[SLOTS], float nx,
                                           const float* cn, float gam, WCol wcol, int& n_recomputed,
                                           int& n_near, const float (&xb)[SLOTS]) {
  const int E = p.E, k = p.k, d = p.d;
  // ranks settled exactly: the top k, and the (k+1)-th too when the backup is asked for
  const int kr = (p.backup != nullptr && k < E) ? k + 1 : k;
  const bool noisy = p.W_n != nullptr;
  float H[SLOTS], B[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int e = lane + 32 * s;
    H[s] = -INFINITY;
    B[s] = 0.f;
    if (e < E) {
      const float b = p.b_g ? __ldg(p.b_g + e) : 0.f;
      const float gb = g[s] + b;
      float h = gb, bound;
      const float cg2 = cn[e];
      if (noisy) {
        const float ep = ep_in[s];
        const float sp = softplus_f32(z[s]);
        const float ns = ep * sp;
        h = gb + ns;
        const float cnz = cn[E + e];
        bound = gam * nx * (cg2 + fabsf(ep) * cnz) + fabsf(ep) * (4e-7f + 3e-7f * sp) +
                4.f * kU * (fabsf(g[s]) + fabsf(b) + fabsf(ns) + fabsf(h));
      } else {
        bound = gam * nx * cg2 + 4.f * kU * (fabsf(g[s]) + fabsf(b) + fabsf(h));
      }
      if (p.logits) p.logits[t * E + e] = h;
      if (h != h) h = -INFINITY;  // NaN ranks last
      H[s] = h;
      B[s] = (bound + xb[s]) * 1.25f + 1e-30f;
      if (p.radius) p.radius[t * E + e] = B[s];
    }
  }
  if (p.idx == nullptr) {
    // expert-choice routing: no per-token top-k; the log-sum-exp of the
    // token's logits gives the router probabilities exp(h - lse)
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) m = fmaxf(m, H[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) sum += (lane + 32 * s < E && m > -INFINITY) ? expf(H[s] - m) : 0.f;
    sum = warp_sum(sum);
    if (lane == 0 && p.lse) p.lse[t] = m > -INFINITY ? m + logf(sum) : -INFINITY;
    return;
  }

  // top-k by fp32 value (ties -> lower index), carrying the bounds; lane r < k
  // holds rank r; trank[s] is the rank slot s was taken at (-1: not taken)
  float my_h = -INFINITY, my_b = 0.f;
  int my_e = 0x7fffffff;
  int trank[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) trank[s] = -1;
  for (int r = 0; r < kr; ++r) {
    float bv = -INFINITY, bb = 0.f;
    int be = 0x7fffffff;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      if (e < E && trank[s] < 0 && better(H[s], e, bv, be)) { bv = H[s]; bb = B[s]; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const float b2 = __shfl_xor_sync(0xffffffffu, bb, o);
      const int e2 = __shfl_xor_sync(0xffffffffu, be, o);
      if (better(v2, e2, bv, be)) { bv = v2; bb = b2; be = e2; }
    }
    if (lane == r) { my_h = bv; my_b = bb; my_e = be; }
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
      if ((be & 31) == lane && (be >> 5) == s) trank[s] = r;
  }
  // best value and best upper bound among the experts left out
  float restH = -INFINITY, restU = -INFINITY;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int e = lane + 32 * s;
    if (e < E && trank[s] < 0) {
      restH = fmaxf(restH, H[s]);
      restU = fmaxf(restU, H[s] + B[s]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    restH = fmaxf(restH, __shfl_xor_sync(0xffffffffu, restH, o));
    restU = fmaxf(restU, __shfl_xor_sync(0xffffffffu, restU, o));
  }
  // rank r is exact when its lower end lies above the upper end of every
  // expert ranked below it: a suffix maximum of the upper ends over lanes
  // (lane k carries the experts left out).
  float sm = lane < kr ? my_h + my_b : (lane == kr ? restU : -INFINITY);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n2 = __shfl_down_sync(0xffffffffu, sm, o);
    if (lane + o < 32) sm = fmaxf(sm, n2);
  }
  const float below = __shfl_down_sync(0xffffffffu, sm, 1);
  const float lo = my_h - my_b;
  const float h_k = __shfl_sync(0xffffffffu, my_h, k & 31);  // the (k+1)-th value when it was ranked
  bool safe = true, near = false;
  if (lane < kr) {
    safe = lo > below && lo > -INFINITY && my_b < INFINITY;
    if (lane == k - 1 && k < E) near = my_h - (kr > k ? h_k : restH) < kNearTie;
  }
  if (__any_sync(0xffffffffu, near)) ++n_near;
  const unsigned unsafe = __ballot_sync(0xffffffffu, !safe) & ((1u << kr) - 1u);

  if (unsafe != 0u) {
    // ranks [0, p0) are exact; re-evaluate in fp64 the experts that may hold
    // ranks p0..k-1: those ranks' experts, and every expert left out whose
    // upper end reaches the lowest of their lower ends
    ++n_recomputed;
    const int p0 = __ffs(unsafe) - 1;
    float L = (lane >= p0 && lane < kr) ? lo : INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L = fminf(L, __shfl_xor_sync(0xffffffffu, L, o));
    const TX* xrow = static_cast<const TX*>(p.x) + t * d;
    double h64[SLOTS];
    unsigned cm[SLOTS], cmask[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      h64[s] = -INFINITY;
      cm[s] = __ballot_sync(0xffffffffu, e < E && (trank[s] >= p0 || (trank[s] < 0 && !(H[s] + B[s] < L))));
      cmask[s] = cm[s];
    }
    // candidates in groups of four experts (warp-uniform), front-filled
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
      double hg[4], hz[4];
      dots_f64<TX>(xrow, d, E, noisy, lane, n, ce, wcol, hg, hz);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < n) {
          double v = hg[q];
          if (p.b_g) v += static_cast<double>(p.b_g[ce[q]]);
          if (noisy) v += static_cast<double>(p.eps[t * E + ce[q]]) * softplus_f64(hz[q]);
          if (v != v) v = -INFINITY;
#pragma unroll
          for (int s = 0; s < SLOTS; ++s)
            if (lane == (ce[q] & 31) && s == (ce[q] >> 5)) h64[s] = v;
        }
      }
    }
    // ranks p0..k-1 from the fp64 values of the candidates (ties -> lower index)
    bool used[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) used[s] = false;
    for (int r = p0; r < kr; ++r) {
      double bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        const bool cand = (cmask[s] >> lane & 1u) != 0u;
        if (cand && !used[s] && better_d(h64[s], e, bv, be)) { bv = h64[s]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const double v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int e2 = __shfl_xor_sync(0xffffffffu, be, o);
        if (better_d(v2, e2, bv, be)) { bv = v2; be = e2; }
      }
      if (lane == r) { my_h = static_cast<float>(bv); my_e = be; }
#pragma unroll
      for (int s = 0; s < SLOTS; ++s)
        if ((be & 31) == lane && (be >> 5) == s) used[s] = true;
    }
  }

  // gates: softmax over the selected logits, shifted by the largest, summed in
  // rank order; raw gates divide by the sum over every expert instead
  const float top = __shfl_sync(0xffffffffu, my_h, 0);
  const float ex = lane < k ? expf(my_h - top) : 0.f;
  float den = 0.f;
  if (p.gate_raw) {
    float all = 0.f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) all += (lane + 32 * s < E && H[s] > -INFINITY) ? expf(H[s] - top) : 0.f;
    den = warp_sum(all);
  } else {
    for (int r = 0; r < k; ++r) den += __shfl_sync(0xffffffffu, ex, r);
  }
  if (lane < k) {
    p.idx[t * k + lane] = my_e;
    p.w[t * k + lane] = ex / den;
  }
  if (p.backup != nullptr && lane == (kr > k ? k : 0)) p.backup[t] = kr > k ? my_e : -1;
}

__device__ __forceinline__ void flush_stats(const RouterParams& p, int* cnt, int lane, int n_recomputed, int n_near) {
  if (lane == 0 && (n_recomputed | n_near)) {
    atomicAdd(&cnt[0], n_recomputed);
    atomicAdd(&cnt[1], n_near);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (cnt[0]) atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats[0]), static_cast<unsigned long long>(cnt[0]));
    if (cnt[1]) atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats[1]), static_cast<unsigned long long>(cnt[1]));
  }
}

}  // namespace router_detail
}  // namespace moe
