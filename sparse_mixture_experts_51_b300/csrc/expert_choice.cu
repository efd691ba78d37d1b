// Expert-choice routing: every expert takes the C' = min(C, T) tokens of the
// batch with the largest router score H[t,e] (equal scores: lower token
// index first); the gate of a chosen (t, e) is the router probability
// p[t,e] = exp(H[t,e] - lse_t).  A token may be taken by no expert (the
// residual carries it) or by several ("Mixture-of-Experts Sparse Model
// Scaling", Advanced Theory & Extensions, expert-choice routing).
//
// Exact selection from fp32 logits.  The router writes each logit v with a
// rigorous radius r (|v - exact| <= r).  For expert e the C'-th largest
// exact score lies in [L, U], L and U the C'-th largest of v - r and of
// v + r (rounded outward).  A token with v - r > U is in the top C', one with
// v + r < L is not; the remaining band is re-evaluated in fp64 and the
// missing places are filled from it by (fp64 score, token index).
//
// One 1024-thread block per expert (the column's bound keys cached in shared
// memory up to 24576 tokens): two 4-pass radix selects (8-bit digits,
// both bounds at once) over the expert's column, an ordered compaction of
// the band, fp64 dot products (a warp per band token), the band ranking,
// and an ordered pass that numbers the chosen tokens in token order: row
// e*C' + j of the expert-grouped buffers holds the expert's j-th token.
#include "common.cuh"
#include "internal.h"
#include "router_rank.cuh"

namespace moe {
namespace {

using router_detail::softplus_f64;

constexpr int ET = 1024;  // threads per block
constexpr int EW = ET / 32;
constexpr int kEcCacheTokens = 24576;  // up to this T the column's bound keys stay in shared memory (192 KB)

// order-preserving maps (a larger value has a larger key; NaN ranks as -inf)
__device__ __forceinline__ uint32_t fkey(float f) {
  if (f != f) f = -INFINITY;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long dkey(double v) {
  if (v != v) v = -INFINITY;
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(v));
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// Sum over the block (every thread gets the total).
__device__ __forceinline__ int block_sum(int v, int* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) s_tmp[warp] = v;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < EW; ++w) tot += s_tmp[w];
  return tot;
}

// Exclusive prefix of `flag` over the block in thread order, plus the block total.
__device__ __forceinline__ int block_scan(bool flag, int* s_tmp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(b & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) s_tmp[warp] = __popc(b);
  __syncthreads();
  int before = 0;
  total = 0;
  for (int w = 0; w < EW; ++w) {
    const int c = s_tmp[w];
    if (w < warp) before += c;
    total += c;
  }
  return before + in_warp;
}

// Warp 0: the digit holding the rem-th largest key from a 256-bin histogram
// (bins scanned from the top); returns the digit and the rank left inside it.
__device__ __forceinline__ void pick_digit(const unsigned* hist, int rem, int& digit, int& rem_out) {
  const int lane = threadIdx.x & 31;
  // lane l covers bins 255-8l .. 248-8l, highest first
  unsigned c[8], s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) { c[i] = hist[255 - 8 * lane - i]; s += c[i]; }
  unsigned inc = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  const unsigned exc = inc - s;
  const bool here = exc < static_cast<unsigned>(rem) && inc >= static_cast<unsigned>(rem);
  const unsigned who = __ballot_sync(0xffffffffu, here);
  const int src = who ? __ffs(who) - 1 : 31;
  int dg = 0, left = rem;
  if (lane == src) {
    unsigned acc = exc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (acc + c[i] >= static_cast<unsigned>(rem)) { dg = 255 - 8 * lane - i; left = rem - static_cast<int>(acc); break; }
      acc += c[i];
    }
  }
  digit = __shfl_sync(0xffffffffu, dg, src);
  rem_out = __shfl_sync(0xffffffffu, left, src);
}

template <typename TX>
__global__ void __launch_bounds__(ET, 1) ec_select_kernel(EcParams p) {
  __shared__ unsigned hist[2][256];
  __shared__ int s_tmp[EW];
  __shared__ int s_dig[2], s_rem[2];
  __shared__ double s_h[ET];
  __shared__ int s_t[ET];
  extern __shared__ uint32_t s_keys[];  // [2][T] when T <= kEcCacheTokens: lower, upper keys
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  const int T = p.T, E = p.E, Cp = p.Cp;
  const bool cached = T <= kEcCacheTokens;
  uint8_t* flag = p.flag + static_cast<long long>(e) * T;
  int32_t* band = p.band + static_cast<long long>(e) * T;
  double* h64 = p.h64 + static_cast<long long>(e) * T;
  pdl_wait();  // logits, radii and lse come from the router

  auto lo_hi_global = [&](int t, uint32_t& klo, uint32_t& khi) {
    const float v = __ldg(p.logits + static_cast<long long>(t) * E + e);
    const float r = __ldg(p.radius + static_cast<long long>(t) * E + e);
    klo = fkey(__fsub_rd(v, r));
    khi = fkey(__fadd_ru(v, r));
  };
  if (cached) {
    for (int t = tid; t < T; t += ET) lo_hi_global(t, s_keys[t], s_keys[T + t]);
    __syncthreads();
  }
  auto lo_hi = [&](int t, uint32_t& klo, uint32_t& khi) {
    if (cached) {
      klo = s_keys[t];
      khi = s_keys[T + t];
    } else {
      lo_hi_global(t, klo, khi);
    }
  };

  if (Cp == 0 || Cp >= T) {
    for (int t = tid; t < T; t += ET) flag[t] = Cp == 0 ? 0 : 1;
  } else {
    // ---- L = Cp-th largest (v - r), U = Cp-th largest (v + r): radix select, both at once
    uint32_t pre[2] = {0u, 0u}, msk = 0u;
    int rem[2] = {Cp, Cp};
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 512; i += ET) (&hist[0][0])[i] = 0u;
      __syncthreads();
      for (int t = tid; t < T; t += ET) {
        uint32_t klo, khi;
        lo_hi(t, klo, khi);
        if ((klo & msk) == pre[0]) atomicAdd(&hist[0][(klo >> shift) & 255u], 1u);
        if ((khi & msk) == pre[1]) atomicAdd(&hist[1][(khi >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        for (int w = 0; w < 2; ++w) {
          int dg, left;
          pick_digit(hist[w], rem[w], dg, left);
          if (lane == 0) { s_dig[w] = dg; s_rem[w] = left; }
        }
      }
      __syncthreads();
      for (int w = 0; w < 2; ++w) {
        pre[w] |= static_cast<uint32_t>(s_dig[w]) << shift;
        rem[w] = s_rem[w];
      }
      msk |= 255u << shift;
    }
    const uint32_t kL = pre[0], kU = pre[1];

    // ---- classify: in (1), out (0), band (2); the band compacted in token order
    int n_in = 0, nb = 0;
    for (int t0 = 0; t0 < T; t0 += ET) {
      const int t = t0 + tid;
      bool in = false, bd = false;
      if (t < T) {
        uint32_t klo, khi;
        lo_hi(t, klo, khi);
        in = klo > kU;
        bd = !in && !(khi < kL);
        flag[t] = in ? 1 : (bd ? 2 : 0);
      }
      n_in += in ? 1 : 0;
      int tot;
      const int pos = block_scan(bd, s_tmp, tot);
      if (bd) band[nb + pos] = t;
      nb += tot;
    }
    n_in = block_sum(n_in, s_tmp);
    const int need = Cp - n_in;  // places left for the band (1 <= need <= nb)
    if (need < 1 || need > nb) {
      if (tid == 0) record_error(p.err, MOE_ERR_BOUNDS);  // cannot happen with valid radii
    }
    __syncthreads();

    // ---- fp64 scores of the band tokens, a warp per token
    const bool noisy = p.W_n != nullptr;
    for (int i = warp; i < nb; i += EW) {
      const int t = band[i];
      const TX* xrow = static_cast<const TX*>(p.x) + static_cast<long long>(t) * p.d;
      double hg = 0.0, hz = 0.0;
      for (int j = lane; j < p.d; j += 32) {
        const double xv = static_cast<double>(to_f32<TX>(xrow[j]));
        hg = fma(xv, static_cast<double>(__ldg(p.W_g + static_cast<long long>(j) * E + e)), hg);
        if (noisy) hz = fma(xv, static_cast<double>(__ldg(p.W_n + static_cast<long long>(j) * E + e)), hz);
      }
      hg = warp_sum_d(hg);
      hz = warp_sum_d(hz);
      double v = hg;
      if (p.b_g) v += static_cast<double>(__ldg(p.b_g + e));
      if (noisy) v += static_cast<double>(__ldg(p.eps + static_cast<long long>(t) * E + e)) * softplus_f64(hz);
      if (lane == 0) h64[i] = v;
    }
    __syncthreads();

    // ---- the `need` best band tokens by (fp64 score desc, token asc)
    if (nb <= ET) {
      if (tid < nb) { s_h[tid] = h64[tid]; s_t[tid] = band[tid]; }
      __syncthreads();
      if (tid < nb) {
        const unsigned long long ki = dkey(s_h[tid]);
        int rank = 0;
        for (int j = 0; j < nb; ++j) {
          const unsigned long long kj = dkey(s_h[j]);
          rank += (kj > ki || (kj == ki && s_t[j] < s_t[tid])) ? 1 : 0;
        }
        if (rank < need) flag[s_t[tid]] = 1;
      }
    } else {
      // radix select of the need-th largest fp64 key (8 passes), then equal
      // keys in band (= token) order
      unsigned long long kpre = 0ull, kmsk = 0ull;
      int krem = need;
      for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += ET) hist[0][i] = 0u;
        __syncthreads();
        for (int i = tid; i < nb; i += ET) {
          const unsigned long long k = dkey(h64[i]);
          if ((k & kmsk) == kpre) atomicAdd(&hist[0][(k >> shift) & 255ull], 1u);
        }
        __syncthreads();
        if (warp == 0) {
          int dg, left;
          pick_digit(hist[0], krem, dg, left);
          if (lane == 0) { s_dig[0] = dg; s_rem[0] = left; }
        }
        __syncthreads();
        kpre |= static_cast<unsigned long long>(s_dig[0]) << shift;
        krem = s_rem[0];
        kmsk |= 255ull << shift;
      }
      // krem = how many of the keys equal to kpre are still needed
      int taken_eq = 0;
      for (int i0 = 0; i0 < nb; i0 += ET) {
        const int i = i0 + tid;
        unsigned long long k = 0ull;
        if (i < nb) k = dkey(h64[i]);
        const bool eq = i < nb && k == kpre;
        int tot;
        const int pos = block_scan(eq, s_tmp, tot);
        if (i < nb && (k > kpre || (eq && taken_eq + pos < krem))) flag[band[i]] = 1;
        taken_eq += tot;
      }
    }
    __syncthreads();
  }
  __syncthreads();

  // ---- number the chosen tokens in token order; gates p[t,e]
  int base = 0;
  const long long row0 = static_cast<long long>(e) * Cp;
  for (int t0 = 0; t0 < T; t0 += ET) {
    const int t = t0 + tid;
    const bool ch = t < T && flag[t] == 1;
    int tot;
    const int j = base + block_scan(ch, s_tmp, tot);
    if (t < T) {
      const long long te = static_cast<long long>(t) * E + e;
      if (ch && j < Cp) {
        const long long row = row0 + j;
        const float v = __ldg(p.logits + te);
        const float g = (v == v) ? expf(v - __ldg(p.lse + t)) : 0.f;
        p.sel[row] = t;
        p.row_of[te] = static_cast<int32_t>(row);
        p.gate_te[te] = g;
      } else {
        p.row_of[te] = -1;
      }
    }
    base += tot;
  }
  if (tid == 0 && base != Cp) record_error(p.err, MOE_ERR_BOUNDS);
  pdl_trigger();
}

// counts / offsets of the expert-grouped rows, and the tokens no expert chose
__global__ void __launch_bounds__(256) ec_finalize_kernel(EcParams p, int32_t* counts, int32_t* offsets,
                                                          long long* dropped) {
  __shared__ int s_cnt;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) {
      if (e < p.E) counts[e] = p.Cp;
      offsets[e] = e * p.Cp;
    }
  }
  bool any = false;
  if (t < p.T) {
    const int32_t* r = p.row_of + static_cast<long long>(t) * p.E;
    for (int e = 0; e < p.E && !any; ++e) any = __ldg(r + e) >= 0;
  }
  const unsigned b = __ballot_sync(0xffffffffu, t < p.T && !any);
  if ((threadIdx.x & 31) == 0 && b) atomicAdd(&s_cnt, __popc(b));
  __syncthreads();
  if (threadIdx.x == 0 && s_cnt) atomicAdd(reinterpret_cast<unsigned long long*>(dropped),
                                           static_cast<unsigned long long>(s_cnt));
}

// x_perm[row] = x[sel[row]], a warp per row
template <int VB>
__global__ void __launch_bounds__(256) ec_gather_kernel(EcParams p, const void* x, void* x_perm, int elem_bytes,
                                                        long long rows) {
  pdl_wait();
  pdl_trigger();
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int t = p.sel[row];
  if (t < 0 || t >= p.T) {
    if (lane == 0) record_error(p.err, MOE_ERR_BOUNDS);
    return;
  }
  const long long row_bytes = static_cast<long long>(p.d) * elem_bytes;
  const char* src = static_cast<const char*>(x) + t * row_bytes;
  char* dst = static_cast<char*>(x_perm) + row * row_bytes;
  if constexpr (VB == 16) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (long long i = lane; i < row_bytes / 16; i += 32) d4[i] = __ldg(&s4[i]);
  } else {
    const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
    uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
    for (long long i = lane; i < row_bytes / 4; i += 32) d1[i] = __ldg(&s1[i]);
  }
}

}  // namespace

template <typename TX>
cudaError_t launch_ec_select_t(const EcParams& p, cudaStream_t st) {
  const size_t smem = p.T <= kEcCacheTokens ? sizeof(uint32_t) * 2 * static_cast<size_t>(p.T) : 0;
  cudaError_t e = cudaFuncSetAttribute(ec_select_kernel<TX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(uint32_t) * 2 * kEcCacheTokens));
  if (e != cudaSuccess) return e;
  return launch_pdl(ec_select_kernel<TX>, dim3(static_cast<unsigned>(p.E)), dim3(ET), smem, st, 1, p);
}

cudaError_t launch_ec_select(const EcParams& p, int dtype, cudaStream_t st) {
  if (p.E == 0 || p.T == 0) return cudaSuccess;
  return dtype == MOE_BF16 ? launch_ec_select_t<__nv_bfloat16>(p, st) : launch_ec_select_t<float>(p, st);
}

cudaError_t launch_ec_finalize(const EcParams& p, int32_t* counts, int32_t* offsets, long long* dropped,
                               cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(dropped, 0, sizeof(long long), st);
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>(p.T > 0 ? (p.T + 255) / 256 : 1);
  return launch_pdl(ec_finalize_kernel, dim3(blocks), dim3(256), 0, st, 1, p, counts, offsets, dropped);
}

cudaError_t launch_ec_gather(const EcParams& p, const void* x, void* x_perm, int elem_bytes, cudaStream_t st) {
  const long long rows = static_cast<long long>(p.E) * p.Cp;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows * 32 + 255) / 256;
  const bool vec16 = (static_cast<long long>(p.d) * elem_bytes) % 16 == 0;
  if (vec16)
    return launch_pdl(ec_gather_kernel<16>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p, x, x_perm,
                      elem_bytes, rows);
  return launch_pdl(ec_gather_kernel<4>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p, x, x_perm,
                    elem_bytes, rows);
}

}  // namespace moe
