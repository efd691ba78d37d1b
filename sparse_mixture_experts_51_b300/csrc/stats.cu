// Routing diagnostics of one batch and the auxiliary load-balancing loss.
//
// "Mixture-of-Experts Sparse Model Scaling", Mathematical Formulation:
// L_aux = N * sum_i f_i * P_i with f_i the fraction of the batch dispatched
// to expert i (hard count) and P_i the mean routing probability of expert i
// (Lab 2: the full softmax of the router logits); "LLM part 09", s4 states
// the same loss; "Mixture-of-experts Models", Level 3 (load-balancing
// diagnostics), wants the probability mass and the realised loads reported
// together, with overflow, utilisation and a named imbalance measure.  With top-k routing f_i counts every
// selected assignment before the capacity cut, over T*k (f sums to 1).
//
// One kernel, deterministic: one wave of blocks, block b taking a
// contiguous run of tokens; a warp per token (four in flight) forms the
// softmax of its logits in fp32 (lane holds experts lane + 32 s).  Every sum
// is an exact integer sum, so its order does not matter: each probability is
// added as the fixed-point integer round(p * 2^sp) (sp = 62 - bits(T), so the
// sum of T of them fits in 63 bits; error at most 2^-(sp+1) per token), each
// token's entropy as round(h * 2^sh) (h <= ln 128 < 8), each selected expert
// as a count.  Lanes, then the block (shared-memory atomics), then the grid
// (global atomics) add them up; the last block to finish (a ticket) turns
// the totals into f, P and the summary in fp64, then clears the totals and
// the ticket for the next call.  (B300's fp64 pipe is slow: long fp64 add
// chains cost more than the whole rest of the kernel.)
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int SB = 256;  // threads per block
constexpr int SW = SB / 32;
constexpr int TPW = 4;   // tokens a warp has in flight

// Sum of v over the 32 lanes in a fixed butterfly order (deterministic).
__device__ __forceinline__ double warp_sum_fixed(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int bit_length(long long v) {
  int b = 0;
  while (v > 0) { ++b; v >>= 1; }
  return b;
}

// SLOTS: 32-expert slots a lane holds (E <= 32 * SLOTS)
template <int SLOTS>
__global__ void __launch_bounds__(SB) routing_stats_kernel(StatsParams p) {
  __shared__ unsigned long long s_p[kMaxExperts], s_h;
  __shared__ int s_load[kMaxExperts];
  __shared__ double s_P[kMaxExperts], s_ld[kMaxExperts], s_cnt[kMaxExperts];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k;
  const long long T = p.T;
  const int nb = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const long long per = (T + nb - 1) / nb;
  const long long t0 = b * per, t1 = min(T, t0 + per);
  // fixed-point scales: T * 2^sp < 2^62 and T * 8 * 2^sh < 2^62
  const int tb = bit_length(T);
  const int sp = 62 - tb, sh = 59 - tb;
  unsigned long long* acc_p = p.acc;            // [E]
  unsigned long long* acc_h = p.acc + E;        // [1]
  unsigned long long* acc_ld = p.acc + E + 1;   // [E]

  for (int e = tid; e < kMaxExperts; e += SB) {
    s_p[e] = 0ull;
    s_load[e] = 0;
  }
  if (tid == 0) s_h = 0ull;
  pdl_wait();  // logits, top-k table and dispatch counts come from the predecessors
  __syncthreads();

  // ---- probability mass and entropy: warp w takes tokens t0 + w + SW*j,
  // TPW of them per round with every load issued before any arithmetic
  unsigned long long up[SLOTS], uh = 0ull;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) up[s] = 0ull;
  for (long long tb0 = t0 + warp; tb0 < t1; tb0 += static_cast<long long>(SW) * TPW) {
    float l[TPW][SLOTS];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const long long t = tb0 + static_cast<long long>(u) * SW;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        l[u][s] = (t < t1 && e < E) ? __ldg(p.logits + t * E + e) : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      if (tb0 + static_cast<long long>(u) * SW >= t1) break;  // warp-uniform
      float m = l[u][0];
#pragma unroll
      for (int s = 1; s < SLOTS; ++s) m = fmaxf(m, l[u][s]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float ex[SLOTS], sum = 0.f;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        ex[s] = lane + 32 * s < E ? expf(l[u][s] - m) : 0.f;
        sum += ex[s];
      }
      sum = warp_sum(sum);
      const float inv = 1.0f / sum;
      float h = 0.f;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const float pr = ex[s] * inv;
        up[s] += __float2ull_rn(ldexpf(pr, sp));
        if (pr > 0.f) h -= pr * logf(pr);
      }
      h = warp_sum(h);
      if (lane == 0) uh += __float2ull_rn(ldexpf(fmaxf(h, 0.f), sh));
    }
  }
#pragma unroll
  for (int s = 0; s < SLOTS; ++s)
    if (lane + 32 * s < E && up[s] != 0ull) atomicAdd(&s_p[lane + 32 * s], up[s]);
  if (lane == 0 && uh != 0ull) atomicAdd(&s_h, uh);

  // ---- routed loads of this block's tokens (before the capacity cut)
  for (long long a = t0 * k + tid; a < t1 * k; a += SB) {
    const int e = __ldg(p.idx + a);
    if (e >= 0 && e < E) atomicAdd(&s_load[e], 1);
    else record_error(p.err, MOE_ERR_BOUNDS);
  }
  __syncthreads();

  // ---- this block's totals into the grid's
  for (int e = tid; e < E; e += SB) {
    if (s_p[e] != 0ull) atomicAdd(acc_p + e, s_p[e]);
    if (s_load[e] != 0) atomicAdd(acc_ld + e, static_cast<unsigned long long>(s_load[e]));
  }
  if (tid == 0 && s_h != 0ull) atomicAdd(acc_h, s_h);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.ticket, 1) == nb - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last block: f, P and the summary
  const double Td = static_cast<double>(T), TK = static_cast<double>(T) * k;
  const double inv_p = T > 0 ? 1.0 / (ldexp(1.0, sp) * Td) : 0.0;
  for (int e = tid; e < E; e += SB) {
    const unsigned long long ap = __ldcg(acc_p + e), al = __ldcg(acc_ld + e);
    s_P[e] = static_cast<double>(ap) * inv_p;
    s_ld[e] = static_cast<double>(al);
    s_cnt[e] = static_cast<double>(__ldg(p.counts + e));
    p.P[e] = s_P[e];
    p.f[e] = T > 0 ? s_ld[e] / TK : 0.0;
  }
  __syncthreads();
  if (warp == 0) {
    // lane holds experts lane + 32 s; fixed-order butterflies
    double aux = 0.0, lsum = 0.0, ksum = 0.0, used = 0.0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      if (e < E) {
        aux += (T > 0 ? s_ld[e] / TK : 0.0) * s_P[e];
        lsum += s_ld[e];
        ksum += s_cnt[e];
        used += s_cnt[e] > 0.0 ? 1.0 : 0.0;
      }
    }
    aux = warp_sum_fixed(aux);
    lsum = warp_sum_fixed(lsum);
    ksum = warp_sum_fixed(ksum);
    used = warp_sum_fixed(used);
    const double lmean = lsum / E, kmean = ksum / E;
    double lvar = 0.0, kvar = 0.0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      if (e < E) {
        const double dl = s_ld[e] - lmean, dk = s_cnt[e] - kmean;
        lvar += dl * dl;
        kvar += dk * dk;
      }
    }
    lvar = warp_sum_fixed(lvar);
    kvar = warp_sum_fixed(kvar);
    if (lane == 0) {
      const unsigned long long ah = __ldcg(acc_h);
      p.summary[0] = static_cast<double>(E) * aux;
      p.summary[1] = T > 0 ? static_cast<double>(ah) / (ldexp(1.0, sh) * Td) : 0.0;
      p.summary[2] = lmean > 0 ? sqrt(lvar / E) / lmean : 0.0;
      p.summary[3] = kmean > 0 ? sqrt(kvar / E) / kmean : 0.0;
      p.summary[4] = used / E;
      p.summary[5] = T > 0 ? static_cast<double>(*p.dropped) / TK : 0.0;
    }
  }
  __syncthreads();
  // the next call starts from zero
  for (int i = tid; i < 2 * E + 1; i += SB) p.acc[i] = 0ull;
  if (tid == 0) *p.ticket = 0;
  pdl_trigger();
}

}  // namespace

int stats_blocks(long long T) {
  // about SW * TPW = 32 tokens per block, so each warp needs one round of
  // loads (measured on B300: 256 tokens per block, eight rounds, took 2.4x longer)
  const long long want = (T + SW * TPW - 1) / (SW * TPW);
  return static_cast<int>(want < 1 ? 1 : (want > kStatsMaxBlocks ? kStatsMaxBlocks : want));
}

cudaError_t launch_routing_stats(const StatsParams& p, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(stats_blocks(p.T)));
  if (p.E <= 32) return launch_pdl(routing_stats_kernel<1>, grid, dim3(SB), 0, st, 1, p);
  if (p.E <= 64) return launch_pdl(routing_stats_kernel<2>, grid, dim3(SB), 0, st, 1, p);
  return launch_pdl(routing_stats_kernel<4>, grid, dim3(SB), 0, st, 1, p);
}

}  // namespace moe
