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
// One kernel, deterministic: block b takes a contiguous run of tokens; a
// warp per token forms the softmax of its logits in fp32 (lane e holds
// expert e + 32 s), accumulates p and the token's entropy in fp64 in token
// order, and the block histograms its tokens' selected experts in shared
// memory (integer adds).  Warps, then blocks, are summed in index order;
// the last block to finish (a ticket) reduces the per-block partials and
// writes f, P and the summary, then clears the ticket for the next call.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int SB = 256;  // threads per block
constexpr int SW = SB / 32;

__global__ void __launch_bounds__(SB) routing_stats_kernel(StatsParams p) {
  constexpr int SLOTS = kMaxExperts / 32;
  __shared__ double s_p[SW][kMaxExperts];
  __shared__ double s_ent[SW];
  __shared__ int s_load[kMaxExperts];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k;
  const long long T = p.T;
  const int nb = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const long long per = (T + nb - 1) / nb;
  const long long t0 = b * per, t1 = min(T, t0 + per);

  for (int e = tid; e < kMaxExperts; e += SB) s_load[e] = 0;
  pdl_wait();  // logits, top-k table and dispatch counts come from the predecessors
  __syncthreads();

  // ---- probability mass and entropy, a warp per token, tokens in order
  double acc[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) acc[s] = 0.0;
  double ent = 0.0;
  for (long long t = t0 + warp; t < t1; t += SW) {
    float l[SLOTS];
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = lane + 32 * s;
      l[s] = e < E ? __ldg(p.logits + t * E + e) : -INFINITY;
      m = fmaxf(m, l[s]);
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    float ex[SLOTS], sum = 0.f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      ex[s] = lane + 32 * s < E ? expf(l[s] - m) : 0.f;
      sum += ex[s];
    }
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
    float h = 0.f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const float pr = ex[s] * inv;
      acc[s] += static_cast<double>(pr);
      if (pr > 0.f) h -= pr * logf(pr);
    }
    ent += static_cast<double>(warp_sum(h));
  }
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) s_p[warp][lane + 32 * s] = acc[s];
  if (lane == 0) s_ent[warp] = ent;

  // ---- routed loads of this block's tokens (before the capacity cut)
  for (long long a = t0 * k + tid; a < t1 * k; a += SB) {
    const int e = __ldg(p.idx + a);
    if (e >= 0 && e < E) atomicAdd(&s_load[e], 1);
    else record_error(p.err, MOE_ERR_BOUNDS);
  }
  __syncthreads();

  // ---- this block's partials, warps summed in order
  double* part = p.part + static_cast<long long>(b) * (E + 1);
  int* lpart = p.load_part + static_cast<long long>(b) * E;
  for (int e = tid; e < E; e += SB) {
    double v = 0.0;
    for (int w = 0; w < SW; ++w) v += s_p[w][e];
    part[e] = v;
    lpart[e] = s_load[e];
  }
  if (tid == 0) {
    double v = 0.0;
    for (int w = 0; w < SW; ++w) v += s_ent[w];
    part[E] = v;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.ticket, 1) == nb - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last block: blocks summed in order; f, P and the summary
  __shared__ double s_f[kMaxExperts], s_P[kMaxExperts], s_ld[kMaxExperts];
  const double Td = static_cast<double>(T), TK = static_cast<double>(T) * k;
  for (int e = tid; e < E; e += SB) {
    double ps = 0.0;
    long long ld = 0;
    for (int b2 = 0; b2 < nb; ++b2) {
      ps += __ldcg(p.part + static_cast<long long>(b2) * (E + 1) + e);
      ld += __ldcg(p.load_part + static_cast<long long>(b2) * E + e);
    }
    s_P[e] = T > 0 ? ps / Td : 0.0;
    s_ld[e] = static_cast<double>(ld);
    s_f[e] = T > 0 ? s_ld[e] / TK : 0.0;
    p.P[e] = s_P[e];
    p.f[e] = s_f[e];
  }
  __syncthreads();
  if (tid == 0) {
    double ent_sum = 0.0;
    for (int b2 = 0; b2 < nb; ++b2) ent_sum += __ldcg(p.part + static_cast<long long>(b2) * (E + 1) + E);
    double aux = 0.0, lmean = 0.0, kmean = 0.0;
    int used = 0;
    for (int e = 0; e < E; ++e) {
      aux += s_f[e] * s_P[e];
      lmean += s_ld[e];
      kmean += p.counts[e];
      used += p.counts[e] > 0;
    }
    lmean /= E;
    kmean /= E;
    double lvar = 0.0, kvar = 0.0;
    for (int e = 0; e < E; ++e) {
      const double dl = s_ld[e] - lmean, dk = p.counts[e] - kmean;
      lvar += dl * dl;
      kvar += dk * dk;
    }
    p.summary[0] = static_cast<double>(E) * aux;
    p.summary[1] = T > 0 ? ent_sum / Td : 0.0;
    p.summary[2] = lmean > 0 ? sqrt(lvar / E) / lmean : 0.0;
    p.summary[3] = kmean > 0 ? sqrt(kvar / E) / kmean : 0.0;
    p.summary[4] = static_cast<double>(used) / E;
    p.summary[5] = T > 0 ? static_cast<double>(*p.dropped) / TK : 0.0;
    *p.ticket = 0;  // the next call starts from zero
  }
  pdl_trigger();
}

}  // namespace

int stats_blocks(long long T) {
  const long long want = (T + 255) / 256;
  return static_cast<int>(want < 1 ? 1 : (want > kStatsMaxBlocks ? kStatsMaxBlocks : want));
}

cudaError_t launch_routing_stats(const StatsParams& p, cudaStream_t st) {
  return launch_pdl(routing_stats_kernel, dim3(static_cast<unsigned>(stats_blocks(p.T))), dim3(SB), 0, st, 1, p);
}

}  // namespace moe
