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
// softmax of its logits in fp32 (lane holds experts lane + 32 s) and adds p
// and the token's entropy to fp64 sums in token order; the block histograms
// its tokens' selected experts in shared memory (integer adds).  Warps,
// then blocks, are summed in a fixed order; the last block to finish (a
// ticket) reduces the per-block partials with every thread, writes f, P
// and the summary, and clears the ticket for the next call.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int SB = 256;  // threads per block
constexpr int SW = SB / 32;
constexpr int TPW = 4;   // tokens a warp has in flight
constexpr int SLOTS = kMaxExperts / 32;

// Sum of v over the 32 lanes in a fixed butterfly order (deterministic).
__device__ __forceinline__ double warp_sum_fixed(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(SB) routing_stats_kernel(StatsParams p) {
  __shared__ double s_p[SW][kMaxExperts + 1];  // per-warp sums of p (column E: entropy)
  __shared__ int s_load[kMaxExperts];
  __shared__ double s_red[2][SB];              // last block: per-thread partial sums
  __shared__ double s_P[kMaxExperts], s_ld[kMaxExperts], s_cnt[kMaxExperts];
  __shared__ double s_ent_total;
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

  // ---- probability mass and entropy: warp w takes tokens t0 + w + SW*j,
  // TPW of them per round with every load issued before any arithmetic
  double acc[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) acc[s] = 0.0;
  double ent = 0.0;
  for (long long tb = t0 + warp; tb < t1; tb += static_cast<long long>(SW) * TPW) {
    float l[TPW][SLOTS];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const long long t = tb + static_cast<long long>(u) * SW;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = lane + 32 * s;
        l[u][s] = (t < t1 && e < E) ? __ldg(p.logits + t * E + e) : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      if (tb + static_cast<long long>(u) * SW >= t1) break;  // warp-uniform
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
        acc[s] += static_cast<double>(pr);
        if (pr > 0.f) h -= pr * logf(pr);
      }
      ent += static_cast<double>(warp_sum(h));
    }
  }
#pragma unroll
  for (int s = 0; s < SLOTS; ++s)
    if (lane + 32 * s < E) s_p[warp][lane + 32 * s] = acc[s];
  if (lane == 0) s_p[warp][E] = ent;

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
  for (int e = tid; e <= E; e += SB) {
    double v = 0.0;
#pragma unroll
    for (int w = 0; w < SW; ++w) v += s_p[w][e];
    part[e] = v;
    if (e < E) lpart[e] = s_load[e];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.ticket, 1) == nb - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last block.  Columns c = 0..E (E: entropy); G threads per column,
  // thread j of column c sums blocks j, j+G, ... in order, then the G
  // partial sums are added in order: a fixed order for a given (T, E).
  const int ncol = E + 1;
  const int G = SB / ncol;  // >= 1 since E <= 128 < SB
  {
    const int c = tid / G, j = tid - c * G;
    double ps = 0.0, ls = 0.0;
    if (c < ncol) {
      for (int b0 = j; b0 < nb; b0 += 8 * G) {
        double pv[8];
        int lv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int b2 = b0 + u * G;
          pv[u] = b2 < nb ? __ldcg(p.part + static_cast<long long>(b2) * ncol + c) : 0.0;
          lv[u] = (b2 < nb && c < E) ? __ldcg(p.load_part + static_cast<long long>(b2) * E + c) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          ps += pv[u];
          ls += static_cast<double>(lv[u]);
        }
      }
    }
    s_red[0][tid] = ps;
    s_red[1][tid] = ls;
  }
  for (int e = tid; e < E; e += SB) s_cnt[e] = static_cast<double>(__ldg(p.counts + e));
  __syncthreads();
  const double Td = static_cast<double>(T), TK = static_cast<double>(T) * k;
  if (tid <= E) {
    double ps = 0.0, ls = 0.0;
    for (int j = 0; j < G; ++j) {
      ps += s_red[0][tid * G + j];
      ls += s_red[1][tid * G + j];
    }
    if (tid < E) {
      s_P[tid] = T > 0 ? ps / Td : 0.0;
      s_ld[tid] = ls;
      p.P[tid] = s_P[tid];
      p.f[tid] = T > 0 ? ls / TK : 0.0;
    } else {
      s_ent_total = ps;
    }
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
      p.summary[0] = static_cast<double>(E) * aux;
      p.summary[1] = T > 0 ? s_ent_total / Td : 0.0;
      p.summary[2] = lmean > 0 ? sqrt(lvar / E) / lmean : 0.0;
      p.summary[3] = kmean > 0 ? sqrt(kvar / E) / kmean : 0.0;
      p.summary[4] = used / E;
      p.summary[5] = T > 0 ? static_cast<double>(*p.dropped) / TK : 0.0;
      *p.ticket = 0;  // the next call starts from zero
    }
  }
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
  return launch_pdl(routing_stats_kernel, dim3(static_cast<unsigned>(stats_blocks(p.T))), dim3(SB), 0, st, 1, p);
}

}  // namespace moe
