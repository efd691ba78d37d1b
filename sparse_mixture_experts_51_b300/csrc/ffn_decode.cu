// Expert FFN and combine of a decode-sized batch (T <= 128 tokens) as one
// persistent tcgen05 kernel whose first phase does not need the routing.
//
// With T <= 128 every expert's rows fit one 128-row M tile, so computing an
// expert over ALL T tokens costs the tensor cores exactly what computing it
// over its kept rows costs (the same single M tile), and each output row
// depends only on its own input row: the rows of the kept (token, expert)
// pairs come out bit for bit as the grouped GEMMs give them.  The layer is
// then a stream of expert weights (SwiGLU: 3 d F bytes per expert, GELU:
// 2 d F):
//
//   phase 1  h[e*128 + t] = act(x[t] W1[e]^T (, x[t] W3[e]^T)) for every
//            expert e and token t < T (the tile's rows t >= T read zeros);
//            one tile = expert e x 128 (SwiGLU) or 256 (GELU) columns of h,
//            A = the token matrix itself; only the rows of kept (t, e)
//            pairs are stored
//   phase 2  y_perm[offsets[e] + pos[t,r]] = h[e*128 + t] W2[e]^T + b2[e]
//            for every kept assignment (t, r) of expert e: the epilogue
//            scatters each row to its grouped row, other rows are not
//            stored; one tile = expert e x 256 columns
//   combine  out[t] = x[t] + sum over t's kept ranks r (in order) of
//            w[t,r] y_perm[row(t,r)] (+ the shared experts' output); one
//            tile = 16 tokens x 256 columns
//
// (the expert FFN of "Mixture-of-Experts Sparse Model Scaling", Core
// Concepts; y = sum_i G(x)_i E_i(x) of "LLM part 09", s1; a dropped
// assignment skips its expert as in s3: its row is computed but never
// stored or combined).
//
// Self-routed layers (overflow drop, nc = E or 2E logit columns a power of
// two up to 256) also route the batch in the same launch, so the kernel has
// no routing kernels before it in the layer:
//
//   rank tiles  4 tokens each: the fp32 logits x W_g (, x W_noise) on CUDA
//               cores (thread = 4 columns x a run of d, partials summed in
//               order), then one warp per token ranks it exactly with the
//               routers' rank_token (fp64 re-evaluation of any rank the
//               rigorous fp32 bound leaves open) and writes idx, w
//               ("LLM part 09", s2: H = x W_g + b_g (+ eps softplus(x W_n)),
//               top-k, softmax over the selected logits)
//   dispatch    one tile, after every rank tile: the slot of assignment
//               (t, r) in expert e is the number of earlier assignments to
//               e in priority order j = r T + t; slot >= C drops it
//               (s3); counts, segment offsets, dropped
//
// Tiles are claimed one at a time from a ticket in the workspace: the
// routing tiles (self-routed layers), every phase-1 tile, then every
// phase-2 tile (experts in order), then the combine tiles.  A phase-2 tile
// of expert e waits until all phase-1 tiles of e have stored their rows,
// and a combine tile until every active expert's phase-2 tile of its column
// block has (counts of finished epilogue warps); a combine tile fetches
// everything but those rows before it waits.  Every tile a CTA waits on was
// claimed earlier by a CTA that is running and does not wait on anything
// later, so the waits always end.  The routing tables (idx, pos, offsets,
// w) are read only after griddepcontrol.wait, or (self-routed) once the
// dispatch tile has published them; phase 1 of a self-routed layer does not
// wait for them (until they are published it stores every token's hidden
// row); a phase-2 tile of an expert without kept rows is skipped.  A CTA
// that claims a routing tile claims nothing more until its epilogue warps
// have run it, so the routing tiles spread over CTAs.  The last CTA to
// finish clears the ticket and counts for the next call.
//
// Roles per CTA (384 threads): warp 0 claims tiles and issues TMA loads
// (4-stage ring of 48 KB: A 128x64, B 256x64, 128-byte swizzle); warp 1
// issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM accumulators;
// warp 2 owns TMEM; warps 4-11 drain the accumulator (two per TMEM lane
// quarter, half of the 32-column chunks each) with whole-sector stores, and
// run the routing tiles and the combine tiles (one (token, 16-column
// chunk) item per thread).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "router_rank.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGES = 4;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NACC = 2;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = NACC * ACC_COLS;
constexpr int NTHREADS = 384;
constexpr int EPI_WARPS = 8;
constexpr int QN = 4;  // tile-queue slots (claimed tiles handed from the producer to the other roles)

constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 512 /*barriers, queue*/;
// routing tiles (self-routed layers)
constexpr int RTOK = 4;        // tokens per rank tile
constexpr int RSLOTS = 4;      // 32-expert slots a lane holds while ranking (E <= 128)
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int RED_FLOATS = RTOK * 4 * EPI_THREADS;   // partial logits [KSPLIT][RTOK][nc]
constexpr int CNP_FLOATS = 4 * EPI_THREADS;          // partial column sums of squares [KSPLIT][nc]
constexpr int XSQ_FLOATS = RTOK * EPI_THREADS;       // partial token sums of squares [KSPLIT][RTOK]
constexpr int ROUTE_SMEM_WORDS = RED_FLOATS + CNP_FLOATS + 256 /*column norms*/ + XSQ_FLOATS;
constexpr int ROUTE_SMEM_BYTES = ROUTE_SMEM_WORDS * 4;
constexpr int kMaxAssign = 128 * kMaxTopK;           // T * k of a decode-sized batch
constexpr int kMaxItems = kMaxAssign / EPI_THREADS;  // assignments a dispatch thread holds
// the dispatch tile's per-(item, warp) expert histogram, the loads, a flag, the segment offsets
__host__ __device__ constexpr int dispatch_words(int Tk, int E) {
  return ((Tk + EPI_THREADS - 1) / EPI_THREADS) * EPI_WARPS * E + E + 1 + E + 1;
}

struct DecodeArgs {
  int T, d, F, E, k;
  int swiglu;
  int n1, n2;    // N tiles per expert: phase 1 (128 h columns SwiGLU, 256 GELU), phase 2 (256 y columns)
  int kb1, kb2;  // 64-wide k-blocks: d / 64, F / 64
  const float* b1;  // [E, F] or null (GELU)
  const float* b2;  // [E, d] or null
  __nv_bfloat16* h;  // [E*128, F] phase-1 output
  int32_t* idx;
  int32_t* pos;
  int32_t* offsets;
  float* y;        // [rows, d]
  long long rows;  // allocated rows of y
  int* ctrl;       // [0] ticket, [1] finished CTAs, [2, 2+E) finished phase-1 epilogue warps per expert,
                   // [2+E, 2+E+n2) finished phase-2 epilogue warps per 256-column block,
                   // [2+E+n2] finished rank tiles, [3+E+n2] routing tables published
  int* err;
  // the combine (residual + gated sum over the token's kept ranks, in rank order, + shared experts)
  const __nv_bfloat16* x_res;  // [T, d] residual (the tokens)
  float* w;                    // [T, k] gates
  const float* y_shared;       // [T, d] fp32 or null
  __nv_bfloat16* out;          // [T, d]
  float* moe_out;              // [T, d] fp32 or null
  // the same weights as plain pointers, for the L2 prefetch of each CTA's first tile
  const __nv_bfloat16* W1;
  const __nv_bfloat16* W3;
  const __nv_bfloat16* W2;
  int pf_bytes_row;  // bytes of every weight row of its first tile that a CTA prefetches into L2
  // self-routed layers: rank tiles, the capacity, the router's inputs and
  // outputs (rp.idx / rp.w are idx / w above), the dispatch's counts
  int nrank;
  int C;
  RouterParams rp;
  int32_t* counts;
  long long* dropped;
  int32_t* row_of;  // [T, k] grouped row of each assignment (-1: dropped), written by the dispatch tile
};

__device__ __forceinline__ float gelu_f(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }
// silu(a) = a (1 + tanh(a/2)) / 2 with the hardware tanh approximation, as
// in the grouped GEMM (the same formula, so the rows agree bit for bit)
__device__ __forceinline__ float tanh_approx(float v) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float silu_f(float a) {
  const float h = 0.5f * a;
  return fmaf(h, tanh_approx(h), h);
}

__device__ __forceinline__ void st_global_32b(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w),
               "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// orders this thread's generic-proxy accesses before its later async-proxy
// (TMA) accesses of global memory
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The grouped row of assignment a (-1: dropped or invalid): the dispatch
// tile's table (self-routed layers), else offsets[idx[a]] + pos[a].
template <bool kRows>
__device__ __forceinline__ int grouped_row(const DecodeArgs& g, long long a) {
  long long row = -1;
  if (kRows) {
    row = __ldcg(g.row_of + a);
  } else {
    const int ps = __ldcg(g.pos + a);
    const int e = __ldcg(g.idx + a);
    if (ps >= 0 && e >= 0 && e < g.E) row = static_cast<long long>(__ldcg(g.offsets + e)) + ps;
    else if (ps >= 0) row = g.rows;  // an expert id out of range: reported below
  }
  if (row >= g.rows) {
    record_error(g.err, MOE_ERR_BOUNDS);
    row = -1;
  }
  return static_cast<int>(row);  // rows < 2^31 (the workspace's grouped rows)
}

// The combine of 16 tokens x one 256-column block (the standalone combine's
// arithmetic, so the layer output is the same bit for bit): per token t and
// 16-element chunk, acc = fma over the kept ranks r = 0..k-1 of
// w[t,r] * y[row(t,r)], + the shared experts' output, out = bf16(x + acc),
// moe_out = acc.  One (token, chunk) item per thread.  It runs once per CTA
// at the end of the kernel, from a cold instruction cache, so the code is
// kept short: the first KF ranks' rows and gates are requested together,
// their y chunks KB ranks at a time; ranks past KF (k > 8) one by one.
// Everything but the y rows is fetched before `wait` (warp-collective,
// called by every lane; false: give up) returns, so a combine tile taken
// early does that part while its column block's rows are still being stored.
constexpr int COMBINE_TOKENS = 16;
template <bool kRows, typename Wait>
__device__ __forceinline__ bool combine_item(const DecodeArgs& g, int cb, int tg, int item, Wait wait) {
  const int t = tg * COMBINE_TOKENS + item / (BN / 16);
  const int c = cb * BN + (item % (BN / 16)) * 16;
  const bool valid = t < g.T && c < g.d;
  const long long base = valid ? static_cast<long long>(t) * g.d + c : 0;
  const long long a0 = static_cast<long long>(t) * g.k;
  constexpr int KF = 8, KB = 2;
  int row[KF];
  float wt[KF];
#pragma unroll
  for (int r = 0; r < KF; ++r) {
    row[r] = -1;
    wt[r] = 0.f;
    if (valid && r < g.k) {
      wt[r] = __ldcg(g.w + a0 + r);
      row[r] = grouped_row<kRows>(g, a0 + r);
    }
  }
  float rv[16];
  float ys[16];
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(g.x_res + base);
    const uint4 a = __ldcg(src), b = __ldcg(src + 1);
    const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      rv[2 * i] = __uint_as_float(u[i] << 16);
      rv[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) ys[i] = 0.f;
  if (valid && g.y_shared) {
    const float4* ssrc = reinterpret_cast<const float4*>(g.y_shared + base);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldcg(ssrc + q);
      ys[4 * q] = v.x;
      ys[4 * q + 1] = v.y;
      ys[4 * q + 2] = v.z;
      ys[4 * q + 3] = v.w;
    }
  }
  if (!wait()) return false;
  if (!valid) return true;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  auto add_rank = [&](const float4 (&v)[4], float w) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[4 * q] = fmaf(w, v[q].x, acc[4 * q]);
      acc[4 * q + 1] = fmaf(w, v[q].y, acc[4 * q + 1]);
      acc[4 * q + 2] = fmaf(w, v[q].z, acc[4 * q + 2]);
      acc[4 * q + 3] = fmaf(w, v[q].w, acc[4 * q + 3]);
    }
  };
#pragma unroll
  for (int r0 = 0; r0 < KF; r0 += KB) {
    float4 v[KB][4];
#pragma unroll
    for (int r = 0; r < KB; ++r) {
      if (row[r0 + r] >= 0) {
        const float4* ysrc = reinterpret_cast<const float4*>(g.y + static_cast<long long>(row[r0 + r]) * g.d + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[r][q] = __ldcg(ysrc + q);
      }
    }
#pragma unroll
    for (int r = 0; r < KB; ++r)
      if (row[r0 + r] >= 0) add_rank(v[r], wt[r0 + r]);
  }
#pragma unroll 1
  for (int r = KF; r < g.k; ++r) {
    const long long rw = grouped_row<kRows>(g, a0 + r);  // widened for the address
    const float w = __ldcg(g.w + a0 + r);
    if (rw >= 0) {
      const float4* ysrc = reinterpret_cast<const float4*>(g.y + rw * g.d + c);
      float4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = __ldcg(ysrc + q);
      add_rank(v, w);
    }
  }
  if (g.y_shared) {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] += ys[i];
  }
  if (g.moe_out) {
    float4* mo = reinterpret_cast<float4*>(g.moe_out + base);
#pragma unroll
    for (int q = 0; q < 4; ++q) mo[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(rv[2 * i] + acc[2 * i], rv[2 * i + 1] + acc[2 * i + 1]);
    pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  uint4* dst = reinterpret_cast<uint4*>(g.out + base);
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  return true;
}

// ---------------------------------------------------------------- routing tiles
// Shared-memory accesses of the routing tables as such (not generic ones,
// which may wait for this thread's outstanding global stores).
__device__ __forceinline__ float lds_f32(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ int lds_s32(const int* p) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(float* p, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(smem_u32(p)), "f"(v) : "memory");
}
__device__ __forceinline__ void sts_s32(int* p, int v) {
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_v4(float* p, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// A barrier of the eight epilogue warps on an mbarrier (8 arrivals a phase):
// bounded like every wait of the kernel, so a warp that has left on an
// abort cannot hold the others; false when the wait gives up.  `phase` is
// the warp's own count of the barrier's completed phases (mod 2).
struct EpiBar {
  uint32_t bar;
  uint32_t phase;
  int* err;
  volatile int* abort_flag;
  __device__ __forceinline__ bool sync() {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait_bounded(bar, phase, err, abort_flag);
    phase ^= 1u;
    return ok;
  }
};

// One thread waits (bounded) until *flag >= target, acquiring; false on the
// time limit or an abort by another role of the CTA (the error is recorded).
// Polls back off from 32 ns to 256 ns: many CTAs may wait on the same word,
// and polling it flat out floods the L2 slice that holds it (every other
// access to that slice then queues behind the polls).
__device__ __forceinline__ bool wait_flag(const int* flag, int target, int* err, volatile int* abort_flag) {
  if (ld_acquire(flag) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned ns = 32;
  while (ld_acquire(flag) < target) {
    if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, MOE_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(ns);
    ns = ns < 256 ? 2 * ns : 256;
  }
  return true;
}

// The same for a word of this CTA's shared memory (no backoff needed past a few polls).
__device__ __forceinline__ bool wait_shared(const volatile int* flag, int* err, volatile int* abort_flag) {
  const unsigned long long t0 = globaltimer_ns();
  while (*flag == 0) {
    if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, MOE_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(64);
  }
  return *flag > 0;
}

// Rank tile rt: tokens [rt*RTOK, rt*RTOK + RTOK), run by the 256 epilogue
// threads.  Thread (cq, ks) accumulates columns
// 4cq..4cq+3 of the logit table (W_g columns, then W_noise's) for RTOK
// tokens over its run [ks*DKS, ks*DKS + DKS) of d, in order, with fmaf; the
// KSPLIT partials are then summed in ks order, so every logit is an fp32 sum
// of depth at most DKS + KSPLIT, the depth rank_token's rounding bound
// takes.  The column and token norms the bound needs come from the same
// loads.  Then one warp per token ranks it.
__device__ __forceinline__ bool rank_tile(const DecodeArgs& g, int rt, int et, float* rs, EpiBar& eb) {
  const RouterParams& p = g.rp;
  const int E = p.E, d = p.d;
  const bool noisy = p.W_n != nullptr;
  const int nc = noisy ? 2 * E : E;
  const int CQ = nc >> 2, KSPLIT = EPI_THREADS / CQ;
  const int DKS = (d + 8 * KSPLIT - 1) / (8 * KSPLIT) * 8;
  const int cq = et % CQ, ks = et / CQ, c0 = 4 * cq;
  const float* wsrc = c0 < E ? p.W_g + c0 : p.W_n + (c0 - E);
  const long long t0 = static_cast<long long>(rt) * RTOK;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x);
  float* red = rs;                    // [KSPLIT][RTOK][nc]
  float* cnp = rs + RED_FLOATS;       // [KSPLIT][nc]
  float* cnf = cnp + CNP_FLOATS;      // [nc]
  float* xsq = cnf + 256;             // [KSPLIT][RTOK]
  const int wr = et >> 5, lane = et & 31;

  // Every load below would otherwise wait behind the weight stream's queue
  // at HBM, once per step of the loop: the router weights (every rank tile
  // reads all of them; each requests its share) and the tile's token rows
  // are requested into L2 first, all at once.
  {
    const long long wbytes = static_cast<long long>(d) * E * 4;  // a multiple of 16 (E % 4 == 0)
    constexpr long long kChunk = 4096;
    const long long nchunk = (wbytes + kChunk - 1) / kChunk;
    for (long long c = rt + static_cast<long long>(g.nrank) * et; c < nchunk;
         c += static_cast<long long>(g.nrank) * EPI_THREADS) {
      const long long o = c * kChunk;
      const uint32_t n = static_cast<uint32_t>(min(kChunk, wbytes - o));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<const char*>(p.W_g) + o), "r"(n)
                   : "memory");
      if (noisy)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<const char*>(p.W_n) + o),
                     "r"(n)
                     : "memory");
    }
    if (et < RTOK && t0 + et < p.T)  // d * 2 bytes a row, a multiple of 16
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(x + (t0 + et) * d), "r"(static_cast<uint32_t>(d * 2))
                   : "memory");
  }
  const int n_eff = DKS + KSPLIT;
  const float gam = (n_eff * router_detail::kU) / (1.0f - n_eff * router_detail::kU);
  int n_recomputed = 0, n_near = 0;
  auto wcol = [&](int c, int j) {
    const float* W = c < E ? p.W_g + c : p.W_n + (c - E);
    const size_t r0 = static_cast<size_t>(j) * E;
    return make_float4(__ldg(W + r0), __ldg(W + r0 + E), __ldg(W + r0 + 2 * E), __ldg(W + r0 + 3 * E));
  };
  const int jb = ks * DKS, je = min(d, jb + DKS);

  {
    float acc[RTOK][4], wsq[4], xs[RTOK];
#pragma unroll
    for (int m = 0; m < RTOK; ++m) {
      xs[m] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) wsq[q] = 0.f;
#pragma unroll 2
    for (int j = jb; j < je; j += 8) {
      float4 wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        wv[i] = __ldg(reinterpret_cast<const float4*>(wsrc + static_cast<long long>(j + i) * E));
      uint4 xv[RTOK];
#pragma unroll
      for (int m = 0; m < RTOK; ++m)
        xv[m] = t0 + m < p.T ? __ldg(reinterpret_cast<const uint4*>(x + (t0 + m) * d + j)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        wsq[0] = fmaf(wv[i].x, wv[i].x, wsq[0]);
        wsq[1] = fmaf(wv[i].y, wv[i].y, wsq[1]);
        wsq[2] = fmaf(wv[i].z, wv[i].z, wsq[2]);
        wsq[3] = fmaf(wv[i].w, wv[i].w, wsq[3]);
      }
#pragma unroll
      for (int m = 0; m < RTOK; ++m) {
        float xf[8];
        router_detail::Vec16<__nv_bfloat16>::unpack(xv[m], xf);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          xs[m] = fmaf(xf[i], xf[i], xs[m]);
          acc[m][0] = fmaf(xf[i], wv[i].x, acc[m][0]);
          acc[m][1] = fmaf(xf[i], wv[i].y, acc[m][1]);
          acc[m][2] = fmaf(xf[i], wv[i].z, acc[m][2]);
          acc[m][3] = fmaf(xf[i], wv[i].w, acc[m][3]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < RTOK; ++m) sts_v4(red + (ks * RTOK + m) * nc + c0, acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    sts_v4(cnp + ks * nc + c0, wsq[0], wsq[1], wsq[2], wsq[3]);
    if (cq == 0) sts_v4(xsq + ks * RTOK, xs[0], xs[1], xs[2], xs[3]);
    static_assert(RTOK == 4, "one 16-byte row of token sums per run of d");
    if (!eb.sync()) return false;
    for (int c = et; c < nc; c += EPI_THREADS) {
      float s2 = 0.f;
      for (int k2 = 0; k2 < KSPLIT; ++k2) s2 += lds_f32(cnp + k2 * nc + c);
      sts_f32(cnf + c, sqrtf(s2));
    }
    if (!eb.sync()) return false;

    // ---- one warp per token: the partials in ks order, the token norm, the exact ranking
    for (int m = wr; m < RTOK; m += EPI_WARPS) {
      const long long t = t0 + m;
      if (t >= p.T) break;
      float gl[RSLOTS], zl[RSLOTS], ep[RSLOTS], xb[RSLOTS];
      router_detail::load_eps<RSLOTS>(p, t, lane, ep);
#pragma unroll
      for (int sl = 0; sl < RSLOTS; ++sl) {
        const int e = lane + 32 * sl;
        gl[sl] = zl[sl] = xb[sl] = 0.f;
        if (e < E) {
          for (int k2 = 0; k2 < KSPLIT; ++k2) {
            gl[sl] += lds_f32(red + (k2 * RTOK + m) * nc + e);
            if (noisy) zl[sl] += lds_f32(red + (k2 * RTOK + m) * nc + E + e);
          }
        }
      }
      float sq = 0.f;
      for (int k2 = lane; k2 < KSPLIT; k2 += 32) sq += lds_f32(xsq + k2 * RTOK + m);
      const float nx = sqrtf(warp_sum(sq));
      router_detail::rank_token<__nv_bfloat16, RSLOTS>(p, t, lane, gl, zl, ep, nx, cnf, gam, wcol, n_recomputed,
                                                        n_near, xb);
    }
  }
  if (p.stats != nullptr && lane == 0) {
    if (n_recomputed)
      atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats[0]), static_cast<unsigned long long>(n_recomputed));
    if (n_near) atomicAdd(reinterpret_cast<unsigned long long*>(&p.stats[1]), static_cast<unsigned long long>(n_near));
  }
  __threadfence();
  return eb.sync();  // idx / w of the tile are written (and fenced); the partial tables are free again
}

// The dispatch tile, once every rank tile has finished.  Thread et holds the
// assignments j = u * 256 + et (u = 0, 1, ...), so (u, warp, lane) runs in the
// priority order j = r T + t.  Per u, the lanes of a warp holding the same
// expert find each other (match), the first of them records their count in
// the histogram cell (u, warp, e); a per-expert exclusive scan over the
// cells in (u, warp) order then gives each cell's first slot, and the slot of
// an assignment is its cell's first slot + its rank among the matching lanes
// before it: the number of earlier assignments to its expert.  Kept iff the
// slot is below C.  Then counts = min(load, C), offsets = their exclusive
// prefix (offsets[E] = the kept total), dropped = the sum of load - count.
// false: the wait for the rank tiles ran out (error recorded, abort set).
__device__ __forceinline__ bool dispatch_tile(const DecodeArgs& g, int et, const int* ranked, int* sbuf, EpiBar& eb) {
  const int T = g.T, k = g.k, E = g.E, C = g.C;
  const int Tk = T * k;                               // <= kMaxAssign
  const int U = (Tk + EPI_THREADS - 1) / EPI_THREADS;  // items a thread holds
  const int wr = et >> 5, lane = et & 31;
  int* hist = sbuf;                      // [U][EPI_WARPS][E]
  int* s_tot = hist + U * EPI_WARPS * E;  // [E] loads
  int* s_ok = s_tot + E;
  int* s_off = s_ok + 1;                  // [E+1] segment offsets
  for (int i = et; i < U * EPI_WARPS * E; i += EPI_THREADS) sts_s32(hist + i, 0);
  // thread 0 waits for the rank tiles; its result reaches the others through
  // shared memory (written before the barrier, read after it)
  if (et == 0) sts_s32(s_ok, wait_flag(ranked, g.nrank, g.err, eb.abort_flag) ? 1 : 0);
  if (!eb.sync()) return false;
  if (lds_s32(s_ok) == 0) return false;
  (void)ld_acquire(ranked);  // every thread's reads below follow the completed count
  int ev[kMaxItems], rk[kMaxItems];
#pragma unroll
  for (int u = 0; u < kMaxItems; ++u) {  // every load issued before the first use
    const int j2 = u * EPI_THREADS + et;
    ev[u] = -1;
    if (u < U && j2 < Tk) {
      const int r = j2 / T, t = j2 - r * T;
      ev[u] = __ldcg(g.idx + t * k + r);
    }
  }
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int u = 0; u < kMaxItems; ++u) {
    rk[u] = 0;
    if (u < U) {  // uniform
      const int e = ev[u] >= 0 && ev[u] < E ? ev[u] : -1;  // an id out of range takes no slot
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      rk[u] = __popc(peers & lt_mask);
      if (e >= 0 && rk[u] == 0) sts_s32(hist + (u * EPI_WARPS + wr) * E + e, __popc(peers));
    }
  }
  if (!eb.sync()) return false;
  for (int e = et; e < E; e += EPI_THREADS) {
    int run = 0;
    for (int q = 0; q < U * EPI_WARPS; ++q) {
      const int c = lds_s32(hist + q * E + e);
      sts_s32(hist + q * E + e, run);
      run += c;
    }
    sts_s32(s_tot + e, run);
  }
  if (!eb.sync()) return false;
#pragma unroll
  for (int u = 0; u < kMaxItems; ++u) {
    const int j2 = u * EPI_THREADS + et;
    if (u < U && j2 < Tk) {
      const int r = j2 / T, t = j2 - r * T;
      int ps = -1;
      if (ev[u] >= 0 && ev[u] < E) {
        const int slot = lds_s32(hist + (u * EPI_WARPS + wr) * E + ev[u]) + rk[u];
        ps = slot < C ? slot : -1;
      } else {
        record_error(g.err, MOE_ERR_BOUNDS);  // the rank tiles write no such id
      }
      g.pos[t * k + r] = ps;
      rk[u] = ps;  // kept for the grouped rows below
    }
  }
  if (wr == 0) {
    int v[4], run = 0;
    long long drop = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ex = lane * 4 + q;
      const int load = ex < E ? lds_s32(s_tot + ex) : 0;
      v[q] = min(load, C);
      drop += load - v[q];
      run += v[q];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int off = incl - run;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ex = lane * 4 + q;
      if (ex < E) {
        g.counts[ex] = v[q];
        g.offsets[ex] = off;
        sts_s32(s_off + ex, off);
      }
      off += v[q];
    }
    if (lane == 31) g.offsets[E] = incl;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) drop += __shfl_xor_sync(0xffffffffu, drop, o);
    if (lane == 0) *g.dropped = drop;
  }
  if (!eb.sync()) return false;
  // the grouped row of every assignment (-1: dropped), which the combine reads
#pragma unroll
  for (int u = 0; u < kMaxItems; ++u) {
    const int j2 = u * EPI_THREADS + et;
    if (u < U && j2 < Tk) {
      const int r = j2 / T, t = j2 - r * T;
      g.row_of[t * k + r] = rk[u] >= 0 ? lds_s32(s_off + ev[u]) + rk[u] : -1;
    }
  }
  __threadfence();
  return eb.sync();
}

template <bool kRoute>
__global__ void __launch_bounds__(NTHREADS, 1)
    ffn_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW1,
                      const __grid_constant__ CUtensorMap tmW3, const __grid_constant__ CUtensorMap tmH,
                      const __grid_constant__ CUtensorMap tmW2, DecodeArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + STAGES * STAGE_BYTES);
  uint64_t* full = bars;                 // [STAGES]
  uint64_t* empty = full + STAGES;       // [STAGES]
  uint64_t* tfull = empty + STAGES;      // [NACC]
  uint64_t* tempty = tfull + NACC;       // [NACC]
  uint64_t* qfull = tempty + NACC;       // [QN]
  uint64_t* qempty = qfull + QN;         // [QN]
  uint64_t* drain = qempty + QN;         // [1]
  uint64_t* ebar = drain + 1;            // [1] the epilogue warps' group barrier (routing tiles)
  int* s_tile = reinterpret_cast<int*>(ebar + 1);  // [QN]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_tile + QN);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* route_seq = abort_flag + 1;  // routing tiles this CTA's epilogue has finished
  volatile int* s_routed = abort_flag + 2;   // 1: the routing tables are published (-1: the wait failed)
  float* rs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512);  // routing tiles' tables

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = g.E;
  // tile ids: [0, nr) routing (rank tiles, then the dispatch tile), [nr, total1)
  // phase 1, [total1, total12) phase 2, [total12, total) combine
  const int nr = kRoute ? g.nrank + 1 : 0;
  const int total1 = nr + E * g.n1;
  const int total12 = total1 + E * g.n2;
  const int n_tg = (g.T + COMBINE_TOKENS - 1) / COMBINE_TOKENS;
  const int total = total12 + g.n2 * n_tg;  // then one combine tile per 256-column block and 16 tokens
  int* ticket = g.ctrl;
  int* finished = g.ctrl + 1;
  int* done1 = g.ctrl + 2;
  int* done2 = done1 + E;
  int* ranked = done2 + g.n2;
  int* route_done = ranked + 1;
  const int done_target = EPI_WARPS * g.n1;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), EPI_WARPS);
    }
    for (int q = 0; q < QN; ++q) {
      mbar_init(smem_u32(&qfull[q]), 1);
      mbar_init(smem_u32(&qempty[q]), 1 + EPI_WARPS);  // the MMA thread and every epilogue warp
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(ebar), EPI_WARPS);
    *abort_flag = 0;
    *route_seq = 0;
    *s_routed = 0;
    fence_mbarrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW1);
    if (g.swiglu) tma_prefetch_desc(&tmW3);
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmW2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Routed by the routing kernels: no griddepcontrol.wait here, phase 1 reads
  // only the tokens and the weights, which were complete before the router
  // (the first kernel of the chain that launched this one) passed its own
  // wait.  Self-routed: this kernel is the layer's first, and its inputs may
  // be the previous kernel's output.
  if (kRoute) pdl_wait();
  // the routing tables may be read: a warp-collective wait (false: timed out)
  auto tables_ready = [&]() -> bool {
    if (!kRoute) {
      pdl_wait();
      return true;
    }
    // one poller per CTA (the first epilogue warp); the others watch its
    // shared-memory copy, then each lane acquires the word once itself
    int ok = 1;
    if (lane == 0) {
      if (warp == 4) {
        ok = wait_flag(route_done, 1, g.err, abort_flag) ? 1 : 0;
        *s_routed = ok ? 1 : -1;
      } else {
        ok = wait_shared(s_routed, g.err, abort_flag) ? 1 : 0;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)ld_acquire(route_done);  // every lane's reads follow the publication
    return ok != 0;
  };

  if (warp == 0) {
    // ================= tile claims + TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_phase = 0;
      int q = 0;
      uint32_t qphase = 0;
      bool routed = false, ok = true;
      int n_routing = 0;  // routing tiles this CTA claimed
      while (true) {
        int id = -1;
        if (ok) {
          // claim the next tile with work (phase-2 tiles of experts without kept rows are skipped)
          while (true) {
            id = atomicAdd(ticket, 1);
            if (id >= total) { id = -1; break; }
            if (id < total1 || id >= total12) break;
            if (!routed) {
              // the routing tables are complete from here on
              if (kRoute) {
                if (!wait_flag(route_done, 1, g.err, abort_flag)) { id = -1; break; }
              } else {
                pdl_wait();
              }
              routed = true;
            }
            const int e = (id - total1) / g.n2;
            if (__ldcg(g.offsets + e + 1) > __ldcg(g.offsets + e)) break;
          }
        }
        // hand it to the MMA thread and the epilogue warps (-1: no more tiles)
        if (!mbar_wait_bounded(smem_u32(&qempty[q]), qphase ^ 1u, g.err, abort_flag)) id = -1;
        s_tile[q] = id;
        mbar_arrive(smem_u32(&qfull[q]));
        if (++q == QN) { q = 0; qphase ^= 1u; }
        if (id < 0) break;
        if (id < nr) {
          // a routing tile needs no loads; claim nothing more until this
          // CTA's epilogue warps have run it (bounded), so that the routing
          // tiles go to different CTAs
          ++n_routing;
          const unsigned long long t0 = globaltimer_ns();
          while (*route_seq < n_routing) {
            if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
              record_error(g.err, MOE_ERR_DEVICE_TIMEOUT);
              *abort_flag = 1;
              ok = false;
              break;
            }
            __nanosleep(128);
          }
          continue;
        }
        if (id >= total12) {
          // a combine tile needs no loads; a CTA takes one at most (when the
          // grid has a CTA for each), so they run side by side
          if (static_cast<int>(gridDim.x) >= total - total12) ok = false;
          continue;
        }

        const bool p1 = id < total1;
        const int e = p1 ? (id - nr) / g.n1 : (id - total1) / g.n2;
        const int nb = p1 ? (id - nr) - e * g.n1 : (id - total1) - e * g.n2;
        const int KB = p1 ? g.kb1 : g.kb2;
        // phase 2: the B panel needs nothing; A (expert e's rows of h) needs
        // every phase-1 tile of e stored.  Issue the first stages' B loads,
        // then wait, then their A loads.
        bool h_ready = p1 || ld_acquire(done1 + e) >= done_target;
        if (!p1 && h_ready) fence_proxy_async_global();  // the TMA loads of h follow the acquire
        int pend_stage[STAGES];
        int npend = 0;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, g.err, abort_flag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = smem_u32(tiles + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          if (p1) {
            tma_load_2d(sa, &tmX, fb, kb * BK, 0);
            if (g.swiglu) {
              tma_load_2d(sb, &tmW1, fb, kb * BK, e * g.F + nb * 128);
              tma_load_2d(sb + B_BYTES / 2, &tmW3, fb, kb * BK, e * g.F + nb * 128);
            } else {
              tma_load_2d(sb, &tmW1, fb, kb * BK, e * g.F + nb * BN);
            }
          } else {
            tma_load_2d(sb, &tmW2, fb, kb * BK, e * g.d + nb * BN);
            if (h_ready) {
              tma_load_2d(sa, &tmH, fb, kb * BK, e * BM);
            } else {
              pend_stage[npend++] = stage;
              if (npend == STAGES || kb == KB - 1) {
                // bounded wait for the phase-1 rows of expert e
                if (!wait_flag(done1 + e, done_target, g.err, abort_flag)) ok = false;
                // the TMA loads of h below are ordered after the acquire (the
                // pending stages still get their A copies so that every
                // expected transaction arrives)
                fence_proxy_async_global();
                for (int i = 0; i < npend; ++i) {
                  const int s2 = pend_stage[i];
                  const int kb2 = kb - (npend - 1 - i);
                  tma_load_2d(smem_u32(tiles + s2 * STAGE_BYTES), &tmH, smem_u32(&full[s2]), kb2 * BK, e * BM);
                }
                npend = 0;
                h_ready = true;
              }
            }
          }
          issued |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (!ok) break;
        }
      }
      // no copy into this CTA's shared memory is still in flight
      for (int s = 0; s < STAGES; ++s)
        if (issued >> s & 1u) mbar_wait_bounded(smem_u32(&full[s]), (last_phase >> s) & 1u, g.err, nullptr);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      int q = 0;
      uint32_t qphase = 0;
      bool any = false;
      while (true) {
        if (!mbar_wait_bounded(smem_u32(&qfull[q]), qphase, g.err, abort_flag)) break;
        const int id = s_tile[q];
        mbar_arrive(smem_u32(&qempty[q]));
        if (++q == QN) { q = 0; qphase ^= 1u; }
        if (id < 0) break;
        if (id < nr || id >= total12) continue;  // a routing or combine tile: no MMA
        const int KB = id < total1 ? g.kb1 : g.kb2;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), aphase ^ 1u, g.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, g.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + stage * STAGE_BYTES);
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(dt, da + static_cast<uint64_t>(kk * 2), db + static_cast<uint64_t>(kk * 2), IDESC,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty[stage]));
          any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[acc]));
        if (++acc == NACC) { acc = 0; aphase ^= 1u; }
      }
      if (any) {
        umma_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, g.err, nullptr);
      }
    }
  } else if (warp >= 4) {
    // ================= epilogue =================
    const int qd = warp & 3;             // TMEM lane quarter
    const int half = (warp - 4) >> 2;    // which half of the tile's 32-column chunks
    const int t = qd * 32 + lane;        // token (row of the tile)
    int acc = 0;
    uint32_t aphase = 0;
    int q = 0;
    uint32_t qphase = 0;
    bool routed = false;
    bool first = true;
    EpiBar eb{smem_u32(ebar), 0u, g.err, abort_flag};
    while (true) {
      if (!mbar_wait_bounded(smem_u32(&qfull[q]), qphase, g.err, abort_flag)) break;
      const int id = s_tile[q];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&qempty[q]));
      if (++q == QN) { q = 0; qphase ^= 1u; }
      if (id < 0) break;
      if (id < nr) {
        // ---- routing tile (self-routed layers)
        const int et = tid - 4 * 32;
        if (id < g.nrank) {
          if (!rank_tile(g, id, et, rs, eb)) break;
          if (et == 0) atomicAdd(ranked, 1);  // after every thread's fence and the barrier in rank_tile
        } else {
          if (!dispatch_tile(g, et, ranked, reinterpret_cast<int*>(rs), eb)) break;
          if (et == 0) atomicExch(route_done, 1);  // publishes the tables (fenced in dispatch_tile)
        }
        if (et == 0) *route_seq = *route_seq + 1;
        continue;
      }
      if (id >= total12) {
        // ---- combine tile: columns [cb*256, cb*256+256) of 16 tokens, once
        // every active expert's phase-2 tile of that block has stored its rows
        const int cb = (id - total12) / n_tg, tg = (id - total12) - cb * n_tg;
        if (!routed) {
          if (!tables_ready()) break;
          routed = true;
        }
        int n_active = 0;
        for (int e2 = lane; e2 < E; e2 += 32) n_active += __ldcg(g.offsets + e2 + 1) > __ldcg(g.offsets + e2) ? 1 : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n_active += __shfl_xor_sync(0xffffffffu, n_active, o);
        auto block_stored = [&]() -> bool {
          bool ready = true;
          if (lane == 0) ready = wait_flag(done2 + cb, EPI_WARPS * n_active, g.err, abort_flag);
          ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
          if (ready) (void)ld_acquire(done2 + cb);  // every lane's reads of y follow the completed count
          return ready;
        };
        static_assert(COMBINE_TOKENS * (BN / 16) == EPI_WARPS * 32, "one combine item per epilogue thread");
        if (!combine_item<kRoute>(g, cb, tg, (warp - 4) * 32 + lane, block_stored)) break;
        continue;
      }
      const bool p1 = id < total1;
      const int e = p1 ? (id - nr) / g.n1 : (id - total1) / g.n2;
      const int nb = p1 ? (id - nr) - e * g.n1 : (id - total1) - e * g.n2;
      if (!kRoute && first) {
        // The kernel was launched while the routing kernels still run, and
        // the hardware holds tensor-map TMA loads of a kernel launched that
        // way until the kernel before it completes.  While the first tile's
        // loads wait, the idle epilogue warps request the leading part of
        // its weight rows into L2 (one bulk prefetch per row).
        first = false;
        const char* base;
        int nrows;
        long long row_bytes;
        if (p1) {
          row_bytes = static_cast<long long>(g.d) * 2;
          nrows = g.swiglu ? 128 : BN;
          base = reinterpret_cast<const char*>(g.W1) + (static_cast<long long>(e) * g.F + nb * nrows) * row_bytes;
        } else {
          row_bytes = static_cast<long long>(g.F) * 2;
          nrows = BN;
          base = reinterpret_cast<const char*>(g.W2) + (static_cast<long long>(e) * g.d + nb * BN) * row_bytes;
        }
        const int et = (warp - 4) * 32 + lane;
        const int last_row = p1 ? (g.E * g.F) : (g.E * g.d);  // rows of the weight tensor
        const int row0 = p1 ? e * g.F + nb * nrows : e * g.d + nb * BN;
        for (int r = et; r < nrows; r += EPI_WARPS * 32) {
          if (row0 + r >= last_row) continue;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + r * row_bytes), "r"(g.pf_bytes_row)
                       : "memory");
          if (p1 && g.swiglu) {
            const char* b3 = reinterpret_cast<const char*>(g.W3) + (static_cast<long long>(e) * g.F + nb * 128) * row_bytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(b3 + r * row_bytes), "r"(g.pf_bytes_row)
                         : "memory");
          }
        }
      }
      // The routing tables are read from here on.  Waiting for the routing
      // kernels costs nothing at this point: the accumulator this warp is
      // about to drain holds data of TMA loads, and those are released only
      // once the kernel before this one has completed.
      if (!routed && kRoute && p1) {
        // Phase 1 of a self-routed layer does not wait for the routing tables
        // (the routing tiles run their code once per CTA, cold, and take a good
        // part of phase 1): until they are published it stores every token's
        // hidden row, and phase 2 scatters the kept ones.  Warp-uniform check.
        int seen = 0;
        if (lane == 0) {
          seen = ld_acquire(route_done) != 0 ? 1 : 0;
          if (seen) *s_routed = 1;  // for the warps that wait on this CTA's copy
        }
        seen = __shfl_sync(0xffffffffu, seen, 0);
        if (seen) {
          (void)ld_acquire(route_done);  // every lane's reads follow the publication
          routed = true;
        }
      } else if (!routed) {
        if (!tables_ready()) break;
        routed = true;
      }
      // the grouped row of this token's kept assignment to e (-1: none or dropped);
      // with the tables, phase 1 stores only the hidden rows phase 2 will scatter
      long long dest = -1;
      bool keep = false;  // phase 1: this token's hidden row is stored
      if (t < g.T) {
        if (routed) {
          for (int r = 0; r < g.k; ++r) {
            const long long a = static_cast<long long>(t) * g.k + r;
            if (__ldcg(g.idx + a) == e) {
              const int ps = __ldcg(g.pos + a);
              if (ps >= 0) dest = static_cast<long long>(__ldcg(g.offsets + e)) + ps;
            }
          }
          if (dest >= g.rows) {
            record_error(g.err, MOE_ERR_BOUNDS);
            dest = -1;
          }
          keep = dest >= 0;
        } else {
          keep = true;
        }
      }
      if (!mbar_wait_bounded(smem_u32(&tfull[acc]), aphase, g.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + static_cast<uint32_t>(acc * ACC_COLS);
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
      };
      if (p1 && g.swiglu) {
        // 4 chunks of 32 h columns (gate at TMEM column c*32, up at 128 + c*32); two per warp
        __nv_bfloat16* hrow = g.h + (static_cast<long long>(e) * BM + t) * g.F;
#pragma unroll 1
        for (int c = half * 2; c < half * 2 + 2; ++c) {
          uint32_t gr[32], ur[32];
          tmem_ld32_issue(tbase + c * 32, gr);
          tmem_ld32_issue(tbase + 128 + c * 32, ur);
          tmem_wait_ld(gr, ur);
          if (c == half * 2 + 1) release();
          const int col = nb * 128 + c * 32;
          if (col < g.F && keep) {
            uint4 pk[4];
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              h2[i] = __floats2bfloat162_rn(silu_f(__uint_as_float(gr[2 * i])) * __uint_as_float(ur[2 * i]),
                                            silu_f(__uint_as_float(gr[2 * i + 1])) * __uint_as_float(ur[2 * i + 1]));
            uint4* dst = reinterpret_cast<uint4*>(hrow + col);
            st_global_32b(dst, pk[0], pk[1]);
            st_global_32b(dst + 2, pk[2], pk[3]);
          }
        }
      } else {
        // 8 chunks of 32 columns, four per warp, two in flight per wait
#pragma unroll 1
        for (int c = half * 4; c < half * 4 + 4; c += 2) {
          uint32_t r0[32], r1[32];
          tmem_ld32_issue(tbase + c * 32, r0);
          tmem_ld32_issue(tbase + (c + 1) * 32, r1);
          tmem_wait_ld(r0, r1);
          if (c + 2 >= half * 4 + 4) release();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t* v = j == 0 ? r0 : r1;
            const int col = nb * BN + (c + j) * 32;
            if (p1) {
              // GELU: h = gelu(a + b1)
              if (col < g.F && keep) {
                const float* bias = g.b1 ? g.b1 + static_cast<long long>(e) * g.F + col : nullptr;
                uint4 pk[4];
                __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  float a0 = __uint_as_float(v[2 * i]), a1 = __uint_as_float(v[2 * i + 1]);
                  if (bias) { a0 += bias[2 * i]; a1 += bias[2 * i + 1]; }
                  h2[i] = __floats2bfloat162_rn(gelu_f(a0), gelu_f(a1));
                }
                uint4* dst = reinterpret_cast<uint4*>(g.h + (static_cast<long long>(e) * BM + t) * g.F + col);
                st_global_32b(dst, pk[0], pk[1]);
                st_global_32b(dst + 2, pk[2], pk[3]);
              }
            } else if (dest >= 0 && col < g.d) {
              // down projection: y = a + b2, scattered to the assignment's grouped row
              const float* bias = g.b2 ? g.b2 + static_cast<long long>(e) * g.d + col : nullptr;
              uint4 o[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float4 f = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                       __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                if (bias) { f.x += bias[4 * i]; f.y += bias[4 * i + 1]; f.z += bias[4 * i + 2]; f.w += bias[4 * i + 3]; }
                o[i] = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
              }
              uint4* dst = reinterpret_cast<uint4*>(g.y + dest * g.d + col);
#pragma unroll
              for (int i = 0; i < 4; ++i) st_global_32b(dst + 2 * i, o[2 * i], o[2 * i + 1]);
            }
          }
        }
      }
      // this warp's rows of the tile are stored: count it, for expert e (its
      // phase-2 tiles read these hidden rows through TMA once the count is
      // complete) or for the column block (its combine tile reads these rows)
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(p1 ? done1 + e : done2 + nb, 1);
      if (++acc == NACC) { acc = 0; aphase ^= 1u; }
    }
  }

  tc_fence_before();
  // the routing tables are complete before this grid is (the combine after
  // it relies on that), whatever tiles this CTA took
  pdl_wait();
  __syncthreads();
  if (tid == 0) {
    // the last CTA to get here clears the ticket and counts for the next call
    __threadfence();
    if (atomicAdd(finished, 1) == static_cast<int>(gridDim.x) - 1) {
      *ticket = 0;
      for (int e = 0; e < E + g.n2 + 2; ++e) done1[e] = 0;  // and done2, ranked, route_done, which follow
      __threadfence();
      *finished = 0;
      __threadfence();
    }
    pdl_trigger();
  }
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
      g_encode_err = e != cudaSuccess ? e : cudaErrorSymbolNotFound;
      return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode_err;
}

// bf16 [rows, K] (K contiguous) read in boxes of box_rows x 64, 128-byte swizzle
cudaError_t make_map(CUtensorMap* m, const void* base, long long rows, int K, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool ffn_decode_applies(const moe_shape_t& s) {
  // every expert's rows fit one 128-row tile, and enough assignments that
  // (nearly) every expert is expected to be active: the dense phase 1 then
  // streams no weights the grouped GEMMs would not
  return s.dtype == MOE_BF16 && s.routing == MOE_ROUTE_TOKEN_CHOICE && s.T >= 1 && s.T <= BM &&
         s.T * static_cast<long long>(s.k) >= 4LL * s.E && s.d % 64 == 0 && s.d_ff % 64 == 0;
}

bool ffn_decode_routes(const moe_shape_t& s, const float* W_g, const float* W_n) {
  const int nc = W_n != nullptr ? 2 * s.E : s.E;
  auto aligned = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
  // rank tiles: thread (cq, ks) with cq < nc / 4 dividing the 256 epilogue threads
  return ffn_decode_applies(s) && s.overflow == MOE_OVERFLOW_DROP && s.E <= RSLOTS * 32 && nc >= 4 && nc <= 256 &&
         (nc & (nc - 1)) == 0 && s.E % 4 == 0 && W_g != nullptr && aligned(W_g) && (W_n == nullptr || aligned(W_n)) &&
         s.d % 8 == 0 && s.T * static_cast<long long>(s.k) <= kMaxAssign &&
         dispatch_words(static_cast<int>(s.T * s.k), s.E) <= ROUTE_SMEM_WORDS;
}

size_t ffn_decode_h_bytes(const moe_shape_t& s) { return static_cast<size_t>(s.E) * BM * s.d_ff * 2; }
size_t ffn_decode_ctrl_bytes(const moe_shape_t& s) {
  return sizeof(int) * (4 + static_cast<size_t>(s.E) + static_cast<size_t>((s.d + BN - 1) / BN));
}

cudaError_t launch_ffn_decode(const DecodeFfnParams& p, cudaStream_t st) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const bool swiglu = p.act == MOE_ACT_SWIGLU;
  CUtensorMap mX, mW1, mW3, mH, mW2;
  if ((e = make_map(&mX, p.x, p.T, p.d, BM)) != cudaSuccess) return e;
  if ((e = make_map(&mW1, p.W1, static_cast<long long>(p.E) * p.F, p.d, swiglu ? BN / 2 : BN)) != cudaSuccess) return e;
  if (swiglu) {
    if ((e = make_map(&mW3, p.W3, static_cast<long long>(p.E) * p.F, p.d, BN / 2)) != cudaSuccess) return e;
  } else {
    mW3 = mW1;
  }
  if ((e = make_map(&mH, p.h, static_cast<long long>(p.E) * BM, p.F, BM)) != cudaSuccess) return e;
  if ((e = make_map(&mW2, p.W2, static_cast<long long>(p.E) * p.d, p.F, BN)) != cudaSuccess) return e;
  DecodeArgs g{};
  g.T = p.T;
  g.d = p.d;
  g.F = p.F;
  g.E = p.E;
  g.k = p.k;
  g.swiglu = swiglu ? 1 : 0;
  g.n1 = swiglu ? (p.F + 127) / 128 : (p.F + BN - 1) / BN;
  g.n2 = (p.d + BN - 1) / BN;
  g.kb1 = p.d / BK;
  g.kb2 = p.F / BK;
  g.b1 = p.b1;
  g.b2 = p.b2;
  g.h = static_cast<__nv_bfloat16*>(p.h);
  g.idx = p.idx;
  g.pos = p.pos;
  g.offsets = p.offsets;
  g.y = p.y_perm;
  g.rows = p.rows;
  g.ctrl = p.ctrl;
  g.err = p.err;
  g.W1 = static_cast<const __nv_bfloat16*>(p.W1);
  g.W3 = static_cast<const __nv_bfloat16*>(p.W3);
  g.W2 = static_cast<const __nv_bfloat16*>(p.W2);
  g.x_res = static_cast<const __nv_bfloat16*>(p.x);
  g.w = p.w;
  g.y_shared = p.y_shared;
  g.out = static_cast<__nv_bfloat16*>(p.out);
  g.moe_out = p.moe_out;
  const bool route = p.self_route != 0;
  if (route) {
    g.nrank = (p.T + RTOK - 1) / RTOK;
    g.C = p.C;
    g.counts = p.counts;
    g.dropped = p.dropped;
    g.row_of = p.row_of;
    RouterParams& rp = g.rp;
    rp.x = p.x;
    rp.W_g = p.W_g;
    rp.b_g = p.b_g;
    rp.W_n = p.W_n;
    rp.eps = p.eps;
    rp.T = p.T;
    rp.d = p.d;
    rp.E = p.E;
    rp.k = p.k;
    rp.idx = p.idx;
    rp.w = p.w;
    rp.logits = p.logits;
    rp.gate_raw = p.gate_raw;
    rp.stats = p.stats;
    rp.err = p.err;
  }
  auto kern = route ? ffn_decode_kernel<true> : ffn_decode_kernel<false>;
  const int smem = SMEM_BYTES + (route ? ROUTE_SMEM_BYTES : 0);
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(p.E) * (g.n1 + g.n2) +
                          static_cast<long long>(g.n2) * ((p.T + 15) / 16) + (route ? g.nrank + 1 : 0);
  const int grid = static_cast<int>(std::min<long long>(sms, tiles));
  // the first-tile L2 prefetch: at most kPrefetchBudget bytes over all CTAs
  // (well inside L2), a multiple of 128 bytes of every row of the tile's panel
  constexpr long long kPrefetchBudget = 80LL << 20;
  const long long tile_rows = swiglu ? 256 : BN;
  const long long per_row = kPrefetchBudget / grid / tile_rows;
  g.pf_bytes_row = static_cast<int>(std::min<long long>(static_cast<long long>(std::min(p.d, p.F)) * 2, per_row) / 128 * 128);
  NvtxRange r("expert_ffn_decode");
  return launch_pdl(kern, dim3(grid), dim3(NTHREADS), static_cast<size_t>(smem), st, 1, mX, mW1, mW3, mH, mW2, g);
}

}  // namespace moe
