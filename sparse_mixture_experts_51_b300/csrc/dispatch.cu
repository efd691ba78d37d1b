// Capacity-limited dispatch and the gather into expert order.
//
// Semantics ("Mixture-of-Experts Sparse Model Scaling", Lab 3 and Advanced
// Theory; "Mixture-of-experts Models", "Capacity limits make dispatch
// observable"): assignments are taken in priority order j = r*T + t (every
// token's first choice, in token order, before any second choice); an
// assignment gets the next slot of its expert while fewer than C slots are
// taken, and is dropped otherwise.  pos[t,r] = number of earlier assignments
// to the same expert, kept iff pos < C.
//
// Design.  One pass, deterministic, no atomics deciding any slot:
//   * each block takes a tile of 256 x ITEMS consecutive priority positions
//     (1024 for short batches, 4096 above 262144 assignments); a block
//     obtains its tile index from a ticket counter, so a block only ever
//     waits on blocks that are already running;
//   * all ITEMS expert ids of a thread are loaded at once; warps rank equal
//     experts with per-bit ballots + popc, the per-(step, warp, expert) counts go
//     to shared memory, and one per-expert exclusive scan over the
//     (step, warp) sequence orders every assignment of the tile;
//   * the per-expert tile totals are scanned across tiles with a decoupled
//     look-back over E-wide descriptors (aggregate / inclusive prefix): one
//     warp reads the flags of 32 predecessors at a time and sums their
//     aggregates up to the nearest inclusive prefix; every wait is bounded
//     and records MOE_ERR_DEVICE_TIMEOUT;
//   * the block holding the last tile turns the loads into counts, segment
//     offsets and the drop count;
//   * the last block to finish (a done counter) clears the ticket, the status
//     flags and the counter, so the next call finds them at zero without a
//     separate memset (the workspace is zero-filled once, at allocation).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int NT = kDispatchThreads;
constexpr int NWARP = NT / 32;

// Lanes of the warp holding the same value v in [0, 2^nbits): one ballot per
// bit, intersected (a constant-cost stand-in for match.any).
__device__ __forceinline__ unsigned same_value_lanes(int v, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (v >> b) & 1;
    const unsigned on = __ballot_sync(0xffffffffu, bit);
    m &= bit ? on : ~on;
  }
  return m;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// dynamic shared memory: s_hist [ITEMS][NWARP][E] ints
template <int ITEMS>
__global__ void __launch_bounds__(NT) dispatch_kernel(DispatchParams p) {
  extern __shared__ int s_hist[];
  __shared__ int s_tot[kMaxExperts];   // assignments to each expert inside this tile
  __shared__ int s_excl[kMaxExperts];  // assignments to each expert before this tile
  __shared__ int s_ticket;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  const long long total = static_cast<long long>(p.T) * p.k;

  if (p.early_trigger) pdl_trigger();
  pdl_wait();  // the top-k table is the predecessor's output
  if (tid == 0) s_ticket = atomicAdd(&p.ctrl[0], 1);
  for (int i = tid; i < ITEMS * NWARP * E; i += NT) s_hist[i] = 0;
  __syncthreads();
  const int b = s_ticket;
  int* status = p.ctrl + 1;
  const long long base = static_cast<long long>(b) * (NT * ITEMS);

  // ---- every expert id of this thread, loaded at once
  int my_e[ITEMS], my_rank[ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const long long j = base + static_cast<long long>(i) * NT + tid;
    int e = -1;
    if (j < total) {
      const int r = static_cast<int>(j / p.T);
      const int t = static_cast<int>(j - static_cast<long long>(r) * p.T);
      e = __ldg(p.idx + static_cast<long long>(t) * p.k + r);
    }
    my_e[i] = e;
  }
  // ---- rank inside the warp step; per-(step, warp, expert) counts
  const unsigned lt_mask = (1u << lane) - 1u;
  const int nbits = 32 - __clz(E);  // expert ids + 1 lie in [0, E] < 2^nbits
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    int e = my_e[i];
    const long long j = base + static_cast<long long>(i) * NT + tid;
    if (j < total && (e < 0 || e >= E)) {  // an expert id out of range takes no slot
      if (!(p.allow_skip && e == -1)) record_error(p.err, MOE_ERR_BOUNDS);
      e = -1;
    }
    my_e[i] = e;
    const unsigned peers = same_value_lanes(e + 1, nbits);
    my_rank[i] = __popc(peers & lt_mask);
    if (e >= 0 && my_rank[i] == 0) s_hist[(i * NWARP + warp) * E + e] = __popc(peers);
  }
  __syncthreads();
  // ---- per expert: exclusive scan over the (step, warp) sequence, in priority order
  for (int ex = tid; ex < E; ex += NT) {
    int run = 0;
    for (int sw = 0; sw < ITEMS * NWARP; ++sw) {
      const int c = s_hist[sw * E + ex];
      s_hist[sw * E + ex] = run;
      run += c;
    }
    s_tot[ex] = run;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < ITEMS; ++i)
    if (my_e[i] >= 0) my_rank[i] += s_hist[(i * NWARP + warp) * E + my_e[i]];

  // ---- publish this tile's per-expert totals, then look back for the prefix
  int* agg = p.agg + static_cast<long long>(b) * E;
  int* incl = p.incl + static_cast<long long>(b) * E;
  for (int ex = tid; ex < E; ex += NT) {
    __stcg(&agg[ex], s_tot[ex]);
    if (b == 0) __stcg(&incl[ex], s_tot[ex]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0 && b != p.stall_block) st_release(&status[b], b == 0 ? 2 : 1);

  if (warp == 0) {
    constexpr int SL = kMaxExperts / 32;
    int ex_acc[SL];
#pragma unroll
    for (int s = 0; s < SL; ++s) ex_acc[s] = 0;
    int pred = b - 1;
    bool timed_out = false;
    const unsigned long long t0 = globaltimer_ns();
    while (pred >= 0) {
      // flags of the 32 predecessors pred, pred-1, ..., pred-31 (lane i: tile pred-i)
      const int tile = pred - lane;
      int f = 0, first_incl = 32;
      unsigned spins = 0;
      while (true) {
        f = tile >= 0 ? ld_acquire(&status[tile]) : -1;
        const unsigned incl_mask = __ballot_sync(0xffffffffu, f == 2);
        const unsigned zero_mask = __ballot_sync(0xffffffffu, f == 0);
        first_incl = incl_mask ? __ffs(incl_mask) - 1 : 32;
        // usable once every tile up to the nearest inclusive prefix has published
        const unsigned need = first_incl >= 31 ? 0xffffffffu : ((2u << first_incl) - 1u);
        if ((zero_mask & need) == 0) break;
        if ((++spins & 15u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
          timed_out = true;
          break;
        }
      }
      if (timed_out) break;
      __threadfence();
      // aggregates of the tiles before the inclusive one, then its inclusive prefix
      const int n_agg = min(first_incl, pred + 1);
#pragma unroll
      for (int s = 0; s < SL; ++s) {
        const int ex = lane + 32 * s;
        if (ex < E) {
          int sum = 0;
          for (int i2 = 0; i2 < n_agg; ++i2) sum += __ldcg(&p.agg[static_cast<long long>(pred - i2) * E + ex]);
          if (first_incl < 32) sum += __ldcg(&p.incl[static_cast<long long>(pred - first_incl) * E + ex]);
          ex_acc[s] += sum;
        }
      }
      if (first_incl < 32) break;
      pred -= 32;
    }
    if (timed_out && lane == 0) record_error(p.err, MOE_ERR_DEVICE_TIMEOUT);
#pragma unroll
    for (int s = 0; s < SL; ++s) {
      const int ex = lane + 32 * s;
      if (ex < E) {
        s_excl[ex] = ex_acc[s];
        if (b > 0) __stcg(&incl[ex], ex_acc[s] + s_tot[ex]);
      }
    }
    __threadfence();
    __syncwarp();
    if (b > 0 && lane == 0 && b != p.stall_block) st_release(&status[b], 2);
  }
  __syncthreads();

  // ---- slots: earlier tiles + rank inside this tile; kept iff below capacity
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const long long j = base + static_cast<long long>(i) * NT + tid;
    if (j < total) {
      const int r = static_cast<int>(j / p.T);
      const int t = static_cast<int>(j - static_cast<long long>(r) * p.T);
      int ps = -1;
      if (my_e[i] >= 0) {
        const int slot = (p.base ? __ldg(p.base + my_e[i]) : 0) + s_excl[my_e[i]] + my_rank[i];
        ps = slot < p.C ? slot : -1;
      }
      p.pos[static_cast<long long>(t) * p.k + r] = ps;
    }
  }

  // ---- the last tile knows every expert's load
  if (b == p.nblk - 1) {
    __shared__ int s_counts[kMaxExperts];
    __shared__ unsigned long long s_drop[NWARP];
    unsigned long long drop = 0;
    for (int ex = tid; ex < kMaxExperts; ex += NT) {
      int c = 0;
      if (ex < E) {
        const int load = (p.base ? __ldg(p.base + ex) : 0) + s_excl[ex] + s_tot[ex];
        c = load < p.C ? load : p.C;
        drop += static_cast<unsigned long long>(load - c);
        p.counts[ex] = c;
      }
      s_counts[ex] = c;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) drop += __shfl_xor_sync(0xffffffffu, drop, o);
    if (lane == 0) s_drop[warp] = drop;
    __syncthreads();
    if (warp == 0) {
      // exclusive scan of counts over E <= 128 experts, 4 per lane
      int v[4], run = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[q] = s_counts[lane * 4 + q];
        run += v[q];
      }
      int incl_sum = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl_sum, o);
        if (lane >= o) incl_sum += n;
      }
      int off = incl_sum - run;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ex = lane * 4 + q;
        if (ex < E) p.offsets[ex] = off;
        off += v[q];
      }
      if (lane == 31) p.offsets[E] = incl_sum;
      if (lane == 0) {
        unsigned long long dsum = 0;
        for (int w2 = 0; w2 < NWARP; ++w2) dsum += s_drop[w2];
        *p.dropped = static_cast<long long>(dsum);
      }
    }
  }

  // ---- every block is past its look-back: the last one to get here clears
  // the control words for the next call
  pdl_trigger();
  __syncthreads();
  if (tid == 0) {
    int* done = p.ctrl + 1 + p.nblk;
    __threadfence();
    if (atomicAdd(done, 1) == p.nblk - 1) {
      for (int i = 0; i < p.nblk; ++i) status[i] = 0;
      p.ctrl[0] = 0;
      *done = 0;
      __threadfence();
    }
  }
}

// Single-CTA dispatch, for batches whose per-(step, warp, expert) histogram
// fits in shared memory: 1024 threads take ITEMS assignments each (thread
// tid, step i: priority position i*1024 + tid), rank equal experts within
// each warp step with per-bit ballots, and one exclusive scan per expert over the
// (step, warp) sequence -- a warp per expert, ITEMS entries per lane -- gives
// every assignment its slot.  No inter-block scan, no atomics, no control
// words; the same results as the tiled kernel.
constexpr int SNT = 1024;
constexpr int SNW = SNT / 32;

template <int ITEMS>
__global__ void __launch_bounds__(SNT, 1) dispatch_single_kernel(DispatchParams p) {
  extern __shared__ int s_hist[];  // [ITEMS * SNW][E]: counts, then exclusive prefixes
  __shared__ int s_tot[kMaxExperts];
  __shared__ unsigned long long s_drop[SNW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  const int total = p.T * p.k;  // < 2^31 (checked on the host)
  constexpr int S = ITEMS * SNW;  // (step, warp) entries per expert

  for (int i = tid; i < S * E; i += SNT) s_hist[i] = 0;
  if (p.early_trigger) pdl_trigger();
  pdl_wait();  // the top-k table is the predecessor's output
  // per item: expert + 1 in bits 0-7 (0: none), rank inside the warp step in bits 8-12
  int my_er[ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int j = i * SNT + tid;
    int e = -1;
    if (j < total) {
      const int r = j / p.T;
      const int t = j - r * p.T;
      e = __ldg(p.idx + t * p.k + r);
      if (e < 0 || e >= E) {  // an expert id out of range takes no slot
        if (!(p.allow_skip && e == -1)) record_error(p.err, MOE_ERR_BOUNDS);
        e = -1;
      }
    }
    my_er[i] = e + 1;
  }
  __syncthreads();  // the histogram is zero
  const unsigned lt_mask = (1u << lane) - 1u;
  const int nbits = 32 - __clz(E);  // expert ids + 1 lie in [0, E] < 2^nbits
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int e = my_er[i] - 1;
    const unsigned peers = same_value_lanes(my_er[i], nbits);
    const int rk = __popc(peers & lt_mask);
    my_er[i] |= rk << 8;
    if (e >= 0 && rk == 0) s_hist[(i * SNW + warp) * E + e] = __popc(peers);
  }
  __syncthreads();
  // ---- per expert: exclusive scan over the (step, warp) sequence (priority order)
  for (int ex = warp; ex < E; ex += SNW) {
    int run = 0;
    for (int q = 0; q < ITEMS; ++q) run += s_hist[(lane * ITEMS + q) * E + ex];
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int off = incl - run;
    for (int q = 0; q < ITEMS; ++q) {
      const int c = s_hist[(lane * ITEMS + q) * E + ex];
      s_hist[(lane * ITEMS + q) * E + ex] = off;
      off += c;
    }
    if (lane == 31) s_tot[ex] = incl;
  }
  __syncthreads();
  // ---- slots; kept iff below capacity
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int j = i * SNT + tid;
    if (j < total) {
      const int r = j / p.T;
      const int t = j - r * p.T;
      int ps = -1;
      const int e = (my_er[i] & 0xff) - 1;
      if (e >= 0) {
        const int slot = (p.base ? __ldg(p.base + e) : 0) + s_hist[(i * SNW + warp) * E + e] + (my_er[i] >> 8);
        ps = slot < p.C ? slot : -1;
      }
      p.pos[t * p.k + r] = ps;
    }
  }
  // ---- counts, segment offsets, drop count
  unsigned long long drop = 0;
  for (int ex = tid; ex < E; ex += SNT) {
    const int load = (p.base ? __ldg(p.base + ex) : 0) + s_tot[ex];
    const int c = load < p.C ? load : p.C;
    drop += static_cast<unsigned long long>(load - c);
    p.counts[ex] = c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) drop += __shfl_xor_sync(0xffffffffu, drop, o);
  if (lane == 0) s_drop[warp] = drop;
  __syncthreads();
  if (warp == 0) {
    int v[4], run = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ex = lane * 4 + q;
      v[q] = ex < E ? min((p.base ? __ldg(p.base + ex) : 0) + s_tot[ex], p.C) : 0;
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
      if (ex < E) p.offsets[ex] = off;
      off += v[q];
    }
    if (lane == 31) p.offsets[E] = incl;
    if (lane == 0) {
      unsigned long long dsum = 0;
      for (int w2 = 0; w2 < SNW; ++w2) dsum += s_drop[w2];
      *p.dropped = static_cast<long long>(dsum);
    }
  }
  pdl_trigger();
}

// Overflow re-routing, requests: the first dropped assignment (lowest rank)
// of each token asks for the token's backup expert; everything else asks
// for nothing (-1).  A thread per token.
__global__ void __launch_bounds__(256) reroute_requests_kernel(RerouteParams p) {
  pdl_wait();
  pdl_trigger();
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= p.T) return;
  bool asked = false;
  const int b = __ldg(p.backup + t);
  for (int r = 0; r < p.k; ++r) {
    const long long a = t * p.k + r;
    const bool ask = !asked && b >= 0 && p.pos[a] < 0;
    p.req[a] = ask ? b : -1;
    asked |= p.pos[a] < 0;
  }
}

// Merge of the second pass: a request that got a slot moves its assignment
// to the backup; the assignments still without a slot are counted.
__global__ void __launch_bounds__(256) reroute_merge_kernel(RerouteParams p) {
  __shared__ int s_cnt;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const long long a = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool lost = false;
  if (a < static_cast<long long>(p.T) * p.k) {
    int ps = p.pos[a];
    const int q = __ldg(p.pos2 + a);
    if (ps < 0 && p.req[a] >= 0 && q >= 0) {
      p.idx[a] = p.req[a];
      p.pos[a] = q;
      ps = q;
    }
    lost = ps < 0;
  }
  const unsigned m = __ballot_sync(0xffffffffu, lost);
  if ((threadIdx.x & 31) == 0 && m) atomicAdd(&s_cnt, __popc(m));
  __syncthreads();
  if (threadIdx.x == 0 && s_cnt)
    atomicAdd(reinterpret_cast<unsigned long long*>(p.dropped), static_cast<unsigned long long>(s_cnt));
}

// One warp per assignment (t, r): copy token t into its expert-ordered row.
template <int VB>
__global__ void __launch_bounds__(256) gather_kernel(GatherParams p, long long rows_alloc) {
  pdl_wait();
  pdl_trigger();
  const long long a = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long total = static_cast<long long>(p.T) * p.k;
  if (a >= total) return;
  const int ps = p.pos[a];
  const int e = ps >= 0 ? p.idx[a] : -1;
  long long row = -1;
  if (ps >= 0) {
    if (e >= 0 && e < p.E) row = static_cast<long long>(p.offsets[e]) + ps;
    if (row < 0 || row >= rows_alloc) {
      if (lane == 0) record_error(p.err, MOE_ERR_BOUNDS);
      row = -1;
    }
  }
  if (lane == 0 && p.row_of) p.row_of[a] = static_cast<int32_t>(row);
  if (row < 0) return;
  const long long t = a / p.k;
  const long long row_bytes = static_cast<long long>(p.d) * p.elem_bytes;
  const char* src = static_cast<const char*>(p.x) + t * row_bytes;
  char* dst = static_cast<char*>(p.x_perm) + row * row_bytes;
  if constexpr (VB == 16) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const long long n = row_bytes / 16;
    for (long long i = lane; i < n; i += 32) d4[i] = __ldg(&s4[i]);
  } else {
    const long long n = row_bytes / 4;
    const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
    uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
    for (long long i = lane; i < n; i += 32) d1[i] = __ldg(&s1[i]);
  }
  if (lane == 0 && p.row_token) p.row_token[row] = static_cast<int32_t>(t);
}

}  // namespace

namespace {
template <int ITEMS>
cudaError_t launch_single(const DispatchParams& p, cudaStream_t st) {
  const size_t smem = sizeof(int) * static_cast<size_t>(ITEMS) * SNW * p.E;
  cudaError_t e = cudaFuncSetAttribute(dispatch_single_kernel<ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(dispatch_single_kernel<ITEMS>, dim3(1), dim3(SNT), smem, st, 1, p);
}
}  // namespace

cudaError_t launch_dispatch(const DispatchParams& p, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  const long long Tk = static_cast<long long>(p.T) * p.k;
  // one CTA for up to 2048 assignments when its histogram (items per thread
  // x 32 warps x E ints) fits in 96 KB; measured on B300 it wins at 768
  // assignments (1.5 us) and loses to the tiled kernel at 8192 (2.5 us)
  int items = 1;
  while (static_cast<long long>(items) * SNT < Tk) items <<= 1;
  // (the testing hook that stalls a tile needs the tiled kernel)
  if (p.stall_block < 0 && items <= 2 && static_cast<long long>(items) * SNW * p.E * 4 <= 96 * 1024) {
    return items == 1 ? launch_single<1>(p, st) : launch_single<2>(p, st);
  }
  if (p.clear_ctrl && (e = cudaMemsetAsync(p.ctrl, 0, sizeof(int) * (2 + p.nblk), st)) != cudaSuccess) return e;
  if (dispatch_items(Tk) == kDispatchItemsSmall) {
    const size_t smem = sizeof(int) * kDispatchItemsSmall * NWARP * p.E;
    e = launch_pdl(dispatch_kernel<kDispatchItemsSmall>, dim3(p.nblk), dim3(NT), smem, st, 1, p);
  } else {
    const size_t smem = sizeof(int) * kDispatchItemsLarge * NWARP * p.E;
    e = cudaFuncSetAttribute(dispatch_kernel<kDispatchItemsLarge>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(dispatch_kernel<kDispatchItemsLarge>, dim3(p.nblk), dim3(NT), smem, st, 1, p);
  }
  return e;
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t st) {
  const long long total = static_cast<long long>(p.T) * p.k;
  if (total == 0) return cudaSuccess;
  const long long blocks = (total * 32 + 255) / 256;
  const long long row_bytes = static_cast<long long>(p.d) * p.elem_bytes;
  const bool vec16 = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(p.x) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(p.x_perm) % 16 == 0;
  if (vec16) return launch_pdl(gather_kernel<16>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p, p.rows_alloc);
  return launch_pdl(gather_kernel<4>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p, p.rows_alloc);
}

cudaError_t launch_reroute_requests(const RerouteParams& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  return launch_pdl(reroute_requests_kernel, dim3(static_cast<unsigned>((p.T + 255) / 256)), dim3(256), 0, st, 1, p);
}

cudaError_t launch_reroute_merge(const RerouteParams& p, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(p.dropped, 0, sizeof(long long), st);
  if (e != cudaSuccess || p.T == 0) return e;
  const long long n = static_cast<long long>(p.T) * p.k;
  return launch_pdl(reroute_merge_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st, 1, p);
}

}  // namespace moe
