// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Each expert e owns the rows [offsets[e], offsets[e+1]) of the expert-grouped
// activations (a dense FFN, such as the shared experts, is one group holding
// every row) and computes, in nn.Linear layout (K contiguous for A and B):
//   GELU   : h = gelu(A W1[e]^T + b1[e])                 -> bf16 [rows, F]
//   SwiGLU : h = silu(A W1[e]^T) * (A W3[e]^T)           -> bf16 [rows, F]
//   down   : y = h W2[e]^T + b2[e]                       -> fp32 [rows, d]
// (the expert FFN of "Mixture-of-Experts Sparse Model Scaling", Core
// Concepts: each expert is the dense FFN it replaces).
//
// Kernel design (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer: 128x64 (or 256x64) A tile + 256x64 B tile per
//               stage, 128-byte swizzle, mbarrier ring of 4 x 48 KB (3 x 64 KB)
//   warp 1      MMA issuer: one thread issues tcgen05.mma M=128 N=256 K=16
//               (per M tile), fp32 accumulator in TMEM; tcgen05.commit frees
//               smem stages
//   warp 2      TMEM allocator (512 columns = two 128x256 fp32 accumulators)
//   warps 4-11  epilogue: two warps per TMEM lane quarter (128-row tiles:
//               half of the 32-column chunks each; 256-row tiles: one M tile
//               each): tcgen05.ld, fused activation, bias, conversion; a
//               warp whose rows all lie in the segment stages 128-byte boxes
//               in shared memory and writes them with TMA stores, the warp
//               at a segment's end stores its valid rows with 32-byte stores
// SwiGLU puts 128 rows of W1 and the matching 128 rows of W3 into one
// 256-row B tile, so one accumulator holds gate | up and the epilogue emits
// 128 columns of h.  Tiles are ordered expert-major, then N, then M, so CTAs
// running side by side share weight panels in L2.  Every barrier wait is
// bounded; on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT, drains its own
// copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int B_BYTES = BN * BK * 2;
constexpr int TMEM_COLS = 512;
constexpr int NTHREADS = 384;
constexpr int EPI_WARPS = 8;  // warps 4-11, two per TMEM lane quarter

// MT = M tiles of 128 rows per CTA tile.  MT = 1: 128x256 tiles, 4 stages of
// 48 KB, two TMEM accumulators (the epilogue of one tile overlaps the next
// tile's mainloop).  MT = 2: 256x256 tiles that share each B stage between
// two M tiles (a third less L2->SM traffic per flop), 3 stages of 64 KB, one
// accumulator pair filling TMEM (the epilogue is not overlapped).
template <int MT>
struct Cfg {
  static constexpr int STAGES = MT == 1 ? 4 : 3;
  static constexpr int A_BYTES = MT * BM * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NACC = MT == 1 ? 2 : 1;  // accumulator buffers
  static constexpr int ACC_COLS = 256 * MT;     // TMEM columns per buffer
  static constexpr int TILE_M = BM * MT;
  static constexpr int STAGING_BYTES = EPI_WARPS * 4096;  // epilogue output boxes, 4 KB per warp
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 256 /*barriers*/ +
                                    (2 * kMaxExperts + 1) * 4 /*tile tables*/;
};

enum { MODE_GELU = 0, MODE_SWIGLU = 1, MODE_DOWN = 2 };

struct GemmArgs {
  const int32_t* offsets;  // [E+1] segment starts; null: one dense group of dense_rows rows
  int dense_rows;
  int a_kwrap;             // > 0: k-block kb of A is read at k-block kb mod a_kwrap (A reused along K)
  int E;
  int N_out;      // output columns
  int N_w;        // weight rows per expert in the B tensor
  int K;          // reduction length (multiple of 64)
  int n_tiles;    // N tiles per expert
  void* out;      // bf16 h or fp32 y
  long long out_ld;
  long long out_rows;  // allocated rows of out
  const float* bias;  // [E, N_out] or null
  int* err;
};

__device__ __forceinline__ float gelu_f(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }
// silu(a) = a * sigmoid(a) = a * (1 + tanh(a/2)) / 2, with the hardware
// tanh approximation (tanh.approx.f32, relative error about 2^-11): one
// special-function op per element instead of an exponential and a
// reciprocal, and the result is rounded to bf16 (2^-8) right after.
__device__ __forceinline__ float tanh_approx(float v) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float silu_f(float a) {
  const float h = 0.5f * a;
  return fmaf(h, tanh_approx(h), h);
}

struct TileInfo {
  int e, row0, rows_valid, n0;
};

// One 32-byte global store (a whole sector): each epilogue lane owns one row
// of the tile, so 16-byte stores would fill only half of every sector they
// touch.  The address must be 32-byte aligned.
__device__ __forceinline__ void st_global_32b(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w),
               "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

template <int MODE, int MT>
__global__ void __launch_bounds__(NTHREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmOut,
                        GemmArgs g) {
  using C = Cfg<MT>;
  constexpr int STAGES = C::STAGES, A_BYTES = C::A_BYTES, STAGE_BYTES = C::STAGE_BYTES, NACC = C::NACC;
  constexpr int BN_OUT = MODE == MODE_SWIGLU ? 128 : 256;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte align the tile ring (128-byte swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* staging = smem + STAGES * STAGE_BYTES;  // [EPI_WARPS][4 KB], 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STAGING_BYTES);
  uint64_t* full = bars;                 // [STAGES]
  uint64_t* empty = bars + STAGES;       // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;   // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* drain = tempty + 2;          // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_total = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_tstart = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + 256);  // [E+1]
  int* s_mt = s_tstart + kMaxExperts + 1;                                        // [E]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = g.E;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), EPI_WARPS);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (MODE == MODE_SWIGLU) tma_prefetch_desc(&tmB3);
  }
  // the prologue above overlaps the predecessor's tail; its outputs (the
  // grouped rows and their segment offsets) are read only from here on
  pdl_wait();
  auto seg = [&](int e) -> int { return g.offsets ? g.offsets[e] : (e == 0 ? 0 : g.dense_rows); };
  // ---- per-expert tile counts from the segment offsets
  for (int e = tid; e < E; e += NTHREADS) {
    const int cnt = seg(e + 1) - seg(e);
    s_mt[e] = cnt > 0 ? (cnt + C::TILE_M - 1) / C::TILE_M : 0;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_tstart[e] = acc;
      acc += s_mt[e] * g.n_tiles;
    }
    s_tstart[E] = acc;
    *s_total = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = *s_total;
  const int KB = g.K / BK;

  auto decode = [&](int tile, int& ecur, TileInfo& ti) {
    while (s_tstart[ecur + 1] <= tile) ++ecur;
    const int local = tile - s_tstart[ecur];
    const int mt = s_mt[ecur];
    const int nb = local / mt, mb = local - nb * mt;
    const int seg0 = seg(ecur);
    const int cnt = seg(ecur + 1) - seg0;
    ti.e = ecur;
    ti.row0 = seg0 + mb * C::TILE_M;
    ti.rows_valid = min(C::TILE_M, cnt - mb * C::TILE_M);
    ti.n0 = nb * BN_OUT;
  };

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_phase = 0;  // per-stage bit masks, for the drain
      int ecur = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        TileInfo ti;
        decode(tile, ecur, ti);
        const int brow = ti.e * g.N_w + ti.n0;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, g.err, abort_flag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = smem_u32(tiles + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          tma_load_2d(sa, &tmA, fb, (g.a_kwrap > 0 ? kb % g.a_kwrap : kb) * BK, ti.row0);
          if (MODE == MODE_SWIGLU) {
            tma_load_2d(sb, &tmB, fb, kb * BK, brow);
            tma_load_2d(sb + B_BYTES / 2, &tmB3, fb, kb * BK, brow);
          } else {
            tma_load_2d(sb, &tmB, fb, kb * BK, brow);
          }
          issued |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // make sure no copy into this CTA's shared memory is still in flight
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
      bool ok = true;
      bool any = false;
      int ecur = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        // a 256-row tile holding at most 128 rows of its expert (the last,
        // partial tile of a segment) computes only its first M half
        TileInfo ti;
        decode(tile, ecur, ti);
        const int mt_used = (MT == 2 && ti.rows_valid <= BM) ? 1 : MT;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), aphase ^ 1u, g.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * C::ACC_COLS);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, g.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const uint64_t db = smem_desc_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m >= mt_used) break;
              // M tile m: rows 128m.. of the A stage (16 KB apart) into TMEM columns 256m..;
              // step 16 bf16 = 32 bytes along K inside the swizzled 128-byte rows
              const uint64_t da = smem_desc_sw128(sa + static_cast<uint32_t>(m * BM * BK * 2));
              umma_bf16(dt + static_cast<uint32_t>(m * 256), da + static_cast<uint64_t>(kk * 2),
                        db + static_cast<uint64_t>(kk * 2), IDESC, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(smem_u32(&empty[stage]));
          any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[acc]));
        if (++acc == NACC) { acc = 0; aphase ^= 1u; }
      }
      if (any) {
        // every MMA issued by this thread has finished before TMEM is freed
        umma_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, g.err, nullptr);
      }
    }
  } else if (warp >= 4) {
    // ================= epilogue =================
    // MT = 1: warps w and w+4 share lane quarter w & 3, each taking half of
    // the 32-column chunks; MT = 2: warps 4-7 drain M tile 0, warps 8-11 M
    // tile 1.  A warp whose 32 rows all lie in the segment stages its rows
    // in shared memory as 32 x 128-byte boxes (two bf16 chunks or one fp32
    // chunk) and writes each with one TMA store; a warp holding the segment's
    // end writes its valid rows directly (TMA would also write the rows past
    // the end, which belong to the next expert).
    constexpr int NCH = BN_OUT / 32;               // 32-column chunks per tile
    constexpr int WCH = MT == 2 ? NCH : NCH / 2;   // chunks per warp
    constexpr int BOX_CH = MODE == MODE_DOWN ? 1 : 2;
    const int q = warp & 3;                             // TMEM lane quarter this warp may access
    const int msel = MT == 2 ? (warp - 4) >> 2 : 0;     // M tile of the CTA tile
    const int cfirst = MT == 2 ? 0 : ((warp - 4) >> 2) * WCH;
    const int rloc = msel * BM + q * 32 + lane;         // row inside the tile
    // direct stores: whole 32-byte sectors when every row start is 32-byte
    // aligned (column offsets are multiples of 32 elements)
    constexpr int OUT_BYTES = MODE == MODE_DOWN ? 4 : 2;
    const bool st32 =
        ((reinterpret_cast<uintptr_t>(g.out) | static_cast<uintptr_t>(g.out_ld * OUT_BYTES)) & uintptr_t(31)) == 0;
    const uint32_t stg = smem_u32(staging + (warp - 4) * 4096);  // this warp's box, 1024-byte aligned
    int acc = 0;
    uint32_t aphase = 0;
    int ecur = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      TileInfo ti;
      decode(tile, ecur, ti);
      if (!mbar_wait_bounded(smem_u32(&tfull[acc]), aphase, g.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * C::ACC_COLS + msel * 256);
      const bool row_ok = rloc < ti.rows_valid;
      const long long row = static_cast<long long>(ti.row0) + rloc;
      // a warp whose 32 rows all lie past the segment reads nothing
      const bool warp_rows = __any_sync(0xffffffffu, row_ok);
      const bool warp_full = __all_sync(0xffffffffu, row_ok);
      // the accumulator is released as soon as this warp's last TMEM load
      // has completed: the math and stores of its last chunks overlap the
      // next tile's MMAs
      bool released = false;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        released = true;
      };
      // writes this lane's row of 32-column chunk c (NV 16-byte units)
      auto emit = [&](int c, const uint4* v, auto nv_tag) {
        constexpr int NV = decltype(nv_tag)::value;
        const int col = ti.n0 + c * 32;
        if (col >= g.N_out) return;
        if (warp_full) {
          const int half = BOX_CH == 2 ? ((c - cfirst) & 1) : 0;  // place of the chunk in its box
          if (half == 0) {
            // the previous box's store has finished reading the buffer
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
          }
          // 128-byte swizzle (16-byte unit u of row r at u ^ (r & 7), the
          // layout the tensor map undoes): the 8 lanes of a store phase hit
          // distinct banks
          const uint32_t rowp = stg + static_cast<uint32_t>(lane * 128);
#pragma unroll
          for (int i = 0; i < NV; ++i)
            st_shared_v4(rowp + static_cast<uint32_t>(((half * 4 + i) ^ (lane & 7)) << 4), v[i]);
          if (half == BOX_CH - 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, stg, col - half * 32, static_cast<int>(row - lane));
              bulk_commit_group();
            }
          }
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.out) +
                                                (row * g.out_ld + col) * OUT_BYTES);
          if (st32) {
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) st_global_32b(dst + 2 * i, v[2 * i], v[2 * i + 1]);
          } else {
#pragma unroll
            for (int i = 0; i < NV; ++i) dst[i] = v[i];
          }
        }
      };
      using NV4 = std::integral_constant<int, 4>;
      using NV8 = std::integral_constant<int, 8>;
      if (!warp_rows) {
      } else if constexpr (MODE == MODE_SWIGLU) {
#pragma unroll 1
        for (int c = cfirst; c < cfirst + WCH; ++c) {
          // gate and up columns in flight together, one wait
          uint32_t gr[32], ur[32];
          tmem_ld32_issue(tbase + c * 32, gr);
          tmem_ld32_issue(tbase + 128 + c * 32, ur);
          tmem_wait_ld(gr, ur);
          if (c == cfirst + WCH - 1) release();
          uint4 pk[4];
          __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            h2[i] = __floats2bfloat162_rn(silu_f(__uint_as_float(gr[2 * i])) * __uint_as_float(ur[2 * i]),
                                          silu_f(__uint_as_float(gr[2 * i + 1])) * __uint_as_float(ur[2 * i + 1]));
          emit(c, pk, NV4{});
        }
      } else {
        // two 32-column chunks in flight per wait
        auto store_chunk = [&](int c, const uint32_t (&v)[32]) {
          const int col = ti.n0 + c * 32;
          const float* bias = (g.bias && col < g.N_out) ? g.bias + static_cast<long long>(ti.e) * g.N_out + col
                                                        : nullptr;
          if constexpr (MODE == MODE_GELU) {
            uint4 pk[4];
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a0 = __uint_as_float(v[2 * i]), a1 = __uint_as_float(v[2 * i + 1]);
              if (bias) { a0 += bias[2 * i]; a1 += bias[2 * i + 1]; }
              h2[i] = __floats2bfloat162_rn(gelu_f(a0), gelu_f(a1));
            }
            emit(c, pk, NV4{});
          } else {
            uint4 o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float4 f = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
              if (bias) { f.x += bias[4 * i]; f.y += bias[4 * i + 1]; f.z += bias[4 * i + 2]; f.w += bias[4 * i + 3]; }
              o[i] = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
            }
            emit(c, o, NV8{});
          }
        };
#pragma unroll 1
        for (int c = cfirst; c < cfirst + WCH; c += 2) {
          uint32_t r0[32], r1[32];
          tmem_ld32_issue(tbase + c * 32, r0);
          tmem_ld32_issue(tbase + (c + 1) * 32, r1);
          tmem_wait_ld(r0, r1);
          if (c + 2 >= cfirst + WCH) release();
          store_chunk(c, r0);
          store_chunk(c + 1, r1);
        }
      }
      if (!released) release();
      if (++acc == NACC) { acc = 0; aphase ^= 1u; }
    }
    // every staged box has been written to global memory
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0) pdl_trigger();
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

// 2-D bf16 tensor [rows, K] (K contiguous) read in boxes of box_rows x 64.
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

// Output tensor [rows, cols] (row stride ld elements, bf16 or fp32) written
// by the epilogue in 128-byte x 32-row boxes, 128-byte swizzle.
cudaError_t make_out_map(CUtensorMap* m, void* base, long long rows, int cols, long long ld, bool f32) {
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE, int MT>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3, const GemmArgs& g,
                        long long rows_bound, int num_sms, cudaStream_t st) {
  CUtensorMap o;
  cudaError_t e = make_out_map(&o, g.out, g.out_rows, g.N_out, g.out_ld, MODE == MODE_DOWN);
  if (e != cudaSuccess) return e;
  auto kern = grouped_gemm_kernel<MODE, MT>;
  constexpr int smem = Cfg<MT>::SMEM_BYTES;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // upper bound on tiles: every expert may add one partial M tile
  const long long mt_bound = (rows_bound + Cfg<MT>::TILE_M - 1) / Cfg<MT>::TILE_M + g.E;
  const long long tiles_bound = mt_bound * g.n_tiles;
  const int grid = static_cast<int>(std::min<long long>(num_sms, std::max<long long>(1, tiles_bound)));
  return launch_pdl(kern, dim3(grid), dim3(NTHREADS), static_cast<size_t>(smem), st, 1, a, b, b3, o, g);
}

}  // namespace

// out[r, n] = sum over k < K of A[r, k mod Ka] * B[n, k], fp32 (dense, one group):
// A [rows, Ka] bf16, B [N, K] bf16, K a multiple of Ka, Ka a multiple of 64.
cudaError_t launch_dense_wrapped_gemm(const void* A, long long rows, int Ka, const void* B, int N, int K, float* out,
                                      int* err, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int MT = rows > 4LL * BM ? 2 : 1;
  CUtensorMap mA, mB;
  if ((e = make_map(&mA, A, rows, Ka, BM * MT)) != cudaSuccess) return e;
  if ((e = make_map(&mB, B, N, K, BN)) != cudaSuccess) return e;
  GemmArgs g{};
  g.offsets = nullptr;
  g.dense_rows = static_cast<int>(rows);
  g.a_kwrap = Ka / BK;
  g.E = 1;
  g.N_out = N;
  g.N_w = N;
  g.K = K;
  g.n_tiles = (N + BN - 1) / BN;
  g.out = out;
  g.out_ld = N;
  g.out_rows = rows;
  g.bias = nullptr;
  g.err = err;
  return MT == 2 ? launch_mode<MODE_DOWN, 2>(mA, mB, mB, g, rows, sms, st)
                 : launch_mode<MODE_DOWN, 1>(mA, mB, mB, g, rows, sms, st);
}

cudaError_t launch_ffn_bf16(const FfnParams& p, cudaStream_t st, cudaEvent_t between_gemms) {
  if (p.rows == 0) return cudaSuccess;
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;

  const bool swiglu = p.act == MOE_ACT_SWIGLU;
  // 256-row tiles when experts are expected to hold more than four M tiles
  // (the unoverlapped epilogue then costs little and the shared B stage
  // pays); 128-row tiles otherwise
  const int MT = p.rows > 4LL * BM * p.E ? 2 : 1;
  CUtensorMap mA1, mB1, mB3, mA2, mB2;
  if ((e = make_map(&mA1, p.x_perm, p.rows, p.d, BM * MT)) != cudaSuccess) return e;
  if ((e = make_map(&mB1, p.W1, static_cast<long long>(p.E) * p.F, p.d, swiglu ? BN / 2 : BN)) != cudaSuccess) return e;
  if (swiglu) {
    if ((e = make_map(&mB3, p.W3, static_cast<long long>(p.E) * p.F, p.d, BN / 2)) != cudaSuccess) return e;
  } else {
    mB3 = mB1;
  }
  if ((e = make_map(&mA2, p.h, p.rows, p.F, BM * MT)) != cudaSuccess) return e;
  if ((e = make_map(&mB2, p.W2, static_cast<long long>(p.E) * p.d, p.F, BN)) != cudaSuccess) return e;

  NvtxRange r1("expert_gemm1");
  GemmArgs g1{};
  g1.offsets = p.offsets;
  g1.dense_rows = p.offsets ? 0 : static_cast<int>(p.rows);
  g1.E = p.E;
  g1.N_out = p.F;
  g1.N_w = p.F;
  g1.K = p.d;
  g1.n_tiles = (p.F + (swiglu ? 127 : 255)) / (swiglu ? 128 : 256);
  g1.out = p.h;
  g1.out_ld = p.F;
  g1.out_rows = p.rows;
  g1.bias = swiglu ? nullptr : p.b1;
  g1.err = p.err;
  if (MT == 2)
    e = swiglu ? launch_mode<MODE_SWIGLU, 2>(mA1, mB1, mB3, g1, p.rows, sms, st)
               : launch_mode<MODE_GELU, 2>(mA1, mB1, mB3, g1, p.rows, sms, st);
  else
    e = swiglu ? launch_mode<MODE_SWIGLU, 1>(mA1, mB1, mB3, g1, p.rows, sms, st)
               : launch_mode<MODE_GELU, 1>(mA1, mB1, mB3, g1, p.rows, sms, st);
  if (e != cudaSuccess) return e;
  if (between_gemms != nullptr) {
    // an external record node when captured into a graph, so it still times
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(st, &cs)) != cudaSuccess) return e;
    const unsigned int flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    if ((e = cudaEventRecordWithFlags(between_gemms, st, flags)) != cudaSuccess) return e;
  }

  NvtxRange r2("expert_gemm2");
  GemmArgs g2{};
  g2.offsets = p.offsets;
  g2.dense_rows = g1.dense_rows;
  g2.E = p.E;
  g2.N_out = p.d;
  g2.N_w = p.d;
  g2.K = p.F;
  g2.n_tiles = (p.d + 255) / 256;
  g2.out = p.y_perm;
  g2.out_ld = p.d;
  g2.out_rows = p.rows;
  g2.bias = p.b2;
  g2.err = p.err;
  return MT == 2 ? launch_mode<MODE_DOWN, 2>(mA2, mB2, mB2, g2, p.rows, sms, st)
                 : launch_mode<MODE_DOWN, 1>(mA2, mB2, mB2, g2, p.rows, sms, st);
}

}  // namespace moe
