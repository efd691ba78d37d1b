// Weighted combine into the residual, and the fp32 CUDA-core expert FFN.
//
// Combine: out[t] = residual[t] + sum over kept ranks r (in order 0..k-1) of
// w[t,r] * y_perm[offsets[idx[t,r]] + pos[t,r]], plus the shared experts'
// output y_shared[t] when there is one  ("LLM part 09: Sparse
// Mixture-of-Experts (MoE)", s1 output equation and s3 residual bypass of
// dropped tokens; "Mixture-of-Experts Sparse Model Scaling", Lab 1 weighted
// accumulation).  Each thread owns 16 (or 8) consecutive elements of one
// token, gathers them from its k expert rows in whole 32-byte sectors (or
// 16-byte loads) and writes them once: deterministic, no atomics, HBM-bound.
//
// fp32 FFN: the grouped expert MLP on CUDA cores for fp32 layers (whose
// tolerance rules out tf32/bf16 tensor cores): one warp per output element,
// lanes split the reduction so every weight row is read with coalesced loads.
// With no segment offsets it is one dense FFN over every row (shared experts).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

template <typename TO>
__device__ __forceinline__ void load4(const TO* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 q = *reinterpret_cast<const float4*>(p);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
  const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
template <typename TO>
__device__ __forceinline__ void store4(TO* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// 32 bytes (a whole sector) from / to global memory in one access when `al`
// (the address is 32-byte aligned), else as two 16-byte accesses.
__device__ __forceinline__ void ld_g32(const void* p, uint4& a, uint4& b, bool al) {
  if (al) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
  } else {
    a = __ldg(static_cast<const uint4*>(p));
    b = __ldg(static_cast<const uint4*>(p) + 1);
  }
}
__device__ __forceinline__ void st_g32(void* p, const uint4& a, const uint4& b, bool al) {
  if (al) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
                 "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
  } else {
    static_cast<uint4*>(p)[0] = a;
    static_cast<uint4*>(p)[1] = b;
  }
}
__device__ __forceinline__ bool al32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
__device__ __forceinline__ void f8_from(const uint4& a, const uint4& b, float* f) {
  f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y); f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
  f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y); f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
}
__device__ __forceinline__ void f8_to(const float* f, uint4& a, uint4& b) {
  a = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  b = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]), __float_as_uint(f[7]));
}

// 16-element chunks (d % 16 == 0): every operand moves in whole 32-byte
// sectors.  One thread per (token, chunk); the chunk's offsets are multiples
// of 32 bytes in every tensor, so a tensor's accesses are 32-byte aligned
// exactly when its base address is.  Same arithmetic as combine_kernel.
template <typename TO>
__global__ void __launch_bounds__(256) combine16_kernel(CombineParams p, long long items, int chunks) {
  pdl_wait();
  pdl_trigger();
  const long long it = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (it >= items) return;
  const long long t = it / chunks;
  const int c = static_cast<int>(it - t * chunks) * 16;
  const int k = p.k, d = p.d;
  const TO* res = static_cast<const TO*>(p.residual);
  float rv[16];
  if (res) {
    const bool al = al32(res);
    if constexpr (sizeof(TO) == 2) {
      uint4 a, b;
      ld_g32(res + t * d + c, a, b, al);
      auto widen = [&](uint32_t u, int i) {
        rv[2 * i] = __uint_as_float(u << 16);
        rv[2 * i + 1] = __uint_as_float(u & 0xffff0000u);
      };
      widen(a.x, 0); widen(a.y, 1); widen(a.z, 2); widen(a.w, 3);
      widen(b.x, 4); widen(b.y, 5); widen(b.z, 6); widen(b.w, 7);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint4 a, b;
        ld_g32(res + t * d + c + 8 * h, a, b, al);
        f8_from(a, b, rv + 8 * h);
      }
    }
  }
  float sv[16];
  if (p.y_shared) {
    const bool al = al32(p.y_shared);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 a, b;
      ld_g32(p.y_shared + t * d + c + 8 * h, a, b, al);
      f8_from(a, b, sv + 8 * h);
    }
  }
  const bool al_y = al32(p.y_perm);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll 2
  for (int r = 0; r < k; ++r) {
    long long row = -1;
    if (p.row_of) {
      row = __ldg(p.row_of + t * k + r);
    } else {
      const int ps = __ldg(p.pos + t * k + r);
      if (ps >= 0) {
        const int e = __ldg(p.idx + t * k + r);
        if (e >= 0 && e < p.E) row = static_cast<long long>(__ldg(p.offsets + e)) + ps;
        if (row < 0) record_error(p.err, MOE_ERR_BOUNDS);
      }
    }
    if (row < 0) continue;  // dropped: the residual carries the token
    if (row >= p.rows) {
      record_error(p.err, MOE_ERR_BOUNDS);
      continue;
    }
    const float wt = __ldg(p.w + t * k + r);
    float yv[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 a, b;
      ld_g32(p.y_perm + row * d + c + 8 * h, a, b, al_y);
      f8_from(a, b, yv + 8 * h);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = fmaf(wt, yv[i], acc[i]);
  }
  if (p.y_shared) {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] += sv[i];
  }
  if (p.moe_out) {
    const bool al = al32(p.moe_out);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 a, b;
      f8_to(acc + 8 * h, a, b);
      st_g32(p.moe_out + t * d + c + 8 * h, a, b, al);
    }
  }
  float o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = res ? rv[i] + acc[i] : acc[i];
  TO* out = static_cast<TO*>(p.out);
  const bool al = al32(out);
  if constexpr (sizeof(TO) == 2) {
    auto pack = [&](int i) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      return *reinterpret_cast<const uint32_t*>(&h2);
    };
    st_g32(out + t * d + c, make_uint4(pack(0), pack(1), pack(2), pack(3)),
           make_uint4(pack(4), pack(5), pack(6), pack(7)), al);
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 a, b;
      f8_to(o + 8 * h, a, b);
      st_g32(out + t * d + c + 8 * h, a, b, al);
    }
  }
}

// One thread per (token, V-element chunk) when d is a multiple of 8 but not
// of 16 (V = 8; 16-element chunks use combine16_kernel): it resolves the
// token's kept expert rows (from the grouped-row map when the dispatch wrote
// one, else from idx / pos / offsets), issues every 16-byte load of the
// chunk at once (k expert rows, the residual), and writes the chunk once.
// Ranks are summed in order 0..k-1 in fp32.
template <typename TO, int V>
__global__ void __launch_bounds__(256) combine_kernel(CombineParams p, long long items, int chunks) {
  pdl_wait();
  pdl_trigger();
  const long long it = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (it >= items) return;
  const long long t = it / chunks;
  const int c = static_cast<int>(it - t * chunks) * V;
  const int k = p.k, d = p.d;
  // the residual chunk first: its load overlaps the expert-row loads
  const TO* res = static_cast<const TO*>(p.residual);
  float rv[V];
  if (res) {
#pragma unroll
    for (int q = 0; q < V; q += 4) {
      float r4[4];
      load4<TO>(res + t * d + c + q, r4);
#pragma unroll
      for (int i = 0; i < 4; ++i) rv[q + i] = r4[i];
    }
  }
  float4 sv[V / 4];
  if (p.y_shared) {
    const float4* src = reinterpret_cast<const float4*>(p.y_shared + t * d + c);
#pragma unroll
    for (int q = 0; q < V / 4; ++q) sv[q] = __ldg(src + q);
  }
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll 2
  for (int r = 0; r < k; ++r) {
    long long row = -1;
    if (p.row_of) {
      row = __ldg(p.row_of + t * k + r);
    } else {
      const int ps = __ldg(p.pos + t * k + r);
      if (ps >= 0) {
        const int e = __ldg(p.idx + t * k + r);
        if (e >= 0 && e < p.E) row = static_cast<long long>(__ldg(p.offsets + e)) + ps;
        if (row < 0) record_error(p.err, MOE_ERR_BOUNDS);
      }
    }
    if (row < 0) continue;  // dropped: the residual carries the token
    if (row >= p.rows) {
      record_error(p.err, MOE_ERR_BOUNDS);
      continue;
    }
    const float wt = __ldg(p.w + t * k + r);
    const float4* src = reinterpret_cast<const float4*>(p.y_perm + row * d + c);
    float4 yv[V / 4];
#pragma unroll
    for (int q = 0; q < V / 4; ++q) yv[q] = __ldg(src + q);
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
      acc[4 * q] = fmaf(wt, yv[q].x, acc[4 * q]);
      acc[4 * q + 1] = fmaf(wt, yv[q].y, acc[4 * q + 1]);
      acc[4 * q + 2] = fmaf(wt, yv[q].z, acc[4 * q + 2]);
      acc[4 * q + 3] = fmaf(wt, yv[q].w, acc[4 * q + 3]);
    }
  }
  if (p.y_shared) {
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
      acc[4 * q] += sv[q].x;
      acc[4 * q + 1] += sv[q].y;
      acc[4 * q + 2] += sv[q].z;
      acc[4 * q + 3] += sv[q].w;
    }
  }
  if (p.moe_out) {
    float4* mo = reinterpret_cast<float4*>(p.moe_out + t * d + c);
#pragma unroll
    for (int q = 0; q < V / 4; ++q) mo[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
  TO* out = static_cast<TO*>(p.out);
#pragma unroll
  for (int q = 0; q < V; q += 4) {
    float o4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o4[i] = res ? rv[q + i] + acc[q + i] : acc[q + i];
    store4<TO>(out + t * d + c + q, o4);
  }
}

// d not a multiple of 8 (fp32 layers with d % 4 == 0): one warp per token, 4 elements per lane.
template <typename TO>
__global__ void __launch_bounds__(256) combine_kernel4(CombineParams p) {
  pdl_wait();
  pdl_trigger();
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= p.T) return;
  const int k = p.k, d = p.d;
  for (int c = lane * 4; c < d; c += 128) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < k; ++r) {
      long long row = -1;
      if (p.row_of) {
        row = p.row_of[t * k + r];
        if (row < 0) continue;
      } else {
        const int ps = p.pos[t * k + r];
        if (ps < 0) continue;
        const int e = p.idx[t * k + r];
        if (e >= 0 && e < p.E) row = static_cast<long long>(p.offsets[e]) + ps;
      }
      if (row < 0 || row >= p.rows) {
        record_error(p.err, MOE_ERR_BOUNDS);
        continue;
      }
      const float wt = p.w[t * k + r];
      const float4 q = __ldg(reinterpret_cast<const float4*>(p.y_perm + row * d + c));
      acc[0] = fmaf(wt, q.x, acc[0]); acc[1] = fmaf(wt, q.y, acc[1]);
      acc[2] = fmaf(wt, q.z, acc[2]); acc[3] = fmaf(wt, q.w, acc[3]);
    }
    if (p.y_shared) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p.y_shared + t * d + c));
      acc[0] += q.x; acc[1] += q.y; acc[2] += q.z; acc[3] += q.w;
    }
    if (p.moe_out) store4<float>(p.moe_out + t * d + c, acc);
    float o[4] = {acc[0], acc[1], acc[2], acc[3]};
    if (p.residual) {
      float rv[4];
      load4<TO>(static_cast<const TO*>(p.residual) + t * d + c, rv);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = rv[i] + acc[i];
    }
    store4<TO>(static_cast<TO*>(p.out) + t * d + c, o);
  }
}

// index of the expert whose segment [offsets[e], offsets[e+1]) holds `row`
__device__ __forceinline__ int expert_of_row(const int32_t* offsets, int E, long long row) {
  int lo = 0, hi = E;  // offsets[lo] <= row < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// h[row, f] = act(x_perm[row] . W1[e, f] (+ b1[e, f]))   (SwiGLU: silu(.) * x_perm[row] . W3[e, f])
__global__ void __launch_bounds__(256) ffn1_f32_kernel(FfnParams p) {
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const int f = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int32_t* off = p.offsets;
  if (row >= (off ? off[p.E] : p.rows) || f >= p.F) return;
  const int e = off ? expert_of_row(off, p.E, row) : 0;
  const float* xr = static_cast<const float*>(p.x_perm) + row * p.d;
  const float* w1 = static_cast<const float*>(p.W1) + (static_cast<long long>(e) * p.F + f) * p.d;
  float a = 0.f, u = 0.f;
  for (int j = lane; j < p.d; j += 32) a = fmaf(xr[j], w1[j], a);
  a = warp_sum(a);
  float h;
  if (p.act == MOE_ACT_SWIGLU) {
    const float* w3 = static_cast<const float*>(p.W3) + (static_cast<long long>(e) * p.F + f) * p.d;
    for (int j = lane; j < p.d; j += 32) u = fmaf(xr[j], w3[j], u);
    u = warp_sum(u);
    h = a / (1.0f + expf(-a)) * u;
  } else {
    if (p.b1) a += p.b1[static_cast<long long>(e) * p.F + f];
    h = 0.5f * a * (1.0f + erff(a * 0.70710678118654752f));
  }
  if (lane == 0) static_cast<float*>(p.h)[row * p.F + f] = h;
}

// y_perm[row, i] = h[row] . W2[e, i] (+ b2[e, i])
__global__ void __launch_bounds__(256) ffn2_f32_kernel(FfnParams p) {
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const int i = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int32_t* off = p.offsets;
  if (row >= (off ? off[p.E] : p.rows) || i >= p.d) return;
  const int e = off ? expert_of_row(off, p.E, row) : 0;
  const float* hr = static_cast<const float*>(p.h) + row * p.F;
  const float* w2 = static_cast<const float*>(p.W2) + (static_cast<long long>(e) * p.d + i) * p.F;
  float a = 0.f;
  for (int j = lane; j < p.F; j += 32) a = fmaf(hr[j], w2[j], a);
  a = warp_sum(a);
  if (p.b2) a += p.b2[static_cast<long long>(e) * p.d + i];
  if (lane == 0) p.y_perm[row * p.d + i] = a;
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  if (p.d % 16 == 0) {
    const int chunks = p.d / 16;
    const long long items = static_cast<long long>(p.T) * chunks;
    const long long blocks = (items + 255) / 256;
    if (p.dtype == MOE_BF16)
      return launch_pdl(combine16_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p,
                        items, chunks);
    else
      return launch_pdl(combine16_kernel<float>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p, items,
                        chunks);
  } else if (p.d % 8 == 0) {
    const int chunks = p.d / 8;
    const long long items = static_cast<long long>(p.T) * chunks;
    const long long blocks = (items + 255) / 256;
    if (p.dtype == MOE_BF16)
      return launch_pdl(combine_kernel<__nv_bfloat16, 8>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p,
                        items, chunks);
    else
      return launch_pdl(combine_kernel<float, 8>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p, items,
                        chunks);
  } else {
    const long long blocks = (static_cast<long long>(p.T) * 32 + 255) / 256;
    if (p.dtype == MOE_BF16)
      return launch_pdl(combine_kernel4<__nv_bfloat16>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p);
    else
      return launch_pdl(combine_kernel4<float>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_ffn_f32(const FfnParams& p, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  dim3 g1(static_cast<unsigned>(p.rows), static_cast<unsigned>((p.F + 7) / 8));
  cudaError_t e = launch_pdl(ffn1_f32_kernel, g1, dim3(256), 0, st, 1, p);
  if (e != cudaSuccess) return e;
  dim3 g2(static_cast<unsigned>(p.rows), static_cast<unsigned>((p.d + 7) / 8));
  return launch_pdl(ffn2_f32_kernel, g2, dim3(256), 0, st, 1, p);
}

}  // namespace moe
