// Element formats of the logit tensors and the small fixed-association
// reductions shared by the vocabulary-sweep kernels.  Every reduction here
// has a fixed association, so every CTA that runs it on the same inputs gets
// bit-identical results.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace ssv {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ---- element formats ---------------------------------------------------------

struct Bf16 {
  static constexpr int PV = 8;  // elements per 16-byte vector
  static constexpr int ES = 2;
  using Raw = uint16_t;
  static constexpr Raw kNegInf = 0xFF80u;
  __device__ static __forceinline__ void unpack(const uint4& w, float (&x)[8]) {
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xFFFF0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xFFFF0000u);
    x[4] = __uint_as_float(w.z << 16);
    x[5] = __uint_as_float(w.z & 0xFFFF0000u);
    x[6] = __uint_as_float(w.w << 16);
    x[7] = __uint_as_float(w.w & 0xFFFF0000u);
  }
  // The 8 values as 4 packed pairs in element order (exact widening).
  __device__ static __forceinline__ void pairs(const uint4& w, f32x2 (&p)[4]) {
    p[0] = f2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
    p[1] = f2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
    p[2] = f2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
    p[3] = f2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
  }
  __device__ static __forceinline__ float to_f32(Raw r) { return __uint_as_float(uint32_t(r) << 16); }
  // Maximum of the 8 values of a vector (packed compares; max needs no rounding).
  __device__ static __forceinline__ float vmax(const uint4& w) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
  // Maximum of a vector ignoring NaN, and whether the vector holds a NaN.
  __device__ static __forceinline__ float vmax_nan(const uint4& w, bool& nan) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
    const __nv_bfloat162 mn = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    const float lo = __low2float(mn), hi = __high2float(mn);
    nan = (lo != lo) || (hi != hi);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
};

struct F32 {
  static constexpr int PV = 4;
  static constexpr int ES = 4;
  using Raw = uint32_t;
  static constexpr Raw kNegInf = 0xFF800000u;
  __device__ static __forceinline__ void unpack(const uint4& w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x);
    x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z);
    x[3] = __uint_as_float(w.w);
  }
  __device__ static __forceinline__ void pairs(const uint4& w, f32x2 (&p)[2]) {
    p[0] = f2(__uint_as_float(w.x), __uint_as_float(w.y));
    p[1] = f2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
  __device__ static __forceinline__ float to_f32(Raw r) { return __uint_as_float(r); }
  __device__ static __forceinline__ float vmax(const uint4& w) {
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
  __device__ static __forceinline__ float vmax_nan(const uint4& w, bool& nan) {
    const float a = __uint_as_float(w.x), b = __uint_as_float(w.y), c = __uint_as_float(w.z), d = __uint_as_float(w.w);
    nan = (a != a) || (b != b) || (c != c) || (d != d);
    return fmaxf(fmaxf(a, b), fmaxf(c, d));
  }
};

// ---- small reductions (fixed association: identical in every CTA) ------------------

template <int N>
__device__ __forceinline__ float tree_sum(const float (&x)[N]) {
  if constexpr (N == 8) {
    return __fadd_rn(__fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3])),
                     __fadd_rn(__fadd_rn(x[4], x[5]), __fadd_rn(x[6], x[7])));
  } else {
    return __fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3]));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v = __fadd_rn(v, t);
  }
  return v;
}

// Two rows at once: the maxima in one warp instruction each, then the
// rescaled sums through one shuffle tree whose two chains overlap.
__device__ __forceinline__ void warp_combine_mz2(float& m1, float& z1, float& m2, float& z2, float s) {
  const float M1 = redux_max_f32(m1), M2 = redux_max_f32(m2);
  const float f1 = (m1 > -INFINITY) ? ex2(__fadd_rn(__fmul_rn(m1, s), -__fmul_rn(M1, s))) : 0.0f;
  const float f2 = (m2 > -INFINITY) ? ex2(__fadd_rn(__fmul_rn(m2, s), -__fmul_rn(M2, s))) : 0.0f;
  float a = __fmul_rn(z1, f1), b = __fmul_rn(z2, f2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ta = __shfl_xor_sync(kFull, a, o);
    const float tb = __shfl_xor_sync(kFull, b, o);
    a = __fadd_rn(a, ta);
    b = __fadd_rn(b, tb);
  }
  z1 = a;
  z2 = b;
  m1 = M1;
  m2 = M2;
}

// Warp argmax in two warp instructions: the largest value, then the smallest
// index among the lanes holding it.
__device__ __forceinline__ void warp_argmax_redux(float& v, int& i) {
  const float M = redux_max_f32(v);
  const uint32_t cand = (v == M) ? (uint32_t)i : 0xFFFFFFFFu;
  i = (int)redux_min_u32(cand);
  v = M;
}

// Sum of a vector's values held as pairs: ((v0 + v1) + (v2 + v3)) per lane.
template <int NP>
__device__ __forceinline__ f32x2 psum(const f32x2 (&v)[NP]) {
  if constexpr (NP == 4) {
    return f2_add(f2_add(v[0], v[1]), f2_add(v[2], v[3]));
  } else {
    return f2_add(v[0], v[1]);
  }
}

// 2^(z s - c) of the values of one vector, as pairs in element order;
// S2 = (s, s), C2 = (-c, -c).  Each lane is fmaf(z, s, -c) then ex2.
template <class E>
__device__ __forceinline__ void exp_pairs(const uint4& w, f32x2 S2, f32x2 C2, f32x2 (&ep)[E::PV / 2]) {
  f32x2 p[E::PV / 2];
  E::pairs(w, p);
#pragma unroll
  for (int h = 0; h < E::PV / 2; ++h) {
    float x0, x1;
    f2_split(f2_fma(p[h], S2, C2), x0, x1);
    ep[h] = f2(ex2(x0), ex2(x1));
  }
}

}  // namespace ssv
