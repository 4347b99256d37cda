// Vocabulary sweep kernels for sm_103a.
//
// A (row b, position k) "unit" is one target row (and, for drafted positions,
// one draft row) of V logits.  A thread-block cluster of S CTAs works on one
// unit at a time: CTA r of the cluster owns the slice [r*L, min((r+1)*L, V)).
// The kernel is persistent: cluster c processes units c, c+G, c+2G, ... and
// every CTA keeps two shared-memory stages, so the 1-D bulk (TMA) copies of
// the next unit's slice are in flight while the current unit is computed.
// Each warp owns a contiguous segment of 16-byte vectors in both stages,
// issues the bulk copies for that segment itself (completing on its own
// mbarrier) and is the only reader of it, so no block-wide barrier orders the
// staging against the compute.
//
// Per unit (sampling, T > 0):
//   pass A  thread-local maxima (packed bf16x2 compares)
//   pass B  thread-local sums of 2^((z - m) s), s = log2(e)/T
//           -> block and cluster combine of (max, sum) pairs   [exchange 1]
//   decide  accept iff u * q(y) <= p(y) (identical in every CTA)
//   pass C  accepted drafts: sum_v min(p, q) through min(log p, log q), one
//           exp per element; the CTA's partial goes to the workspace.
//           rejected drafts / bonus: weights max(0, p - q) (or p) with per
//           round warp scans; CTA totals are exchanged           [exchange 2]
//           and the owning CTA / warp / round / lane / element of
//           u' * total is located; one warp recomputes one round.
// Thread 0 of each CTA writes the unit's record / overlap partial and queues
// an arrival for the unit's row.  Arrivals are published in batches (one
// release fence, then up to 32 counter updates in parallel by warp 0) when
// 32 rows are queued and at the end; the CTA completing a row decides the
// prefix-order outcome, sums the overlap partials in rank order and re-zeroes
// the workspace it used.
#pragma once

#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "ptx.cuh"

namespace ssv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPartStride = 16;    // partial slots per unit (max cluster size)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait
constexpr unsigned kFull = 0xFFFFFFFFu;

constexpr uint32_t kBadToken = 1u, kBadLogits = 2u, kBadUniform = 4u, kTimeout = 8u, kEmptyResidual = 16u;

// Earliest-rejection word of a row: kRejBase - j for a rejection at position j
// (larger = earlier; 0 = none seen yet).
constexpr uint32_t kRejBase = 128u;

// kVerifyGrouped is kVerify with rows in groups of one row per cluster,
// position-major inside a group (for at least as many rows as clusters).
// kVerifyRagged is kVerify over flattened rows of their own lengths: unit u is
// flattened target row u, described by a packed word (row, position, bonus).
// kVerifyRelaxed is kVerify with the relaxed (lossy) acceptance: target top-k
// rank and log-probability gap; a rejection draws from the full target.
// kArgmax writes the target argmax of every unit (a candidate tree's slots)
// to out_tokens, with no row completion.
enum Mode : int { kVerify = 0, kVerifyGreedy = 1, kOverlap = 2, kOverlapGreedy = 3, kE2E = 4, kDiag = 5,
                  kVerifyGrouped = 6, kVerifyRagged = 7, kVerifyRelaxed = 8, kArgmax = 9 };

// Packed unit word of the ragged verify: row << 8 | bonus << 7 | position.
__host__ __device__ constexpr uint32_t pack_unit(uint32_t row, uint32_t pos, bool bonus) {
  return (row << 8) | (bonus ? 0x80u : 0u) | pos;
}

struct VerifyRecord {  // one per (b, k), k = 0..K
  int32_t acc;         // 1 accepted, 0 rejected, 2 rejected with an empty residual (draft positions)
  int32_t token;       // correction / bonus / greedy choice; -1 if none
  uint32_t pad0, pad1;
};

struct E2EStats {  // one per (b, k), k = 0..K-1
  float c1t;       // fl(M_t * s): exponent offset of the target row
  float cd;        // offset of the draft row with log2(Z_d / Z_t) folded in
  float izt;       // 1 / Z_t
  float smass;     // S = sum_{q_v < p_v} q_v
  float alpha;
  float b1, b0;    // gradient multipliers for indicator 1 / 0
  float pad;
};

struct SweepParams {
  const void* target;
  const void* draft;
  int B, K, KT, V;
  int units;
  int S;        // CTAs per cluster
  int L;        // slice length in elements (multiple of 8)
  int cpt;      // 16-byte vectors per thread (odd, cpt * kThreads >= L / elements per vector)
  int aligned;  // rows start on 16-byte boundaries: bulk copies allowed
  int nst;      // shared-memory stages per CTA (1 or 2)
  int rows;     // logit rows staged per unit: 2 (target and draft) or 1 (target only)
  float s;      // log2(e) / T
  float inv_t;  // 1 / T
  float grad_scale;
  const int32_t* draft_tokens;
  const float* u_accept;
  const float* u_final;
  int32_t* out_tokens;
  int32_t* n_accepted;
  float* alpha;
  float* tv;
  float* surv;
  float* exp_acc;
  float* loss;
  VerifyRecord* rec;
  E2EStats* stats;
  float* part;   // [units][kPartStride] overlap partials
  float* part2;  // [units][kPartStride] E2E S-mass partials; diagnostics: entropy partials
  float* part3;  // [units][kPartStride] diagnostics: KL partials
  float* ent;    // [B, K] diagnostics outputs (each may be null)
  float* ce;
  float* kl;
  float* ato;
  float* row_loss;
  uint32_t* row_cnt;
  uint32_t* rej;  // [B] sampling verify: kRejBase - (earliest rejected position seen), 0 if none
  const uint2* uinfo;      // ragged: [units] {flattened target row, packed unit word}, drafts first
  const int32_t* roff;     // ragged: [B + 1] first flattened target row of every row
  const uint32_t* ragbad;  // ragged: nonzero when the offsets were rejected (nothing runs)
  int relax_k;             // relaxed: top-k rank bound (<= 0: none)
  float relax_delta;       // relaxed: log-probability gap bound (+inf: none)
  uint32_t* glob_cnt;
  uint32_t* status;
};

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

// Per-element weights of the residual / target draws and their vector total.
// The sweep and the owner's walk call this same function, so both see
// bit-identical weights and totals.  NR = (-Z_t/Z_d, -Z_t/Z_d).
template <class E, bool kResidual>
__device__ __forceinline__ float draw_weights(const uint4& wt, const uint4& wd, f32x2 S2, f32x2 CT, f32x2 CD,
                                              f32x2 NR, float (&w)[E::PV], f32x2& min_mass) {
  constexpr int NP = E::PV / 2;
  f32x2 et[NP], wp[NP];
  exp_pairs<E>(wt, S2, CT, et);
  if constexpr (kResidual) {
    f32x2 ed[NP], mp[NP];
    exp_pairs<E>(wd, S2, CD, ed);
    const f32x2 N1 = f2(-1.0f, -1.0f);
#pragma unroll
    for (int h = 0; h < NP; ++h) {
      // rho' = Z_t * max(0, p - q) = max(0, e_t - e_d * Z_t / Z_d)
      float r0, r1;
      f2_split(f2_fma(ed[h], NR, et[h]), r0, r1);
      r0 = fmaxf(r0, 0.0f);
      r1 = fmaxf(r1, 0.0f);
      wp[h] = f2(r0, r1);
      mp[h] = f2_fma(wp[h], N1, et[h]);  // Z_t * min(p, q) = e_t - rho'
      w[2 * h] = r0;
      w[2 * h + 1] = r1;
    }
    min_mass = f2_add(min_mass, psum(mp));
  } else {
#pragma unroll
    for (int h = 0; h < NP; ++h) {
      wp[h] = et[h];
      f2_split(et[h], w[2 * h], w[2 * h + 1]);
    }
  }
  return f2_hsum(psum(wp));
}

// ---- per-row completion (one warp of the CTA whose arrival completes the row) ----
// Decides the prefix-order outcome, sums the CTA partials in rank order and
// re-zeroes the workspace of row b.
template <int MODE>
__device__ __forceinline__ void complete_row(const SweepParams& P, int b, int S, int lane) {
  constexpr bool kVerifyMode = (MODE == kVerify || MODE == kVerifyGreedy || MODE == kVerifyGrouped ||
                                 MODE == kVerifyRagged || MODE == kVerifyRelaxed);
  // units of row b: [base, base + per_row); drafted positions K of them,
  // the first at dbase
  int K = P.K;
  int per_row = kVerifyMode ? K + 1 : K;
  int base = b * per_row;
  if constexpr (MODE == kVerifyRagged) {
    base = __ldg(P.roff + b);
    per_row = __ldg(P.roff + b + 1) - base;
    K = per_row - 1;
  }
  const int dbase = (MODE == kVerifyRagged) ? base - b : b * K;
  const float* pp0 = P.part + (long long)base * kPartStride;
  // overlap of position kk: partials summed in rank order
  auto alpha_of = [&](int kk) {
    const float* pp = pp0 + kk * kPartStride;
    float a = 0.0f;
    for (int r = 0; r < S; ++r) a = __fadd_rn(a, __ldcg(pp + r));
    return a;
  };
  if constexpr (kVerifyMode) {
    const VerifyRecord* rr = P.rec + base;
    // acc: 1 accepted, 0 rejected, 2 rejected with an empty residual
    int nacc = K, acc_first = 1;
    for (int k0 = 0; k0 < K; k0 += 32) {
      const int kk = k0 + lane;
      const int a = (kk < K) ? __ldcg(&rr[kk].acc) : 1;
      const unsigned m = __ballot_sync(kFull, (a & 1) == 0);
      if (m) {
        const int l = __ffs(m) - 1;
        nacc = k0 + l;
        acc_first = __shfl_sync(kFull, a, l);
        break;
      }
    }
    const int corr = __ldcg(&rr[nacc].token);
    if (lane == 0 && acc_first == 2 && P.status) atomicOr(P.status, kEmptyResidual);
    for (int kk = lane; kk <= K; kk += 32) {
      int tokv = -1;
      if (kk < nacc) tokv = P.draft_tokens[dbase + kk];
      else if (kk == nacc) tokv = corr;
      P.out_tokens[base + kk] = tokv;
      if (kk < K && P.alpha) P.alpha[dbase + kk] = alpha_of(kk);
    }
    __syncwarp();
    VerifyRecord* rw = P.rec + base;
    float* pw = P.part + (long long)base * kPartStride;
    for (int kk = lane; kk <= K; kk += 32) rw[kk] = VerifyRecord{0, 0, 0u, 0u};
    for (int i = lane; i < per_row * kPartStride; i += 32) pw[i] = 0.0f;
    if (lane == 0) {
      P.n_accepted[b] = nacc;
      P.row_cnt[b] = 0;
      if (P.rej) P.rej[b] = 0;
    }
  } else if constexpr (MODE == kOverlap || MODE == kOverlapGreedy) {
    float al[2];
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      al[h] = (kk < K) ? alpha_of(kk) : 0.0f;
      if (kk < K) {
        P.alpha[b * K + kk] = al[h];
        if (P.tv) P.tv[b * K + kk] = 1.0f - al[h];
      }
    }
    // prefix products in position order
    float pr = 1.0f, sum = 0.0f;
    for (int kk = 0; kk < K; ++kk) {
      const float a = __shfl_sync(kFull, al[kk >> 5], kk & 31);
      pr = __fmul_rn(pr, a);
      sum = __fadd_rn(sum, pr);
      if (lane == 0 && P.surv) P.surv[b * K + kk] = pr;
    }
    __syncwarp();
    float* pw = P.part + (long long)b * per_row * kPartStride;
    for (int i = lane; i < per_row * kPartStride; i += 32) pw[i] = 0.0f;
    if (lane == 0) {
      if (P.exp_acc) P.exp_acc[b] = sum;
      P.row_cnt[b] = 0;
    }
  } else if constexpr (MODE == kDiag) {
    const float* hh0 = P.part2 + (long long)b * K * kPartStride;
    const float* kk0 = P.part3 + (long long)b * K * kPartStride;
    const float ln2 = 0.69314718055994531f;
    for (int kk = lane; kk < K; kk += 32) {
      const float* hh = hh0 + kk * kPartStride;
      const float* kq = kk0 + kk * kPartStride;
      float hs = 0.0f, ks = 0.0f;
      for (int r = 0; r < S; ++r) {
        hs = __fadd_rn(hs, __ldcg(hh + r));
        ks = __fadd_rn(ks, __ldcg(kq + r));
      }
      const float H = __fmul_rn(-ln2, hs), KL = __fmul_rn(ln2, ks);
      if (P.alpha) P.alpha[b * K + kk] = alpha_of(kk);
      if (P.ent) P.ent[b * K + kk] = H;
      if (P.kl) P.kl[b * K + kk] = KL;
      if (P.ce) P.ce[b * K + kk] = __fadd_rn(H, KL);
    }
    __syncwarp();
    float* pw = P.part + (long long)b * K * kPartStride;
    float* pw2 = P.part2 + (long long)b * K * kPartStride;
    float* pw3 = P.part3 + (long long)b * K * kPartStride;
    for (int i = lane; i < K * kPartStride; i += 32) {
      pw[i] = 0.0f;
      pw2[i] = 0.0f;
      pw3[i] = 0.0f;
    }
    if (lane == 0) P.row_cnt[b] = 0;
  } else {  // kE2E
    E2EStats* sr = P.stats + (long long)b * K;
    const float* qq0 = P.part2 + (long long)b * K * kPartStride;
    float al[2], sm2[2];
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      al[h] = 0.0f;
      sm2[h] = 0.0f;
      if (kk < K) {
        al[h] = alpha_of(kk);
        const float* qq = qq0 + kk * kPartStride;
        for (int r = 0; r < S; ++r) sm2[h] = __fadd_rn(sm2[h], __ldcg(qq + r));
        if (P.alpha) P.alpha[b * K + kk] = al[h];
      }
    }
    // prefix products P_{k-1}, suffix sums G_k = 1 + alpha_{k+1} G_{k+1}
    float pre[2] = {1.0f, 1.0f}, suf[2] = {1.0f, 1.0f};
    float pr = 1.0f, rowl = 0.0f;
    for (int kk = 0; kk < K; ++kk) {
      if ((kk & 31) == lane) pre[kk >> 5] = pr;
      pr = __fmul_rn(pr, __shfl_sync(kFull, al[kk >> 5], kk & 31));
      rowl = __fadd_rn(rowl, pr);
    }
    float g = 1.0f;
    for (int kk = K - 1; kk >= 0; --kk) {
      if ((kk & 31) == lane) suf[kk >> 5] = g;
      g = fmaf(__shfl_sync(kFull, al[kk >> 5], kk & 31), g, 1.0f);
    }
    const float scale = P.grad_scale / (float)P.B;
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      if (kk < K) {
        const float coef = __fmul_rn(__fmul_rn(scale, pre[h]), suf[h]);
        const float A = __fmul_rn(__fmul_rn(coef, __ldcg(&sr[kk].izt)), P.inv_t);
        sr[kk].smass = sm2[h];
        sr[kk].alpha = al[h];
        sr[kk].b1 = __fmul_rn(A, 1.0f - sm2[h]);
        sr[kk].b0 = __fmul_rn(A, -sm2[h]);
      }
    }
    __syncwarp();
    float* pw = P.part + (long long)b * K * kPartStride;
    float* pw2 = P.part2 + (long long)b * K * kPartStride;
    for (int i = lane; i < K * kPartStride; i += 32) {
      pw[i] = 0.0f;
      pw2[i] = 0.0f;
    }
    int glast = 0;
    if (lane == 0) {
      P.row_loss[b] = rowl;
      P.row_cnt[b] = 0;
      __threadfence();
      const uint32_t old = atomicAdd(P.glob_cnt, 1u);
      glast = (old == (uint32_t)P.B - 1) ? 1 : 0;
      if (glast) __threadfence();
    }
    glast = __shfl_sync(kFull, glast, 0);
    if (glast) {
      float acc_l = 0.0f;
      for (int i = lane; i < P.B; i += 32) {
        acc_l = __fadd_rn(acc_l, __ldcg(&P.row_loss[i]));
        P.row_loss[i] = 0.0f;
      }
      acc_l = warp_sum(acc_l);
      if (lane == 0) {
        *P.loss = acc_l / (float)P.B;
        *P.glob_cnt = 0;
      }
    }
  }
}

// ---- the sweep kernel ----------------------------------------------------------

struct SweepSmem {
  uint64_t mbar[2][kWarps];
  float wred[kWarps][4];
  int wredi[kWarps][2];
  float wtot[kWarps];
  float wamax[kWarps];  // diagnostics: per-warp draft arg-maximum
  int wamaxi[kWarps];
  uint32_t wcnt[kWarps];  // relaxed: per-warp count of tokens ranked above the drafted one
  float woff[kWarps + 1];
  alignas(16) uint32_t rejw[4];  // sampling verify: the 16-byte group of row words holding this unit's row
  alignas(16) float mbox[2][kPartStride][8];  // pushed by peers: [exchange slot][sender rank][field]
  float bcf[8];
  int bci[8];
  int pend_row[32];  // rows with arrivals not yet published (thread 0)
  int pend_cnt[32];
  int npend;
};

// 16-byte remote vector stores into the mailbox need 16-byte alignment.
static_assert(offsetof(SweepSmem, mbox) % 16 == 0, "mailbox must be 16-byte aligned");
static_assert(sizeof(float) * 8 % 16 == 0, "mailbox rows must be 16-byte multiples");

template <class E, int MODE>
__global__ void __launch_bounds__(kThreads, 4) sweep_kernel(const SweepParams P) {
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ __align__(16) SweepSmem sm;

  constexpr int PV = E::PV;
  using Raw = typename E::Raw;
  constexpr bool kGreedy = (MODE == kVerifyGreedy || MODE == kOverlapGreedy || MODE == kArgmax);
  constexpr bool kVerifyMode = (MODE == kVerify || MODE == kVerifyGreedy || MODE == kVerifyGrouped ||
                                 MODE == kVerifyRagged || MODE == kVerifyRelaxed);
  constexpr bool kSample =
      (MODE == kVerify || MODE == kVerifyGrouped || MODE == kVerifyRagged || MODE == kVerifyRelaxed);
  constexpr bool kRagged = (MODE == kVerifyRagged);
  constexpr bool kRelaxed = (MODE == kVerifyRelaxed);
  if constexpr (kRagged) {
    if (__ldg(P.ragbad)) return;  // the same word for every CTA: the whole grid returns
  }

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = P.S;
  const uint32_t rank = cluster_rank();
  const int cl = blockIdx.x / S;
  const int G = gridDim.x / S;
  const int K = P.K, V = P.V;
  const int per_row = kVerifyMode ? K + 1 : K;
  const float s = P.s;
  const int nst = P.nst;  // shared-memory stages: 1, or 2 (next unit prefetched)

  // slice of this CTA, segment of this warp
  const int e0 = (int)rank * P.L;
  const int e1 = min(e0 + P.L, V);
  const int n = max(e1 - e0, 0);
  const int nvec = (n + PV - 1) / PV;
  const int nvec_alloc = P.L / PV;
  // thread t owns the contiguous chunk [t*cpt, (t+1)*cpt) of 16-byte vectors
  // (cpt odd: the 8 lanes of a quarter warp hit distinct bank groups); a warp's
  // segment is the union of its lanes' chunks
  const int cpt = P.cpt;
  const int seg = 32 * cpt;
  const int v_lo = min(warp * seg, nvec);
  const int v_hi = min(v_lo + seg, nvec);
  const int t_lo = min(v_lo + lane * cpt, v_hi);
  const int t_hi = min(t_lo + cpt, v_hi);
  const bool bulk = P.aligned && v_hi > v_lo;
  const size_t stage_bytes = (size_t)P.rows * (size_t)nvec_alloc * 16u;
  auto stage_t = [&](int st) { return reinterpret_cast<uint4*>(dyn_smem + st * stage_bytes); };

  if (bulk && lane == 0) {
    mbar_init(smem_addr(&sm.mbar[0][warp]), 1);
    mbar_init(smem_addr(&sm.mbar[1][warp]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol = l2_evict_first_policy();

  struct Unit {
    int b, k;
    int u;  // ragged: the unit (its flattened target row and record index)
    bool bonus, has_draft;
    const Raw* tg;
    const Raw* dg;
  };
  auto decode = [&](int u) {
    Unit x;
    if constexpr (kRagged) {
      const uint2 w2 = __ldg(P.uinfo + u);
      x.u = (int)w2.x;  // the unit's flattened target row (its record index)
      const uint32_t w = w2.y;
      x.b = (int)(w >> 8);
      x.k = (int)(w & 0x7Fu);
      x.bonus = (w & 0x80u) != 0u;
    } else if constexpr (MODE == kVerifyGrouped) {
      // Rows in groups of G, position-major inside a group: a unit starts
      // about one unit-time after the earlier positions of its row have
      // decided, so that it can skip a draw that cannot be emitted, and rows
      // keep completing all through the launch.
      const int gsz = G * (K + 1);
      const int g = u / gsz;
      const int j = u - g * gsz;
      const int r0 = g * G;
      const int rg = min(G, P.B - r0);
      x.k = j / rg;
      x.b = r0 + (j - x.k * rg);
      x.bonus = (x.k == K);
    } else if constexpr (MODE == kVerify) {
      // drafted positions row-major, then every row's bonus: the last units
      // read the target only and usually skip their draw (a rejection in
      // the row is known by then)
      const int nd = P.B * K;
      if (u < nd) {
        x.b = u / K;
        x.k = u - x.b * K;
        x.bonus = false;
      } else {
        x.b = u - nd;
        x.k = K;
        x.bonus = true;
      }
    } else if constexpr (kVerifyMode) {
      x.b = u / (K + 1);
      x.k = u - x.b * (K + 1);
      x.bonus = (x.k == K);
    } else {
      x.b = u / K;
      x.k = u - x.b * K;
      x.bonus = false;
    }
    x.has_draft = !x.bonus;
    if constexpr (MODE == kVerifyGreedy) x.has_draft = !x.bonus && P.alpha != nullptr;
    if constexpr (MODE == kArgmax) x.has_draft = false;
    if constexpr (kRagged) {
      x.tg = reinterpret_cast<const Raw*>(P.target) + (long long)x.u * V;
      x.dg = x.has_draft ? reinterpret_cast<const Raw*>(P.draft) + (long long)(x.u - x.b) * V : nullptr;
    } else {
      x.tg = reinterpret_cast<const Raw*>(P.target) + ((long long)x.b * P.KT + x.k) * V;
      x.dg = x.has_draft ? reinterpret_cast<const Raw*>(P.draft) + ((long long)x.b * K + x.k) * V : nullptr;
    }
    return x;
  };

  // index of a unit's record and partials: b * per_row + k
  auto rec_idx = [&](const Unit& x) {
    if constexpr (kRagged) return x.u;
    return x.b * per_row + x.k;
  };

  // Bulk copies of this warp's segment of unit u into stage st (lane 0).
  auto issue = [&](int u, int st) {
    if (!bulk || lane != 0) return;
    const Unit x = decode(u);
    const uint32_t bar = smem_addr(&sm.mbar[st][warp]);
    const uint32_t bytes = (uint32_t)(v_hi - v_lo) * 16u;
    fence_proxy_async_smem();  // earlier generic reads of this segment come first
    mbar_arrive_expect_tx(bar, x.has_draft ? 2u * bytes : bytes);
    uint4* dt = stage_t(st);
    bulk_load(smem_addr(dt + v_lo), x.tg + e0 + (long long)v_lo * PV, bytes, bar, pol);
    if (x.has_draft) bulk_load(smem_addr(dt + nvec_alloc + v_lo), x.dg + e0 + (long long)v_lo * PV, bytes, bar, pol);
  };
  // L2 prefetch of this warp's segment of unit u (lane 0), so that its bulk
  // copy, issued once a stage is free, is served from L2.
  auto prefetch = [&](int u) {
    if (!bulk || lane != 0 || u >= P.units) return;
    const Unit x = decode(u);
    const uint32_t bytes = (uint32_t)(v_hi - v_lo) * 16u;
    bulk_prefetch_l2(x.tg + e0 + (long long)v_lo * PV, bytes);
    if (x.has_draft) bulk_prefetch_l2(x.dg + e0 + (long long)v_lo * PV, bytes);
  };

  // Warp 0 pushes eight values (held by every lane) into slot `slot` of every
  // CTA's mailbox; after the next cluster barrier each CTA reads them locally.
  auto push8 = [&](int slot, float f0, float f1, float f2, float f3, float f4, float f5, float f6, float f7) {
    if (lane < S) {
      const uint32_t a = map_rank(smem_addr(&sm.mbox[slot][rank][0]), (uint32_t)lane);
      st_cluster_v4(a, f0, f1, f2, f3);
      st_cluster_v4(a + 16u, f4, f5, f6, f7);
    }
  };
  auto mb = [&](int slot, int f, float dflt) { return lane < S ? sm.mbox[slot][lane][f] : dflt; };

  // Publishes the queued arrivals (warp 0, converged): one release fence, one
  // counter update per queued row (lanes in parallel), then the rows whose
  // arrivals are complete are finished by the whole warp.
  auto flush = [&]() {
    __syncwarp();
    const int np = __shfl_sync(kFull, sm.npend, 0);  // lane 0 (thread 0) owns the queue
    if (np == 0) return;
    if (lane == 0) __threadfence();
    __syncwarp();
    int row = -1, last = 0;
    if (lane < np) {
      row = sm.pend_row[lane];
      const uint32_t c = (uint32_t)sm.pend_cnt[lane];
      int units_of_row = per_row;
      if constexpr (kRagged) units_of_row = __ldg(P.roff + row + 1) - __ldg(P.roff + row);
      const uint32_t old = atomicAdd(&P.row_cnt[row], c);
      last = (old + c == (uint32_t)(units_of_row * S)) ? 1 : 0;
    }
    unsigned m = __ballot_sync(kFull, last);
    if (m) __threadfence();
    while (m) {
      const int l = __ffs(m) - 1;
      m &= m - 1;
      complete_row<MODE>(P, __shfl_sync(kFull, row, l), S, lane);
    }
    __syncwarp();
    if (lane == 0) sm.npend = 0;
    __syncwarp();
  };
  // Queues one arrival for row b (thread 0).
  auto queue_arrival = [&](int b) {
    const int np = sm.npend;
    if (np > 0 && sm.pend_row[np - 1] == b) {
      sm.pend_cnt[np - 1] += 1;
    } else {
      sm.pend_row[np] = b;
      sm.pend_cnt[np] = 1;
      sm.npend = np + 1;
    }
  };

  int xc = 0;  // exchange counter: mailbox slot xc & 1
  if (tid == 0) sm.npend = 0;
  if (cl < P.units) issue(cl, 0);

  // decision scalars of a unit (thread 0): drafted token and uniforms,
  // fetched one unit ahead
  auto fetch_scalars = [&](int u, int& y_, float& ua_, float& uf_) {
    y_ = -1;
    ua_ = 0.0f;
    uf_ = 0.0f;
    if constexpr (kVerifyMode) {
      const Unit x = decode(u);
      const long long di = kRagged ? (long long)(x.u - x.b) : (long long)x.b * K + x.k;  // drafted position
      if (!x.bonus) y_ = P.draft_tokens[di];
      if constexpr (kSample) {
        if (!x.bonus) ua_ = P.u_accept[di];
        uf_ = P.u_final[x.b];
      }
    }
  };
  int y_next = -1;
  float ua_next = 0.0f, uf_next = 0.0f;
  if (tid == 0 && cl < P.units) fetch_scalars(cl, y_next, ua_next, uf_next);

  for (int it = 0;; ++it) {
    const int u = cl + it * G;
    if (u >= P.units) break;
    const int stg = (nst == 2) ? (it & 1) : 0;
    const uint32_t par = (nst == 2) ? ((uint32_t)(it >> 1) & 1u) : ((uint32_t)it & 1u);

    if (nst == 2) {
      if (u + G < P.units) issue(u + G, stg ^ 1);
      prefetch(u + 2 * G);
    } else {
      if (it > 0) issue(u, 0);  // this warp finished reading its segment of the previous unit
      prefetch(u + G);
    }
    const Unit x = decode(u);

    // this unit's scalars (thread 0), and the next unit's in flight
    const int y = y_next;
    const float ua = ua_next, uf = uf_next;
    if (tid == 0 && u + G < P.units) fetch_scalars(u + G, y_next, ua_next, uf_next);
    const bool tok_ok = x.bonus || (y >= 0 && y < V);
    // earliest rejection of this row seen so far: copied to shared memory
    // (thread 0) while pass A runs, read before the first exchange
    if constexpr (kSample) {
      if (tid == 0) cp_async_16_cg(smem_addr(sm.rejw), P.rej + (x.b & ~3));
    }
    // relaxed: the drafted token and its target logit (lane 0 of every warp,
    // in flight during pass A)
    int ry = -1;
    float rzy = -INFINITY;
    if constexpr (kRelaxed) {
      if (lane == 0 && !x.bonus) {
        ry = P.draft_tokens[(long long)x.b * K + x.k];
        if (ry >= 0 && ry < V) rzy = E::to_f32(x.tg[ry]);
      }
    }

    // queued arrivals are published when the queue is full
    if (warp == 0 && __shfl_sync(kFull, sm.npend, 0) == 32) flush();

    uint4* st = stage_t(stg);
    uint4* sd = st + nvec_alloc;
    bool ok = true;
    if (bulk) {
      ok = mbar_wait_bounded(smem_addr(&sm.mbar[stg][warp]), par, kWaitLimitNs);
    } else if (v_hi > v_lo) {
      // element-wise staging for rows off 16-byte boundaries (-inf padding)
      Raw* rt = reinterpret_cast<Raw*>(st);
      Raw* rd = reinterpret_cast<Raw*>(sd);
      const int lo = v_lo * PV, hi = v_hi * PV;
      for (int i = lo + lane; i < hi; i += 32) {
        const bool in = (e0 + i) < e1;
        rt[i] = in ? x.tg[e0 + i] : E::kNegInf;
        if (x.has_draft) rd[i] = in ? x.dg[e0 + i] : E::kNegInf;
      }
      __syncwarp();
    }
    if (!ok && lane == 0 && P.status) atomicOr(P.status, kTimeout);

    if constexpr (kGreedy) {
      // ============ greedy: argmax of target (and draft) ============
      float bt = -INFINITY, bd = -INFINITY;
      int jt = -1, jd = -1;
      bool nan_seen = false;
      if (ok) {
        // packed maximum per vector; only the winning vector is unpacked later
        for (int j = v_lo + lane; j < v_hi; j += 32) {
          bool nn;
          float vm = E::vmax_nan(st[j], nn);
          nan_seen |= nn;
          if (vm > bt) {
            bt = vm;
            jt = j;
          }
          if (x.has_draft) {
            vm = E::vmax_nan(sd[j], nn);
            nan_seen |= nn;
            if (vm > bd) {
              bd = vm;
              jd = j;
            }
          }
        }
      }
      int it_ = 0x7FFFFFFF, id_ = 0x7FFFFFFF;
      if (jt >= 0) {
        float xv[PV];
        E::unpack(st[jt], xv);
        for (int i = PV - 1; i >= 0; --i)
          if (xv[i] == bt) it_ = e0 + jt * PV + i;
      }
      if (jd >= 0) {
        float xv[PV];
        E::unpack(sd[jd], xv);
        for (int i = PV - 1; i >= 0; --i)
          if (xv[i] == bd) id_ = e0 + jd * PV + i;
      }
      warp_argmax_redux(bt, it_);
      warp_argmax_redux(bd, id_);
      const bool nan_w = __any_sync(kFull, nan_seen);
      if (lane == 0) {
        sm.wred[warp][0] = bt;
        sm.wred[warp][1] = bd;
        sm.wred[warp][2] = nan_w ? 1.0f : 0.0f;
        sm.wredi[warp][0] = it_;
        sm.wredi[warp][1] = id_;
      }
      __syncthreads();
      const int slot = xc & 1;
      if (warp == 0) {
        float v1 = -INFINITY, v2 = -INFINITY, nn = 0.0f;
        int i1 = 0x7FFFFFFF, i2 = 0x7FFFFFFF;
        if (lane < kWarps) {
          v1 = sm.wred[lane][0];
          v2 = sm.wred[lane][1];
          nn = sm.wred[lane][2];
          i1 = sm.wredi[lane][0];
          i2 = sm.wredi[lane][1];
        }
        warp_argmax_redux(v1, i1);
        warp_argmax_redux(v2, i2);
        nn = redux_max_f32(nn);
        push8(slot, v1, v2, nn, __int_as_float(i1), __int_as_float(i2), 0.0f, 0.0f, 0.0f);
      }
      cluster_sync();  // ---- exchange 1
      ++xc;
      if (warp == 0) {
        float v1 = mb(slot, 0, -INFINITY), v2 = mb(slot, 1, -INFINITY), nn = mb(slot, 2, 0.0f);
        int i1 = lane < S ? __float_as_int(sm.mbox[slot][lane][3]) : 0x7FFFFFFF;
        int i2 = lane < S ? __float_as_int(sm.mbox[slot][lane][4]) : 0x7FFFFFFF;
        warp_argmax_redux(v1, i1);
        warp_argmax_redux(v2, i2);
        nn = redux_max_f32(nn);
        if (rank == 0 && lane == 0) {
          uint32_t flags = 0;
          const bool bad = nn != 0.0f || !(v1 < INFINITY) || i1 == 0x7FFFFFFF ||
                           (x.has_draft && (!(v2 < INFINITY) || i2 == 0x7FFFFFFF));
          if (bad) flags |= kBadLogits;
          const int am_t = bad ? -1 : i1;
          const float al = x.has_draft ? ((am_t >= 0 && am_t == i2) ? 1.0f : 0.0f) : 0.0f;
          if constexpr (MODE == kVerifyGreedy) {
            if (!x.bonus && !tok_ok) flags |= kBadToken;
            VerifyRecord r;
            r.acc = (!x.bonus && tok_ok && y == am_t) ? 1 : 0;
            r.token = am_t;
            r.pad0 = r.pad1 = 0;
            P.rec[rec_idx(x)] = r;
          }
          if constexpr (MODE == kArgmax) {
            P.out_tokens[rec_idx(x)] = am_t;
          } else {
            P.part[(long long)rec_idx(x) * kPartStride] = al;
          }
          if (flags && P.status) atomicOr(P.status, flags);
        }
        if (MODE != kArgmax && lane == 0) queue_arrival(x.b);
      }
      continue;
    } else {
      // ============ sampling path: T > 0 ============
      const f32x2 S2 = f2(s, s);
      // ---- pass A: per-thread sums of 2^(z s - c) over the thread's chunk ----
      // c is fl(s * max of the chunk's first vector).  A chunk whose sum is not
      // below 2^100 (a value far above that offset, an infinity or a NaN) is
      // summed again with a running maximum.
      float mt = -INFINITY, md = -INFINITY, zt = 0.0f, zd = 0.0f;
      if (ok && t_lo < t_hi) {
        auto chunk_sum = [&](const uint4* base, float& m, float& z) {
          m = E::vmax(base[t_lo]);
          const float c = __fmul_rn(m, s);
          const f32x2 C2 = f2(-c, -c);
          f32x2 acc = f2(0.0f, 0.0f);
          for (int i = t_lo; i < t_hi; ++i) {
            f32x2 ep[PV / 2];
            exp_pairs<E>(base[i], S2, C2, ep);
            acc = f2_add(acc, psum(ep));
          }
          z = f2_hsum(acc);
          if (!(z < 0x1p100f) || !(c > -INFINITY)) {
            m = -INFINITY;
            z = 0.0f;
            float cm = 0.0f;
            for (int i = t_lo; i < t_hi; ++i) {
              const uint4 w = base[i];
              const float vm = E::vmax(w);
              if (vm > m) {
                const float cn = __fmul_rn(vm, s);
                z = (m > -INFINITY) ? __fmul_rn(z, ex2(__fadd_rn(cm, -cn))) : 0.0f;
                cm = cn;
                m = vm;
              }
              if (m > -INFINITY) {
                f32x2 ep[PV / 2];
                exp_pairs<E>(w, S2, f2(-cm, -cm), ep);
                z = __fadd_rn(z, f2_hsum(psum(ep)));
              }
            }
          }
        };
        chunk_sum(st, mt, zt);
        if (x.has_draft) chunk_sum(sd, md, zd);
      }
      if constexpr (kRelaxed) {
        // tokens ranked above the drafted one: larger logit, or equal at a smaller index
        const int yy = __shfl_sync(kFull, ry, 0);
        const float zy = __shfl_sync(kFull, rzy, 0);
        uint32_t cnt = 0;
        if (ok && yy >= 0 && yy < V) {
          for (int i = t_lo; i < t_hi; ++i) {
            float xv[PV];
            E::unpack(st[i], xv);
#pragma unroll
            for (int k = 0; k < PV; ++k) cnt += (xv[k] > zy || (xv[k] == zy && e0 + i * PV + k < yy)) ? 1u : 0u;
          }
        }
        cnt = __reduce_add_sync(kFull, cnt);
        if (lane == 0) sm.wcnt[warp] = cnt;
      }
      if constexpr (MODE == kDiag) {
        // arg-maximum of the draft logits (smallest index on ties): y_hat
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF, jb = -1;
        if (ok) {
          for (int i = t_lo; i < t_hi; ++i) {
            const float vm = E::vmax(sd[i]);
            if (vm > bv) {
              bv = vm;
              jb = i;
            }
          }
        }
        if (jb >= 0) {
          float xv[PV];
          E::unpack(sd[jb], xv);
          for (int k = PV - 1; k >= 0; --k)
            if (xv[k] == bv) bi = e0 + jb * PV + k;
        }
        warp_argmax_redux(bv, bi);
        if (lane == 0) {
          sm.wamax[warp] = bv;
          sm.wamaxi[warp] = bi;
        }
      }
      warp_combine_mz2(mt, zt, md, zd, s);
      if (lane == 0) {
        sm.wred[warp][0] = mt;
        sm.wred[warp][1] = zt;
        sm.wred[warp][2] = md;
        sm.wred[warp][3] = zd;
      }
      __syncthreads();
      int slot = xc & 1;
      if (warp == 0) {
        float a = -INFINITY, za = 0.0f, d = -INFINITY, zda = 0.0f;
        if (lane < kWarps) {
          a = sm.wred[lane][0];
          za = sm.wred[lane][1];
          d = sm.wred[lane][2];
          zda = sm.wred[lane][3];
        }
        warp_combine_mz2(a, za, d, zda, s);
        // the CTA holding the drafted token publishes its two logits
        float gt = 0.0f, gd = 0.0f;
        if constexpr (kSample) {
          if (lane == 0 && !x.bonus && tok_ok && y >= e0 && y < e1) {
            gt = E::to_f32(reinterpret_cast<const Raw*>(st)[y - e0]);
            gd = E::to_f32(reinterpret_cast<const Raw*>(sd)[y - e0]);
          }
          gt = __shfl_sync(kFull, gt, 0);
          gd = __shfl_sync(kFull, gd, 0);
        }
        float av = -INFINITY;
        int ai = 0x7FFFFFFF;
        if constexpr (kSample) {
          uint32_t seen = 0;
          if (lane == 0) {
            cp_async_wait_all();
            seen = sm.rejw[x.b & 3];
          }
          av = __uint_as_float(__shfl_sync(kFull, seen, 0));
        }
        if constexpr (kRelaxed) {
          uint32_t c = lane < kWarps ? sm.wcnt[lane] : 0u;
          c = __reduce_add_sync(kFull, c);
          ai = (int)c;
        }
        if constexpr (MODE == kDiag) {
          if (lane < kWarps) {
            av = sm.wamax[lane];
            ai = sm.wamaxi[lane];
          }
          warp_argmax_redux(av, ai);
        }
        push8(slot, a, za, d, zda, gt, gd, av, __int_as_float(ai));
      }
      cluster_sync();  // ---- exchange 1: (max, sum) of both rows
      ++xc;
      if (warp == 0) {
        float a = mb(slot, 0, -INFINITY), za = mb(slot, 1, 0.0f);
        float d = mb(slot, 2, -INFINITY), zda = mb(slot, 3, 0.0f);
        float zty = 0.0f, zdy = 0.0f;
        if constexpr (kSample) {
          const int yy = __shfl_sync(kFull, y, 0);
          const bool ok_y = __shfl_sync(kFull, (int)tok_ok, 0) != 0;
          const int own = (ok_y && !x.bonus) ? yy / P.L : 0;
          zty = sm.mbox[slot][own][4];
          zdy = sm.mbox[slot][own][5];
        }
        warp_combine_mz2(a, za, d, zda, s);
        uint32_t rrank = 0;
        if constexpr (kRelaxed) {
          uint32_t c = lane < S ? __float_as_uint(sm.mbox[slot][lane][7]) : 0u;
          rrank = __reduce_add_sync(kFull, c);  // rank of the drafted token in the whole row
        }
        if constexpr (MODE == kDiag) {
          float av = mb(slot, 6, -INFINITY);
          int ai = lane < S ? __float_as_int(sm.mbox[slot][lane][7]) : 0x7FFFFFFF;
          warp_argmax_redux(av, ai);
          if (lane == 0) sm.bci[5] = ai;  // y_hat, identical in every CTA
        }
        if (lane == 0) {
          const float Zt = za, Zd = zda;
          const float c1t = __fmul_rn(a, s), c1d = __fmul_rn(d, s);
          const bool valid = (Zt > 0.0f && Zt < INFINITY) && (!x.has_draft || (Zd > 0.0f && Zd < INFINITY));
          const float izt = __frcp_rn(Zt), izd = __frcp_rn(Zd);
          uint32_t flags = 0;
          int mode_c = 0;  // 0: overlap only, 1: residual draw, 2: draw from p, 3: invalid
          int acc = 1;
          if constexpr (kSample) {
            if (x.bonus) {
              mode_c = 2;
            } else if constexpr (kRelaxed) {
              // in the target's top-k and within delta of its largest log-probability
              const bool in_k = P.relax_k <= 0 || rrank < (uint32_t)P.relax_k;
              const float gap = __fmul_rn(__fsub_rn(rzy, a), P.inv_t);
              const bool in_d = !(P.relax_delta < INFINITY) || gap >= -P.relax_delta;
              acc = (tok_ok && in_k && in_d) ? 1 : 0;
              mode_c = acc ? 0 : 2;  // a rejection draws from the full target
              if (!tok_ok) flags |= kBadToken;
            } else {
              // u * q(y) <= p(y), with p(y), q(y) formed like the per-element values
              const float py = __fmul_rn(ex2(fmaf(zty, s, -c1t)), izt);
              const float qy = __fmul_rn(ex2(fmaf(zdy, s, -c1d)), izd);
              acc = (tok_ok && __fmul_rn(ua, qy) <= py) ? 1 : 0;
              mode_c = acc ? 0 : 1;
              if (!(ua >= 0.0f && ua < 1.0f)) flags |= kBadUniform;
              if (!tok_ok) flags |= kBadToken;
            }
            if (!(uf >= 0.0f && uf < 1.0f)) flags |= kBadUniform;
          }
          if (!valid) {
            flags |= kBadLogits;
            mode_c = 3;
          }
          int skip = 0;
          if constexpr (kSample) {
            // publish a rejection (the record will hold acc = 0), then skip a
            // draw that cannot be emitted: rank 0's reading of the row's word
            // decides for the whole cluster
            if (rank == 0 && !x.bonus && (mode_c == 1 || mode_c == 3 || (kRelaxed && mode_c == 2)))
              atomicMax(&P.rej[x.b], kRejBase - (uint32_t)x.k);
            const uint32_t seen = __float_as_uint(sm.mbox[slot][0][6]);
            if (seen > kRejBase - (uint32_t)x.k) {
              if (mode_c == 2) mode_c = 0;     // bonus of a row with a rejection
              else if (mode_c == 1) skip = 1;  // a later rejection: overlap partial only
            }
          }
          sm.bci[7] = skip;
          if (skip) sm.bci[2] = 0;
          if (flags && rank == 0 && P.status) atomicOr(P.status, flags);
          sm.bcf[0] = c1t;
          sm.bcf[1] = c1d;
          sm.bcf[2] = (x.has_draft && valid) ? c1d + __log2f(__fmul_rn(Zd, izt)) : 0.0f;  // c1d + log2(Z_d / Z_t)
          sm.bcf[3] = izt;
          sm.bcf[4] = __fmul_rn(Zt, izd);
          sm.bcf[5] = uf;
          if constexpr (MODE == kDiag) sm.bcf[6] = __log2f(Zt);
          sm.bci[0] = mode_c;
          sm.bci[1] = acc;
        }
      }
      __syncthreads();
      const float c1t = sm.bcf[0], c1d = sm.bcf[1], cd2 = sm.bcf[2], izt = sm.bcf[3], ratio = sm.bcf[4];
      const float ufin = sm.bcf[5];
      int mode_c = sm.bci[0];
      const int acc = sm.bci[1];
      const f32x2 CT = f2(-c1t, -c1t);

      if (mode_c == 0 || mode_c == 3) {
        // ---- pass C: overlap (and E2E S-mass) partials, no exchange ----
        float a = 0.0f, m2 = 0.0f, m3 = 0.0f;
        if (mode_c == 0 && ok && x.has_draft) {
          const f32x2 CD = f2(-cd2, -cd2);
          f32x2 a2 = f2(0.0f, 0.0f), g2 = f2(0.0f, 0.0f), k2 = f2(0.0f, 0.0f);
          for (int i = t_lo; i < t_hi; ++i) {
            f32x2 pt[PV / 2], pd[PV / 2], ep[PV / 2], gp[PV / 2], kp[PV / 2];
            E::pairs(st[i], pt);
            E::pairs(sd[i], pd);
#pragma unroll
            for (int h = 0; h < PV / 2; ++h) {
              float t0, t1, d0, d1;
              f2_split(f2_fma(pt[h], S2, CT), t0, t1);
              f2_split(f2_fma(pd[h], S2, CD), d0, d1);
              const float e0 = ex2(fminf(t0, d0)), e1 = ex2(fminf(t1, d1));
              ep[h] = f2(e0, e1);
              if constexpr (MODE == kE2E) gp[h] = f2(d0 < t0 ? e0 : 0.0f, d1 < t1 ? e1 : 0.0f);
              if constexpr (MODE == kDiag) {
                // Z_t p log2-terms, x_t = log2(Z_t p), x_d = log2(Z_t q):
                // e_t x_t (entropy) and e_t (x_t - x_d) (KL); a token with
                // p = 0 adds nothing (0 log 0 = 0)
                const float et0 = ex2(t0), et1 = ex2(t1);
                gp[h] = f2(et0 > 0.0f ? __fmul_rn(et0, t0) : 0.0f, et1 > 0.0f ? __fmul_rn(et1, t1) : 0.0f);
                kp[h] = f2(et0 > 0.0f ? __fmul_rn(et0, __fsub_rn(t0, d0)) : 0.0f,
                           et1 > 0.0f ? __fmul_rn(et1, __fsub_rn(t1, d1)) : 0.0f);
              }
            }
            a2 = f2_add(a2, psum(ep));
            if constexpr (MODE == kE2E || MODE == kDiag) g2 = f2_add(g2, psum(gp));
            if constexpr (MODE == kDiag) k2 = f2_add(k2, psum(kp));
          }
          a = f2_hsum(a2);
          if constexpr (MODE == kE2E || MODE == kDiag) m2 = f2_hsum(g2);
          if constexpr (MODE == kDiag) m3 = f2_hsum(k2);
        }
        a = warp_sum(a);
        if constexpr (MODE == kE2E || MODE == kDiag) m2 = warp_sum(m2);
        if constexpr (MODE == kDiag) m3 = warp_sum(m3);
        if (lane == 0) {
          sm.wred[warp][0] = a;
          sm.wred[warp][1] = m2;
          sm.wred[warp][2] = m3;
        }
        // p(y_hat) from the CTA whose slice holds y_hat, read before the
        // barrier: past it the other warps refill their segments
        float py_hat = -1.0f;
        if constexpr (MODE == kDiag) {
          const int yh = sm.bci[5];
          if (tid == 0 && mode_c == 0 && yh >= e0 && yh < e1) {
            const float zy = E::to_f32(reinterpret_cast<const Raw*>(st)[yh - e0]);
            py_hat = __fmul_rn(ex2(fmaf(zy, s, -c1t)), izt);
          }
        }
        __syncthreads();
        if (warp == 0) {
          float A = lane < kWarps ? sm.wred[lane][0] : 0.0f;
          float M2 = lane < kWarps ? sm.wred[lane][1] : 0.0f;
          float M3 = lane < kWarps ? sm.wred[lane][2] : 0.0f;
          A = warp_sum(A);
          if constexpr (MODE == kE2E || MODE == kDiag) M2 = warp_sum(M2);
          if constexpr (MODE == kDiag) M3 = warp_sum(M3);
          if (lane == 0) {
            const float nanv = __int_as_float(0x7FC00000);
            P.part[(long long)rec_idx(x) * kPartStride + rank] = (mode_c == 3) ? nanv : __fmul_rn(A, izt);
            if constexpr (MODE == kDiag) {
              // entropy partial sum_v p x_t; rank 0 folds in -log2 Z_t, so
              // that the rank-ordered sum is -H / ln 2
              float h2 = __fmul_rn(M2, izt);
              if (rank == 0) h2 = __fsub_rn(h2, sm.bcf[6]);
              P.part2[(long long)rec_idx(x) * kPartStride + rank] = (mode_c == 3) ? nanv : h2;
              P.part3[(long long)rec_idx(x) * kPartStride + rank] = (mode_c == 3) ? nanv : __fmul_rn(M3, izt);
              if (P.ato && py_hat >= 0.0f) P.ato[rec_idx(x)] = py_hat;
              if (P.ato && mode_c == 3 && rank == 0) P.ato[rec_idx(x)] = nanv;
            }
            if constexpr (MODE == kE2E) {
              P.part2[(long long)rec_idx(x) * kPartStride + rank] = (mode_c == 3) ? nanv : __fmul_rn(M2, izt);
              if (rank == 0) {
                E2EStats e2;
                e2.c1t = c1t;
                e2.cd = cd2;
                e2.izt = izt;
                e2.smass = e2.alpha = e2.b1 = e2.b0 = e2.pad = 0.0f;
                P.stats[rec_idx(x)] = e2;
              }
            }
            if constexpr (kSample) {
              if (rank == 0) {
                VerifyRecord r;
                r.acc = (mode_c == 3) ? 0 : acc;
                r.token = -1;
                r.pad0 = r.pad1 = 0;
                P.rec[rec_idx(x)] = r;
              }
            }
            queue_arrival(x.b);
          }
        }
        continue;
      }

      // ---- pass C': residual (mode 1) or target (mode 2) draw ----
      // Prefix order is (CTA, warp, lane, vector, element): every thread sums
      // its contiguous chunk in order, a warp scan orders the lanes, and the
      // warp of the owning thread walks that thread's chunk again with the
      // same per-element arithmetic, one vector per lane.
      const f32x2 CDd = f2(-c1d, -c1d);
      const f32x2 NR = f2(-ratio, -ratio);
      const bool skip = sm.bci[7] != 0;
      bool emptied = false;
      for (int attempt = 0; attempt < 2; ++attempt) {
        const bool resid = (mode_c == 1);
        float tot = 0.0f;
        f32x2 mm2 = f2(0.0f, 0.0f);
        // relaxed rejection: the overlap partial, element by element as pass C forms it
        const bool ralpha = kRelaxed && attempt == 0 && x.has_draft;
        const f32x2 CD = f2(-cd2, -cd2);
        if (ok) {
          for (int i = t_lo; i < t_hi; ++i) {
            float w[PV];
            const float rs = resid ? draw_weights<E, true>(st[i], sd[i], S2, CT, CDd, NR, w, mm2)
                                   : draw_weights<E, false>(st[i], st[i], S2, CT, CDd, NR, w, mm2);
            tot = __fadd_rn(tot, rs);
            if (ralpha) {
              f32x2 pt[PV / 2], pd[PV / 2], ep[PV / 2];
              E::pairs(st[i], pt);
              E::pairs(sd[i], pd);
#pragma unroll
              for (int h = 0; h < PV / 2; ++h) {
                float t0, t1, d0, d1;
                f2_split(f2_fma(pt[h], S2, CT), t0, t1);
                f2_split(f2_fma(pd[h], S2, CD), d0, d1);
                ep[h] = f2(ex2(fminf(t0, d0)), ex2(fminf(t1, d1)));
              }
              mm2 = f2_add(mm2, psum(ep));
            }
          }
        }
        const float incl = warp_incl_scan(tot, lane);
        float excl = __shfl_up_sync(kFull, incl, 1);
        if (lane == 0) excl = 0.0f;
        const float mm = warp_sum(f2_hsum(mm2));
        if (lane == 31) sm.wtot[warp] = incl;
        if (lane == 0) sm.wred[warp][0] = mm;
        __syncthreads();
        slot = xc & 1;
        if (warp == 0) {
          // warp offsets inside the CTA, the CTA total and the overlap partial
          const float wt = lane < kWarps ? sm.wtot[lane] : 0.0f;
          const float wincl = warp_incl_scan(wt, lane);
          if (lane < kWarps) sm.woff[lane + 1] = wincl;
          if (lane == 0) sm.woff[0] = 0.0f;
          const float ctot = __shfl_sync(kFull, wincl, kWarps - 1);
          float A = lane < kWarps ? sm.wred[lane][0] : 0.0f;
          A = warp_sum(A);
          if (lane == 0 && attempt == 0 && (resid || ralpha))
            P.part[(long long)rec_idx(x) * kPartStride + rank] = __fmul_rn(A, izt);
          if (!skip) push8(slot, ctot, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f);
        }
        // a later rejection keeps the overlap partial, computed with the
        // draw's arithmetic (bits independent of the skip), and draws nothing
        if (skip) break;
        cluster_sync();  // ---- exchange 2: CTA totals of the draw weights
        ++xc;
        if (warp == 0) {
          const float tr = mb(slot, 0, 0.0f);
          const float cincl = warp_incl_scan(tr, lane);
          const float total = __shfl_sync(kFull, cincl, 31);
          const float thr = __fmul_rn(ufin, total);
          const unsigned hit = __ballot_sync(kFull, lane < S && tr > 0.0f && cincl > thr);
          const unsigned pos = __ballot_sync(kFull, lane < S && tr > 0.0f);
          int owner = -1;
          bool fb = false;
          if (hit) {
            owner = __ffs(hit) - 1;
          } else if (pos) {
            owner = 31 - __clz(pos);
            fb = true;
          }
          const float cexcl = __shfl_up_sync(kFull, cincl, 1);
          const float ex_o = __shfl_sync(kFull, cexcl, owner > 0 ? owner : 0);
          if (lane == 0) {
            sm.bci[2] = (total > 0.0f) ? 1 : 0;
            sm.bci[3] = owner;
            sm.bcf[6] = fb ? INFINITY : __fadd_rn(thr, owner > 0 ? -ex_o : 0.0f);
          }
        }
        __syncthreads();
        if (!sm.bci[2]) {
          if (attempt == 0 && resid) {  // rejection with no residual mass (rounding): draw from p
            // reported by the row's completion if this position is the one emitted
            emptied = true;
            mode_c = 2;
            continue;
          }
          break;  // nothing to draw: the token stays -1
        }
        if (sm.bci[3] == (int)rank) {
          if (tid == 0) {
            // the warp holding the local threshold (warps with positive mass only)
            const float th = sm.bcf[6];
            int wsel = -1, wlast = -1;
            for (int w = 0; w < kWarps; ++w) {
              const bool posw = sm.wtot[w] > 0.0f;
              if (posw && wsel < 0 && sm.woff[w + 1] > th) wsel = w;
              if (posw) wlast = w;
            }
            float thw = INFINITY;
            if (wsel >= 0) {
              thw = __fadd_rn(th, -sm.woff[wsel]);
            } else {
              wsel = wlast;
            }
            sm.bci[4] = wsel;
            sm.bci[6] = -1;
            sm.bcf[7] = thw;
          }
          __syncthreads();
          if (warp == sm.bci[4]) {
            const float thw = sm.bcf[7];
            const unsigned hit = __ballot_sync(kFull, tot > 0.0f && incl > thw);
            const unsigned pos = __ballot_sync(kFull, tot > 0.0f);
            const bool fb = (hit == 0u);
            const int l = hit ? (__ffs(hit) - 1) : (pos ? 31 - __clz(pos) : -1);
            if (l >= 0) {
              // The whole warp walks thread l's chunk: lane k takes its k-th
              // vector, a warp scan orders the vector totals, and the lane
              // whose vector crosses the threshold walks its 8 weights.
              const float th = fb ? INFINITY : thw;
              const int o_lo = min(v_lo + l * cpt, v_hi);
              const int o_hi = min(o_lo + cpt, v_hi);
              float carry = __shfl_sync(kFull, excl, l);
              int pick = -1, ilast = -1;
              for (int base = o_lo; base < o_hi; base += 32) {
                const int i = base + lane;
                float w[PV];
                float rs = 0.0f;
                if (i < o_hi) {
                  f32x2 dummy = f2(0.0f, 0.0f);
                  rs = resid ? draw_weights<E, true>(st[i], sd[i], S2, CT, CDd, NR, w, dummy)
                             : draw_weights<E, false>(st[i], st[i], S2, CT, CDd, NR, w, dummy);
                }
                const float run = __fadd_rn(carry, warp_incl_scan(rs, lane));
                const float up = __shfl_up_sync(kFull, run, 1);
                const float before = (lane == 0) ? carry : up;
                const unsigned pos2 = __ballot_sync(kFull, rs > 0.0f);
                if (pos2) ilast = base + 31 - __clz(pos2);
                const unsigned h2 = __ballot_sync(kFull, rs > 0.0f && run > th);
                if (h2) {
                  const int k = __ffs(h2) - 1;
                  int pk = -1;
                  if (lane == k) {
                    float a = before;
                    int lastp = -1;
#pragma unroll
                    for (int j = 0; j < PV; ++j) {
                      a = __fadd_rn(a, w[j]);
                      if (w[j] > 0.0f) {
                        lastp = j;
                        if (pk < 0 && a > th) pk = j;
                      }
                    }
                    if (pk < 0) pk = lastp;  // the vector crosses but no element does (rounding)
                    pk = i * PV + pk;
                  }
                  pick = __shfl_sync(kFull, pk, k);
                  break;
                }
                carry = __shfl_sync(kFull, run, 31);
              }
              if (pick < 0 && ilast >= 0) {  // no crossing (rounding): the last positive weight
                if (lane == 0) {
                  float w[PV];
                  f32x2 dummy = f2(0.0f, 0.0f);
                  if (resid)
                    draw_weights<E, true>(st[ilast], sd[ilast], S2, CT, CDd, NR, w, dummy);
                  else
                    draw_weights<E, false>(st[ilast], st[ilast], S2, CT, CDd, NR, w, dummy);
#pragma unroll
                  for (int k = 0; k < PV; ++k)
                    if (w[k] > 0.0f) pick = ilast * PV + k;
                }
                pick = __shfl_sync(kFull, pick, 0);
              }
              if (lane == 0 && pick >= 0) sm.bci[6] = e0 + pick;
            }
          }
        }
        break;
      }
      __syncthreads();  // the owner thread's token reaches thread 0
      if (tid == 0) {
        if (rank == 0) {
          P.rec[rec_idx(x)].acc = (kSample && !x.bonus) ? (emptied ? 2 : acc) : 0;
          if (!sm.bci[2]) P.rec[rec_idx(x)].token = -1;
        }
        if (sm.bci[2] && sm.bci[3] == (int)rank) P.rec[rec_idx(x)].token = sm.bci[6];
        queue_arrival(x.b);
      }
    }
  }
  __syncthreads();
  if (warp == 0) flush();
  cluster_sync();  // no CTA leaves while a peer may still write to its mailbox
}

// ---- E2E-TV gradient: one streaming pass over both logit tensors ------------------

struct GradParams {
  const void* target;
  const void* draft;
  int B, K, KT, V;
  int units;
  int aligned;
  float s;
  const E2EStats* stats;
  float* grad;
};

template <class E>
__global__ void __launch_bounds__(256) e2e_grad_kernel(const GradParams P) {
  constexpr int PV = E::PV;
  const int V = P.V, K = P.K;
  for (int unit = blockIdx.y; unit < P.units; unit += gridDim.y) {
    const int b = unit / K, k = unit - b * K;
    const E2EStats st = P.stats[unit];
    const float s = P.s;
    const typename E::Raw* tg = reinterpret_cast<const typename E::Raw*>(P.target) + ((long long)b * P.KT + k) * V;
    const typename E::Raw* dg = reinterpret_cast<const typename E::Raw*>(P.draft) + (long long)unit * V;
    float* gg = P.grad + (long long)unit * V;
    if (P.aligned) {
      const int nvec = V / PV;
      const uint4* tv = reinterpret_cast<const uint4*>(tg);
      const uint4* dv = reinterpret_cast<const uint4*>(dg);
      for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < nvec; j += gridDim.x * blockDim.x) {
        float t[PV], d[PV], g[PV];
        E::unpack(__ldcs(tv + j), t);
        E::unpack(__ldcs(dv + j), d);
#pragma unroll
        for (int i = 0; i < PV; ++i) {
          const float xt = fmaf(t[i], s, -st.c1t);
          const float xd = fmaf(d[i], s, -st.cd);
          g[i] = __fmul_rn(ex2(xd), (xd < xt) ? st.b1 : st.b0);
        }
        float4* go = reinterpret_cast<float4*>(gg + (long long)j * PV);
#pragma unroll
        for (int i = 0; i < PV / 4; ++i) __stcs(go + i, make_float4(g[4 * i], g[4 * i + 1], g[4 * i + 2], g[4 * i + 3]));
      }
    } else {
      for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
        const float xt = fmaf(E::to_f32(tg[v]), s, -st.c1t);
        const float xd = fmaf(E::to_f32(dg[v]), s, -st.cd);
        gg[v] = __fmul_rn(ex2(xd), (xd < xt) ? st.b1 : st.b0);
      }
    }
  }
}

}  // namespace ssv
