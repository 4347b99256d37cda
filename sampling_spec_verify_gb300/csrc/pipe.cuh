// Pipelined vocabulary sweep for sm_103a.
//
// Work decomposition
// ------------------
// A "unit" is one (batch row b, position k): one target row of V logits and,
// for a drafted position, one draft row.  Each unit is cut into C chunks of at
// most Lc logits; a "task" is one chunk of one unit.  Tasks are numbered
// t = u * C + c and dealt round-robin to a persistent grid of G CTAs (one per
// SM, launched cooperatively so that every CTA is resident): CTA g runs tasks
// g, g + G, g + 2G, ...  Every logit is copied from HBM into shared memory
// exactly once, by a 1-D bulk (TMA) copy.
//
// Two passes over each chunk, both on the copy held in shared memory:
//   phase 1  softmax normalisers: per-thread sums of 2^(z s - c) (s = log2(e)/T)
//            for the target and draft rows (greedy: arg-maxima instead);
//   phase 2  with the unit's normalisers known: the overlap sum of min(p, q)
//            and, for units that draw a token (a rejected draft or the bonus
//            position), the draw weights max(0, p - q) or p, summed per
//            segment of 32 vectors.
// Phase 2 of a unit needs the phase-1 partials of all of its C chunks, which
// other CTAs compute.  All partials are published as self-validating words
// (each 32-bit field is stored bitwise inverted, so an all-zero field means
// "not written yet"; the workspace is zero between calls), which needs no
// memory fence or atomic on the per-task path.  Phase 2 of a task runs kLag
// tasks after its phase 1, by which time the other chunks of the unit are
// normally done: nothing on the data path waits for another CTA.
//
// Warp roles (one CTA)
// --------------------
//   warps 0..15  compute: phase 2 of task i - kLag, then phase 1 of task i;
//   warp 16      producer: bulk copies into a ring of D shared-memory stages;
//   warps 17..20 control: warp 17 + r serves the tasks i with i % 4 == r.  It
//                combines the compute warps' partials, publishes the task's
//                chunk partials, reads back the unit's partials, decides
//                acceptance (identically in every CTA of the unit) and
//                publishes phase-2 partials; the CTA holding a unit's
//                finalising chunk (u mod C) reads back the unit's phase-2
//                partials and hands the unit to the finaliser.  Four control warps keep four tasks'
//                round trips to L2 in flight at once;
//   warp 21      finaliser: sums the unit's phase-2 partials into alpha,
//                locates the inverse-CDF token (chunk -> segment -> vector ->
//                element, re-reading one 32-vector segment from L2), writes
//                the unit's record and completes batch rows (prefix-order
//                outcome, prefix products, E2E-TV loss), re-zeroing the
//                row's workspace.
// Warps hand work to each other through shared-memory mbarriers.  Every wait
// is bounded: on a timeout the kernel sets SPEC_DEV_TIMEOUT, raises an abort
// flag that ends every other wait at once, and runs to completion.
#pragma once

#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "elem.cuh"
#include "ptx.cuh"

namespace ssv {

constexpr int kCompWarps = 16;
constexpr int kCompThreads = kCompWarps * 32;
constexpr int kP1Warps = 8;  // T > 0: warps 0..7 run phase 1, warps 8..15 phase 2
constexpr int kP2Warps = kCompWarps - kP1Warps;
constexpr int kP1Threads = kP1Warps * 32;
constexpr int kP2Threads = kP2Warps * 32;
constexpr int kCtlWarps = 4;  // control warp r serves the tasks i with i % 4 == r
constexpr int kProducerWarp = kCompWarps;
constexpr int kControlWarp0 = kCompWarps + 1;
constexpr int kFinalWarp = kCompWarps + 1 + kCtlWarps;
constexpr int kThreads = (kFinalWarp + 1) * 32;
constexpr int kMaxStages = 16;
constexpr int kLag = 4;     // a control warp publishes task i - 4's phase-2 partials after task i's decision
constexpr int kSlots = 4;   // phase-1 hand-off slots (task i uses slot i % 4)
constexpr int kSlots2 = 8;  // decision / phase-2 hand-off slots (task i uses slot i % 8)
constexpr int kJobSlots = 8;
static_assert(kLag == kSlots && kCtlWarps == kSlots && kSlots2 == 2 * kSlots,
              "task i's control warp is i % 4; its decision slot stays live until task i + 4 is decided");
constexpr int kSegVecs = 32;  // 16-byte vectors per draw segment
constexpr int kMaxSegs = 32;  // segments per chunk in sampling modes
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait

constexpr uint32_t kBadToken = 1u, kBadLogits = 2u, kBadUniform = 4u, kTimeout = 8u, kEmptyResidual = 16u;

enum Mode : int { kVerify = 0, kVerifyGreedy = 1, kOverlap = 2, kOverlapGreedy = 3, kE2E = 4 };

// ctl[] words of the workspace
constexpr int kCtlLoss = 0;   // E2E rows completed
constexpr int kCtlAbort = 1;  // set by a timed-out wait
constexpr int kCtlExit = 2;   // CTAs finished

struct Rec {      // one per unit (verify, overlap)
  int32_t acc;    // 1 accepted, 0 rejected or invalid
  int32_t token;  // correction / bonus / greedy choice; -1 if none
  float alpha;
  uint32_t pad;
};

struct E2EStats {  // one per unit (E2E-TV); read by the gradient kernel
  float c1t;       // fl(M_t * s): exponent offset of the target row
  float cd;        // offset of the draft row with log2(Z_d / Z_t) folded in
  float izt;       // 1 / Z_t
  float smass;     // S = sum_{q_v < p_v} q_v
  float alpha;
  float b1, b0;    // gradient multipliers for indicator 1 / 0
  float pad;
};

struct PipeParams {
  const void* target;
  const void* draft;
  int B, K, KT, V;
  int units;
  int C;        // chunks per unit
  int Lc;       // chunk length in elements (multiple of the vector width)
  int D;        // shared-memory stages
  int stage;    // bytes per stage
  int doff;     // byte offset of the draft row inside a stage
  int aligned;  // rows start on 16-byte boundaries: bulk copies allowed
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
  // workspace
  uint64_t* part1;  // [units * C][4] tagged phase-1 words
  uint64_t* part2;  // [units * C] tagged phase-2 partials (alpha_c, R_c or S_c)
  uint32_t* seg;    // [units * C][kMaxSegs] tagged draw-weight segment totals (verify, T > 0)
  uint32_t* cnt;    // [units] chunks finished
  Rec* rec;         // [units] (verify, overlap)
  E2EStats* stats;  // [units] (E2E-TV)
  uint32_t* row_cnt;
  float* row_loss;
  uint32_t* ctl;
  uint8_t* ws;
  size_t ws_bytes;
  uint32_t* status;
};

// ---- tagged words -----------------------------------------------------------

__device__ __forceinline__ uint32_t tag_bits(uint32_t b) { return ~(b == 0xFFFFFFFFu ? 0x7FC00000u : b); }
__device__ __forceinline__ uint64_t tag2(float lo, float hi) {
  return (uint64_t)tag_bits(__float_as_uint(lo)) | ((uint64_t)tag_bits(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ uint64_t tag2i(float lo, int hi) {
  return (uint64_t)tag_bits(__float_as_uint(lo)) | ((uint64_t)tag_bits((uint32_t)hi) << 32);
}
__device__ __forceinline__ bool tag_ok(uint64_t w) { return (uint32_t)w != 0u && (uint32_t)(w >> 32) != 0u; }
__device__ __forceinline__ float tag_lo(uint64_t w) { return __uint_as_float(~(uint32_t)w); }
__device__ __forceinline__ float tag_hi(uint64_t w) { return __uint_as_float(~(uint32_t)(w >> 32)); }
__device__ __forceinline__ int tag_hi_i(uint64_t w) { return (int)~(uint32_t)(w >> 32); }

// ---- units and tasks ----------------------------------------------------------

template <class E>
struct UnitInfo {
  int b, k;
  bool bonus, has_d;
  const typename E::Raw* tg;
  const typename E::Raw* dg;
};

template <class E, int MODE>
__device__ __forceinline__ UnitInfo<E> unit_info(const PipeParams& P, int u) {
  UnitInfo<E> x;
  if constexpr (MODE == kVerify || MODE == kVerifyGreedy) {
    x.b = u / (P.K + 1);
    x.k = u - x.b * (P.K + 1);
    x.bonus = (x.k == P.K);
  } else {
    x.b = u / P.K;
    x.k = u - x.b * P.K;
    x.bonus = false;
  }
  x.has_d = !x.bonus;
  if constexpr (MODE == kVerifyGreedy) x.has_d = !x.bonus && P.alpha != nullptr;
  using Raw = typename E::Raw;
  x.tg = reinterpret_cast<const Raw*>(P.target) + ((long long)x.b * P.KT + x.k) * P.V;
  x.dg = x.has_d ? reinterpret_cast<const Raw*>(P.draft) + ((long long)x.b * P.K + x.k) * P.V : nullptr;
  return x;
}

struct TaskInfo {
  int u, c, e0, len, nv;
};

// The chunk whose CTA reads back a unit's partials and hands the unit to its
// finaliser.  u mod C spreads units over the CTAs: the last chunk would
// concentrate them on gcd(C, G) residues (8 CTAs when C = 19, G = 152).
__device__ __forceinline__ int fin_chunk(const PipeParams& P, int u) { return u % P.C; }

template <class E>
__device__ __forceinline__ TaskInfo task_info(const PipeParams& P, int t) {
  TaskInfo x;  // the host keeps units * C below 2^31
  x.u = t / P.C;
  x.c = t - x.u * P.C;
  x.e0 = x.c * P.Lc;
  x.len = min(P.Lc, P.V - x.e0);
  x.nv = (x.len + E::PV - 1) / E::PV;
  return x;
}

// ---- shared state -------------------------------------------------------------

struct Nrm {  // decision of one task's unit, written by the control warp
  float c1t, c1d, cd2, izt, uf;
  int mode;  // 0 overlap only, 1 residual draw, 2 draw from p (bonus), 3 invalid
  int acc;
  int unit;
};

struct StageDesc {  // the task held by a shared-memory stage, written by the producer
  int u, c, e0, nv;
  int has_d;
  int pad[3];
};

struct Job {  // a unit whose chunks are all finished, for the finaliser
  int unit, mode, acc, stop;
  float c1t, cd2, izt, uf;
};

struct PipeSmem {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t p1done[kSlots], p1free[kSlots], p2done[kSlots2], nrm_bar[kSlots2];
  uint64_t job_full[kJobSlots], job_empty[kJobSlots];
  float4 wp1[kSlots][kCompWarps];
  float wnan[kSlots][kCompWarps];
  float4 wp2[kSlots2][kP2Warps];
  Nrm nrm[kSlots2];
  StageDesc desc[kMaxStages];
  Job job[kJobSlots];
  int job_tail;
  int dead;
  int wipe;
};

// ---- bounded waits ------------------------------------------------------------------

__device__ __forceinline__ bool aborted(const PipeParams& P, const PipeSmem& sm) {
  return *(volatile const int*)&sm.dead != 0 || ld_relaxed_u32(P.ctl + kCtlAbort) != 0u;
}

__device__ __noinline__ void give_up(const PipeParams& P, PipeSmem& sm) {
  *(volatile int*)&sm.dead = 1;
  if (P.status) atomicOr(P.status, kTimeout);
  st_relaxed_u32(P.ctl + kCtlAbort, 1u);
}

// Waits for phase `parity` of an mbarrier; false after the time bound or once
// any wait of the grid has given up.  After two probes the warp sleeps
// between probes (64 ns, growing to 256 ns), and the abort flag (a global
// load) and the clock are looked at only every 64 probes: a waiting warp
// takes almost no issue slots from the warps of its SM that do work.
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const PipeParams& P, PipeSmem& sm) {
  if (mbar_test(bar, parity)) return true;
  uint64_t t0 = 0;
  uint32_t back = 64;
  for (uint32_t k = 1;; ++k) {
    if (mbar_probe(bar, parity)) return true;
    if (k >= 2) {
      __nanosleep(back);
      if (back < 256) back <<= 1;
    }
    if ((k & 63u) == 0u) {
      if (aborted(P, sm)) return false;
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitLimitNs) {
        give_up(P, sm);
        return false;
      }
    }
  }
}

// ---- per-element arithmetic ------------------------------------------------------

// Draw weights of one vector and their total (fixed association).  KIND 1:
// Z_t * max(0, p - q) = e_t - e_m with e_t = 2^(z_t s - c1t) and
// e_m = 2^min(z_t s - c1t, z_d s - cd2) = Z_t * min(p, q) (cd2 folds
// log2(Z_d / Z_t) in); e_m is added to `mn`.  Where p <= q the two exponents
// are the same value, so the weight is exactly 0.  KIND 2: Z_t * p = e_t.
// Phase 2 and the finaliser's walk call this same function, so both see
// bit-identical weights.
template <class E, int KIND>
__device__ __forceinline__ float vec_weights(const uint4& wt, const uint4& wd, f32x2 S2, f32x2 CT, f32x2 CD,
                                             float (&w)[E::PV], f32x2& mn) {
  constexpr int NP = E::PV / 2;
  f32x2 pt[NP], wp[NP];
  E::pairs(wt, pt);
  if constexpr (KIND == 1) {
    f32x2 pd[NP], mp[NP];
    E::pairs(wd, pd);
#pragma unroll
    for (int h = 0; h < NP; ++h) {
      float t0, t1, d0, d1;
      f2_split(f2_fma(pt[h], S2, CT), t0, t1);
      f2_split(f2_fma(pd[h], S2, CD), d0, d1);
      const float et0 = ex2(t0), et1 = ex2(t1);
      const float em0 = ex2(fminf(t0, d0)), em1 = ex2(fminf(t1, d1));
      const float r0 = __fsub_rn(et0, em0), r1 = __fsub_rn(et1, em1);
      wp[h] = f2(r0, r1);
      mp[h] = f2(em0, em1);
      w[2 * h] = r0;
      w[2 * h + 1] = r1;
    }
    mn = f2_add(mn, psum(mp));
  } else {
#pragma unroll
    for (int h = 0; h < NP; ++h) {
      float t0, t1;
      f2_split(f2_fma(pt[h], S2, CT), t0, t1);
      const float e0 = ex2(t0), e1 = ex2(t1);
      wp[h] = f2(e0, e1);
      w[2 * h] = e0;
      w[2 * h + 1] = e1;
    }
  }
  return f2_hsum(psum(wp));
}

// Per-thread (max, sum) of one row with a running maximum: the slow path for
// threads whose fast sum overflowed or met an infinity / NaN.  Returns
// (max, sum) by value so that the callers' variables stay in registers.
template <class E>
__device__ __noinline__ float2 row_sum_slow(const uint4* base, int j, int nv, float s, int stride) {
  constexpr int PV = E::PV;
  const f32x2 S2 = f2(s, s);
  float m = -INFINITY;
  float z = 0.0f;
  float cm = 0.0f;
  for (int v = j; v < nv; v += stride) {
    const uint4 w = base[v];
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
  return make_float2(m, z);
}

// Phase 1 (T > 0): per-thread (max, sum) of the target and draft rows over
// the vectors j, j + stride, ... of the chunk.  The sum is taken relative to
// fl(s * max of the thread's first vector); a sum that is not below 2^100
// (a much larger value later, an infinity or a NaN) is redone by the slow path.
template <class E, int kStride>
__device__ __forceinline__ void phase1_sample(const uint4* st, const uint4* sd, bool has_d, int j, int nv, float s,
                                              float& mt, float& zt, float& md, float& zd) {
  constexpr int NP = E::PV / 2;
  mt = md = -INFINITY;
  zt = zd = 0.0f;
  if (j >= nv) return;
  const f32x2 S2 = f2(s, s);
  mt = E::vmax(st[j]);
  const float ct = __fmul_rn(mt, s);
  const f32x2 CT = f2(-ct, -ct);
  f32x2 at = f2(0.0f, 0.0f);
  if (has_d) {
    md = E::vmax(sd[j]);
    const float cd = __fmul_rn(md, s);
    const f32x2 CD = f2(-cd, -cd);
    f32x2 ad = f2(0.0f, 0.0f);
#pragma unroll 2
    for (int v = j; v < nv; v += kStride) {
      f32x2 et[NP], ed[NP];
      exp_pairs<E>(st[v], S2, CT, et);
      exp_pairs<E>(sd[v], S2, CD, ed);
      at = f2_add(at, psum(et));
      ad = f2_add(ad, psum(ed));
    }
    zd = f2_hsum(ad);
    if (!(zd < 0x1p100f) || !(cd > -INFINITY)) {
      const float2 r = row_sum_slow<E>(sd, j, nv, s, kStride);
      md = r.x;
      zd = r.y;
    }
  } else {
#pragma unroll 4
    for (int v = j; v < nv; v += kStride) {
      f32x2 et[NP];
      exp_pairs<E>(st[v], S2, CT, et);
      at = f2_add(at, psum(et));
    }
  }
  zt = f2_hsum(at);
  if (!(zt < 0x1p100f) || !(ct > -INFINITY)) {
    const float2 r = row_sum_slow<E>(st, j, nv, s, kStride);
    mt = r.x;
    zt = r.y;
  }
}

// Phase 1 (T == 0): per-thread arg-maximum of one row (smallest index on ties).
template <class E>
__device__ __forceinline__ void phase1_greedy_row(const uint4* base, int j, int nv, int e0, float& best, int& idx,
                                                  bool& nan_seen) {
  constexpr int PV = E::PV;
  best = -INFINITY;
  int jb = -1;
  for (int v = j; v < nv; v += kCompThreads) {  // greedy: all compute warps
    bool nn;
    const float vm = E::vmax_nan(base[v], nn);
    nan_seen |= nn;
    if (vm > best) {
      best = vm;
      jb = v;
    }
  }
  idx = 0x7FFFFFFF;
  if (jb >= 0) {
    float x[PV];
    E::unpack(base[jb], x);
#pragma unroll
    for (int i = PV - 1; i >= 0; --i)
      if (x[i] == best) idx = e0 + jb * PV + i;
  }
}

// Phase 2 (T > 0) of one chunk for one thread.  mode 0: A = Z_t * sum min(p, q)
// (and, for E2E-TV, Sm = Z_t * sum_{q < p} q) with one exp per element.
// mode 1 / 2: draw weights per vector; the total of every 32-vector segment
// is stored to seg[] by lane 0 of the warp that covers it, R = the warp's
// segment totals in order (lane 0), and A the min mass (mode 1).
template <class E, int MODE>
__device__ __forceinline__ void phase2_sample(const uint4* st, const uint4* sd, int j, int wi, int lane, int nv,
                                              int mode, float s, float c1t, float cd2, uint32_t* seg, float& A,
                                              float& R, float& Sm) {
  constexpr int NP = E::PV / 2;
  A = R = Sm = 0.0f;
  if (mode == 3) return;
  const f32x2 S2 = f2(s, s), CT = f2(-c1t, -c1t), CD = f2(-cd2, -cd2);
  if (mode == 0) {
    f32x2 a2 = f2(0.0f, 0.0f), g2 = f2(0.0f, 0.0f);
#pragma unroll 2
    for (int v = j; v < nv; v += kP2Threads) {
      f32x2 pt[NP], pd[NP], ep[NP], gp[NP];
      E::pairs(st[v], pt);
      E::pairs(sd[v], pd);
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        float t0, t1, d0, d1;
        f2_split(f2_fma(pt[h], S2, CT), t0, t1);
        f2_split(f2_fma(pd[h], S2, CD), d0, d1);
        const float e0 = ex2(fminf(t0, d0)), e1 = ex2(fminf(t1, d1));
        ep[h] = f2(e0, e1);
        if constexpr (MODE == kE2E) gp[h] = f2(d0 < t0 ? e0 : 0.0f, d1 < t1 ? e1 : 0.0f);
      }
      a2 = f2_add(a2, psum(ep));
      if constexpr (MODE == kE2E) g2 = f2_add(g2, psum(gp));
    }
    A = f2_hsum(a2);
    if constexpr (MODE == kE2E) Sm = f2_hsum(g2);
    return;
  }
  if constexpr (MODE == kVerify) {
    const int rounds = (nv + kP2Threads - 1) / kP2Threads;
    f32x2 mn = f2(0.0f, 0.0f);
    float racc = 0.0f;
    for (int r = 0; r < rounds; ++r) {
      const int v = r * kP2Threads + j;
      float tot = 0.0f;
      if (v < nv) {
        float w[E::PV];
        tot = (mode == 1) ? vec_weights<E, 1>(st[v], sd[v], S2, CT, CD, w, mn)
                          : vec_weights<E, 2>(st[v], st[v], S2, CT, CD, w, mn);
      }
      const float segt = warp_sum(tot);
      if (lane == 0) {
        const int s0 = r * kP2Threads + wi * kSegVecs;
        if (s0 < nv) st_relaxed_u32(seg + s0 / kSegVecs, tag_bits(__float_as_uint(segt)));
        racc = __fadd_rn(racc, segt);
      }
    }
    A = f2_hsum(mn);
    R = racc;
  }
}

// ---- warp helpers for the finaliser -------------------------------------------------

// Inverse-CDF selection over n non-negative weights in order, 32 per step:
// the first index whose running sum exceeds thr (weights > 0 only), with
// rem = thr - (running sum before it).  If rounding leaves no crossing, the
// last positive index and rem = +inf.  -1 if no weight is positive.  get(i)
// is called by every lane with its index (i < n).
template <class F>
__device__ __forceinline__ int scan_select(int n, float thr, float& rem, int lane, F get) {
  float carry = 0.0f;
  int lastpos = -1;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float x = (i < n) ? get(i) : 0.0f;
    const float run = __fadd_rn(carry, warp_incl_scan(x, lane));
    const float up = __shfl_up_sync(kFull, run, 1);
    const float before = (lane == 0) ? carry : up;
    const unsigned hit = __ballot_sync(kFull, x > 0.0f && run > thr);
    if (hit) {
      const int l = __ffs(hit) - 1;
      rem = __fsub_rn(thr, __shfl_sync(kFull, before, l));
      return base + l;
    }
    const unsigned pos = __ballot_sync(kFull, x > 0.0f);
    if (pos) lastpos = base + 31 - __clz(pos);
    carry = __shfl_sync(kFull, run, 31);
  }
  rem = INFINITY;
  return lastpos;
}

// Waits (bounded) until ok() holds in every lane, calling reload() in the
// lanes where it does not; gives up after the time bound or once the grid has
// aborted.  Used for the self-validating words written by other CTAs.
__device__ __noinline__ void give_up_global(const PipeParams& P) {
  if (P.status) atomicOr(P.status, kTimeout);
  st_relaxed_u32(P.ctl + kCtlAbort, 1u);
}

template <class Ok, class Reload>
__device__ __forceinline__ bool poll_words(const PipeParams& P, int lane, Ok ok, Reload reload) {
  if (__all_sync(kFull, ok())) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t back = 32;
  for (;;) {
    __nanosleep(back);
    if (back < 512) back <<= 1;
    if (!ok()) reload();
    if (__all_sync(kFull, ok())) return true;
    int stop = 0;
    if (lane == 0) {
      if (ld_relaxed_u32(P.ctl + kCtlAbort) != 0u) {
        stop = 1;
      } else if (global_timer_ns() - t0 > kWaitLimitNs) {
        give_up_global(P);
        stop = 1;
      }
    }
    if (__shfl_sync(kFull, stop, 0)) return false;
  }
}

// One vector of a row read from global memory (L2): 16-byte load when rows
// are aligned, element loads padded with -inf otherwise.
template <class E>
__device__ __forceinline__ uint4 load_vec(const typename E::Raw* row, int e, int V, bool aligned) {
  if (aligned) return __ldcg(reinterpret_cast<const uint4*>(row + e));
  using Raw = typename E::Raw;
  Raw x[E::PV];
#pragma unroll
  for (int i = 0; i < E::PV; ++i) x[i] = (e + i < V) ? row[e + i] : E::kNegInf;
  uint4 w;
  memcpy(&w, x, 16);
  return w;
}

// Draw one token of unit `ui` from its weights (KIND 1 residual, 2 target)
// given chunk totals get_c(c), threshold thr; seg != nullptr selects the
// stored segment totals, otherwise the chosen chunk is walked segment by
// segment.  Returns the token (all lanes) or -1.
template <class E, int KIND, class F>
__device__ int draw_token(const PipeParams& P, const UnitInfo<E>& ui, int u, float thr, float c1t, float cd2,
                          int lane, F get_c) {
  constexpr int PV = E::PV;
  float rem;
  const int cs = scan_select(P.C, thr, rem, lane, get_c);
  if (cs < 0) return -1;
  const int e0 = cs * P.Lc;
  const int len = min(P.Lc, P.V - e0);
  const int nv = (len + PV - 1) / PV;
  const int nseg = (nv + kSegVecs - 1) / kSegVecs;
  const f32x2 S2 = f2(P.s, P.s), CT = f2(-c1t, -c1t), CD = f2(-cd2, -cd2);
  const bool al = P.aligned != 0;
  auto weights = [&](int vi, float (&w)[PV]) {
    f32x2 dummy = f2(0.0f, 0.0f);
    if (vi >= nv) {
#pragma unroll
      for (int k = 0; k < PV; ++k) w[k] = 0.0f;
      return 0.0f;
    }
    const int e = e0 + vi * PV;
    const uint4 wt = load_vec<E>(ui.tg, e, P.V, al);
    if constexpr (KIND == 1) {
      const uint4 wd = load_vec<E>(ui.dg, e, P.V, al);
      return vec_weights<E, 1>(wt, wd, S2, CT, CD, w, dummy);
    } else {
      return vec_weights<E, 2>(wt, wt, S2, CT, CD, w, dummy);
    }
  };
  int sel_seg = -1;
  float rem2 = INFINITY;
  float w[PV];
  float tot = 0.0f;
  const uint32_t* segs = (P.seg != nullptr) ? P.seg + ((long long)u * P.C + cs) * kMaxSegs : nullptr;
  if (segs != nullptr) {
    // the chunk's segment totals (nseg <= 32: one per lane), once all are written
    uint32_t wv = ~0u;
    if (lane < nseg) wv = ld_relaxed_u32(segs + lane);
    poll_words(P, lane, [&]() { return wv != 0u; }, [&]() { wv = ld_relaxed_u32(segs + lane); });
    const float sv = (lane < nseg) ? __uint_as_float(~wv) : 0.0f;
    sel_seg = scan_select(nseg, rem, rem2, lane, [&](int) { return sv; });
    if (sel_seg < 0) return -1;
    tot = weights(sel_seg * kSegVecs + lane, w);
  } else {
    // walk the chunk one segment at a time
    float carry = 0.0f;
    int last_seg = -1;
    float last_tot = 0.0f;
    float lw[PV];
    for (int sg = 0; sg < nseg; ++sg) {
      float ww[PV];
      const float t = weights(sg * kSegVecs + lane, ww);
      const float st = warp_sum(t);
      if (st > 0.0f) {
        last_seg = sg;
        last_tot = t;
#pragma unroll
        for (int k = 0; k < PV; ++k) lw[k] = ww[k];
      }
      const float nxt = __fadd_rn(carry, st);
      if (st > 0.0f && nxt > rem) {
        sel_seg = sg;
        rem2 = __fsub_rn(rem, carry);
        tot = t;
#pragma unroll
        for (int k = 0; k < PV; ++k) w[k] = ww[k];
        break;
      }
      carry = nxt;
    }
    if (sel_seg < 0) {
      if (last_seg < 0) return -1;
      sel_seg = last_seg;
      rem2 = INFINITY;
      tot = last_tot;
#pragma unroll
      for (int k = 0; k < PV; ++k) w[k] = lw[k];
    }
  }
  float rem3;
  const int l = scan_select(32, rem2, rem3, lane, [&](int) { return tot; });
  if (l < 0) return -1;
  int pick = -1;
  if (lane == l) {
    float run = 0.0f;
    int lastp = -1;
#pragma unroll
    for (int k = 0; k < PV; ++k) {
      run = __fadd_rn(run, w[k]);
      if (w[k] > 0.0f) {
        lastp = k;
        if (pick < 0 && run > rem3) pick = k;
      }
    }
    if (pick < 0) pick = lastp;
    pick = (pick < 0) ? -1 : e0 + (sel_seg * kSegVecs + l) * PV + pick;
  }
  return __shfl_sync(kFull, pick, l);
}

// ---- row completion (finaliser warp) -----------------------------------------------
// Decides the prefix-order outcome of row b from its unit records, writes the
// row's outputs and re-zeroes the part of the workspace that the row used.
template <class E, int MODE>
__device__ __noinline__ void complete_row(const PipeParams& P, int b, int lane) {
  constexpr bool kVerifyMode = (MODE == kVerify || MODE == kVerifyGreedy);
  const int K = P.K;
  const int per_row = kVerifyMode ? K + 1 : K;
  const int u0 = b * per_row;
  if constexpr (kVerifyMode) {
    const Rec* rr = P.rec + u0;
    int nacc = K;
    for (int base = 0; base < K; base += 32) {
      const int kk = base + lane;
      const bool rej = (kk < K) && (__ldcg(&rr[kk].acc) == 0);
      const unsigned m = __ballot_sync(kFull, rej);
      if (m) {
        nacc = base + __ffs(m) - 1;
        break;
      }
    }
    const int corr = __ldcg(&rr[nacc].token);
    for (int kk = lane; kk <= K; kk += 32) {
      int tokv = -1;
      if (kk < nacc) tokv = P.draft_tokens[b * K + kk];
      else if (kk == nacc) tokv = corr;
      P.out_tokens[(long long)b * (K + 1) + kk] = tokv;
      if (kk < K && P.alpha) P.alpha[b * K + kk] = __ldcg(&rr[kk].alpha);
    }
    if (lane == 0) P.n_accepted[b] = nacc;
  } else if constexpr (MODE == kOverlap || MODE == kOverlapGreedy) {
    const Rec* rr = P.rec + u0;
    float al[2];
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      al[h] = (kk < K) ? __ldcg(&rr[kk].alpha) : 0.0f;
      if (kk < K) {
        P.alpha[b * K + kk] = al[h];
        if (P.tv) P.tv[b * K + kk] = 1.0f - al[h];
      }
    }
    float pr = 1.0f, sum = 0.0f;
    for (int kk = 0; kk < K; ++kk) {
      const float a = __shfl_sync(kFull, al[kk >> 5], kk & 31);
      pr = __fmul_rn(pr, a);
      sum = __fadd_rn(sum, pr);
      if (lane == 0 && P.surv) P.surv[b * K + kk] = pr;
    }
    if (lane == 0 && P.exp_acc) P.exp_acc[b] = sum;
  } else {  // kE2E
    E2EStats* sr = P.stats + u0;
    float al[2], sm2[2];
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      al[h] = (kk < K) ? __ldcg(&sr[kk].alpha) : 0.0f;
      sm2[h] = (kk < K) ? __ldcg(&sr[kk].smass) : 0.0f;
      if (kk < K && P.alpha) P.alpha[b * K + kk] = al[h];
    }
    // prefix products P_{k-1} and suffix sums G_k = 1 + alpha_{k+1} G_{k+1}
    float pre[2] = {1.0f, 1.0f}, suf[2] = {1.0f, 1.0f};
    float pr = 1.0f, rowl = 0.0f;
    for (int kk = 0; kk < K; ++kk) {
      if ((kk & 31) == lane) pre[kk >> 5] = pr;
      pr = __fmul_rn(pr, __shfl_sync(kFull, al[kk >> 5], kk & 31));
      rowl = __fadd_rn(rowl, pr);
    }
    float gsuf = 1.0f;
    for (int kk = K - 1; kk >= 0; --kk) {
      if ((kk & 31) == lane) suf[kk >> 5] = gsuf;
      gsuf = fmaf(__shfl_sync(kFull, al[kk >> 5], kk & 31), gsuf, 1.0f);
    }
    const float scale = P.grad_scale / (float)P.B;
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      if (kk < K) {
        const float coef = __fmul_rn(__fmul_rn(scale, pre[h]), suf[h]);
        const float A = __fmul_rn(__fmul_rn(coef, __ldcg(&sr[kk].izt)), P.inv_t);
        sr[kk].b1 = __fmul_rn(A, 1.0f - sm2[h]);
        sr[kk].b0 = __fmul_rn(A, -sm2[h]);
      }
    }
    if (lane == 0) P.row_loss[b] = rowl;
  }
  // re-zero the row's workspace
  __syncwarp();
  const long long nw = (long long)per_row * P.C;
  uint64_t* p1 = P.part1 + (long long)u0 * P.C * 4;
  for (long long i = lane; i < nw * 4; i += 32) p1[i] = 0ull;
  uint64_t* p2 = P.part2 + (long long)u0 * P.C;
  for (long long i = lane; i < nw; i += 32) p2[i] = 0ull;
  if (P.seg) {
    uint32_t* sg = P.seg + (long long)u0 * P.C * kMaxSegs;
    for (long long i = lane; i < nw * kMaxSegs; i += 32) sg[i] = 0u;
  }
  for (int i = lane; i < per_row; i += 32) {
    P.cnt[u0 + i] = 0u;
    if (P.rec) P.rec[u0 + i] = Rec{0, 0, 0.0f, 0u};
  }
  __syncwarp();
  if constexpr (MODE == kE2E) {
    int glast = 0;
    if (lane == 0) {
      P.row_cnt[b] = 0u;
      __threadfence();
      const uint32_t old = atomicAdd(P.ctl + kCtlLoss, 1u);
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
        P.ctl[kCtlLoss] = 0u;
      }
    }
  } else {
    if (lane == 0) P.row_cnt[b] = 0u;
  }
}

// ---- finaliser: one unit -------------------------------------------------------------

template <class E, int MODE>
__device__ __noinline__ void finalize_unit(const PipeParams& P, const Job& jb, int lane) {
  constexpr bool kGreedy = (MODE == kVerifyGreedy || MODE == kOverlapGreedy);
  constexpr bool kVerifyMode = (MODE == kVerify || MODE == kVerifyGreedy);
  const int u = jb.unit;
  const UnitInfo<E> ui = unit_info<E, MODE>(P, u);
  const int C = P.C;
  uint32_t flags = 0;
  // wait until every chunk of the unit has published its words (phase-1
  // arg-maxima at T == 0, phase-2 partials otherwise)
  for (int base = 0; base < C; base += 32) {
    const int c = base + lane;
    const uint64_t* w = kGreedy ? P.part1 + ((long long)u * C + c) * 4 : P.part2 + (long long)u * C + c;
    uint64_t a0 = ~0ull, a1 = ~0ull, a2 = ~0ull;  // each word is validated on its own
    auto load = [&]() {
      a0 = (c < C) ? ld_relaxed_u64(w) : ~0ull;
      if (kGreedy) {
        a1 = (c < C) ? ld_relaxed_u64(w + 1) : ~0ull;
        a2 = (c < C) ? ld_relaxed_u64(w + 2) : ~0ull;
      }
    };
    load();
    poll_words(P, lane, [&]() { return tag_ok(a0) && tag_ok(a1) && tag_ok(a2); }, load);
  }
  if constexpr (kGreedy) {
    // arg-maxima of the chunks, in chunk order
    float bt = -INFINITY, bd = -INFINITY, nn = 0.0f;
    int it = 0x7FFFFFFF, id = 0x7FFFFFFF;
    for (int c = lane; c < C; c += 32) {
      const uint64_t* w = P.part1 + ((long long)u * C + c) * 4;
      const uint64_t w0 = __ldcg(w), w2 = __ldcg(w + 2);
      const float vt = tag_lo(w0);
      const int xt = tag_hi_i(w0);
      if (vt > bt || (vt == bt && xt < it)) {
        bt = vt;
        it = xt;
      }
      if (ui.has_d) {
        const uint64_t w1 = __ldcg(w + 1);
        const float vd = tag_lo(w1);
        const int xd = tag_hi_i(w1);
        if (vd > bd || (vd == bd && xd < id)) {
          bd = vd;
          id = xd;
        }
      }
      nn = fmaxf(nn, tag_lo(w2));
    }
    warp_argmax_redux(bt, it);
    warp_argmax_redux(bd, id);
    nn = redux_max_f32(nn);
    if (lane == 0) {
      const bool bad = nn != 0.0f || !(bt < INFINITY) || it == 0x7FFFFFFF ||
                       (ui.has_d && (!(bd < INFINITY) || id == 0x7FFFFFFF));
      if (bad) flags |= kBadLogits;
      const int am_t = bad ? -1 : it;
      const float al = ui.has_d ? ((am_t >= 0 && am_t == id) ? 1.0f : 0.0f) : 0.0f;
      Rec r{0, -1, al, 0u};
      if constexpr (kVerifyMode) {
        const int y = ui.bonus ? -1 : P.draft_tokens[ui.b * P.K + ui.k];
        const bool tok_ok = ui.bonus || (y >= 0 && y < P.V);
        if (!tok_ok) flags |= kBadToken;
        r.acc = (!ui.bonus && tok_ok && y == am_t) ? 1 : 0;
        r.token = am_t;
      }
      P.rec[u] = r;
    }
  } else {
    // phase-2 partials of the chunks: alpha_c and R_c (E2E-TV: S_c)
    float a = 0.0f, r2 = 0.0f;
    for (int c = lane; c < C; c += 32) {
      const uint64_t w = __ldcg(P.part2 + (long long)u * C + c);
      a = __fadd_rn(a, tag_lo(w));
      r2 = __fadd_rn(r2, tag_hi(w));
    }
    const float alpha = warp_sum(a);
    const float tot2 = warp_sum(r2);
    if constexpr (MODE == kVerify) {
      int token = -1;
      if (jb.mode == 1 || jb.mode == 2) {
        auto get_r = [&](int c) { return tag_hi(__ldcg(P.part2 + (long long)u * C + c)); };
        if (tot2 > 0.0f) {
          const float thr = __fmul_rn(jb.uf, tot2);
          token = (jb.mode == 1) ? draw_token<E, 1>(P, ui, u, thr, jb.c1t, jb.cd2, lane, get_r)
                                 : draw_token<E, 2>(P, ui, u, thr, jb.c1t, jb.cd2, lane, get_r);
        } else if (jb.mode == 1) {
          // rejection with no residual mass (rounding only): draw from p, with
          // the chunk masses of p from the phase-1 partials
          flags |= kEmptyResidual;
          auto get_p = [&](int c) {
            const uint64_t w0 = __ldcg(P.part1 + ((long long)u * C + c) * 4);
            const float m = tag_lo(w0), z = tag_hi(w0);
            return (m > -INFINITY) ? __fmul_rn(z, ex2(__fadd_rn(__fmul_rn(m, P.s), -jb.c1t))) : 0.0f;
          };
          float pt = 0.0f;
          for (int c = lane; c < C; c += 32) pt = __fadd_rn(pt, get_p(c));
          pt = warp_sum(pt);
          PipeParams Q = P;
          Q.seg = nullptr;  // walk the chosen chunk segment by segment
          token = draw_token<E, 2>(Q, ui, u, __fmul_rn(jb.uf, pt), jb.c1t, jb.cd2, lane, get_p);
        }
      }
      if (lane == 0) {
        Rec r;
        r.acc = (jb.mode == 0) ? 1 : 0;
        r.token = token;
        r.alpha = ui.bonus ? 0.0f : alpha;
        r.pad = 0u;
        P.rec[u] = r;
      }
    } else if constexpr (MODE == kOverlap) {
      if (lane == 0) P.rec[u] = Rec{0, -1, alpha, 0u};
    } else {  // kE2E
      if (lane == 0) {
        E2EStats e2;
        e2.c1t = jb.c1t;
        e2.cd = jb.cd2;
        e2.izt = jb.izt;
        e2.smass = tot2;
        e2.alpha = alpha;
        e2.b1 = e2.b0 = e2.pad = 0.0f;
        P.stats[u] = e2;
      }
    }
  }
  // arrival on the row; the last one completes it
  int last = 0;
  if (lane == 0) {
    if (flags && P.status) atomicOr(P.status, flags);
    __threadfence();
    const int per_row = kVerifyMode ? P.K + 1 : P.K;
    const uint32_t old = atomicAdd(P.row_cnt + ui.b, 1u);
    last = (old == (uint32_t)per_row - 1) ? 1 : 0;
    if (last) __threadfence();
  }
  last = __shfl_sync(kFull, last, 0);
  if (last) complete_row<E, MODE>(P, ui.b, lane);
}

// ---- the kernel ------------------------------------------------------------------

template <class E, int MODE>
__global__ void __launch_bounds__(kThreads, 1) pipe_kernel(const __grid_constant__ PipeParams P) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(16) PipeSmem sm;

  constexpr int PV = E::PV;
  using Raw = typename E::Raw;
  constexpr bool kGreedy = (MODE == kVerifyGreedy || MODE == kOverlapGreedy);
  constexpr bool kSample = !kGreedy;
  constexpr int kP1Count = kGreedy ? kCompWarps : kP1Warps;     // warps running phase 1
  constexpr int kRelease = kGreedy ? kCompWarps : kP2Warps;     // warps releasing a stage

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, G = gridDim.x;
  const long long T = (long long)P.units * P.C;
  const int n = (g < T) ? (int)((T - 1 - g) / G + 1) : 0;
  const int D = P.D;
  const float s = P.s;

  if (threadIdx.x == 0) {
    for (int d = 0; d < D; ++d) {
      mbar_init(smem_addr(&sm.full[d]), 1);
      mbar_init(smem_addr(&sm.empty[d]), kRelease);
    }
    for (int h = 0; h < kSlots; ++h) {
      mbar_init(smem_addr(&sm.p1done[h]), kP1Count);
      mbar_init(smem_addr(&sm.p1free[h]), 1);
    }
    for (int h = 0; h < kSlots2; ++h) {
      mbar_init(smem_addr(&sm.p2done[h]), kP2Warps);
      mbar_init(smem_addr(&sm.nrm_bar[h]), 1);
    }
    for (int q = 0; q < kJobSlots; ++q) {
      mbar_init(smem_addr(&sm.job_full[q]), 1);
      mbar_init(smem_addr(&sm.job_empty[q]), 1);
    }
    sm.job_tail = 0;
    sm.dead = 0;
    sm.wipe = 0;
    fence_mbar_init();
  }
  __syncthreads();

  auto stage_t = [&](int i) { return reinterpret_cast<const uint4*>(stage_mem + (size_t)(i % D) * P.stage); };
  auto stage_d = [&](int i) {
    return reinterpret_cast<const uint4*>(stage_mem + (size_t)(i % D) * P.stage + P.doff);
  };
  auto task_of = [&](int i) { return task_info<E>(P, g + i * G); };
  // the k-th use of a slot (task i = slots * k + slot) completes phase k of its barriers
  auto par = [](int i) { return (uint32_t)(i / kSlots) & 1u; };
  auto par2 = [](int i) { return (uint32_t)(i / kSlots2) & 1u; };

  if (warp < kCompWarps && (kGreedy || warp < kP1Warps)) {
    // ================= phase-1 warps =================
    const int j = warp * 32 + lane;
    for (int i = 0; i < n; ++i) {
      const int slot = i % kSlots;
      pwait(smem_addr(&sm.full[i % D]), (uint32_t)(i / D) & 1u, P, sm);
      const StageDesc dsc = sm.desc[i % D];
      float4 part;
      float nanw = 0.0f;
      if constexpr (kSample) {
        float mt, zt, md, zd;
        phase1_sample<E, kP1Threads>(stage_t(i), stage_d(i), dsc.has_d != 0, j, dsc.nv, s, mt, zt, md, zd);
        warp_combine_mz2(mt, zt, md, zd, s);
        part = make_float4(mt, zt, md, zd);
      } else {
        float bt, bd = -INFINITY;
        int it, id = 0x7FFFFFFF;
        bool nn = false;
        phase1_greedy_row<E>(stage_t(i), j, dsc.nv, dsc.e0, bt, it, nn);
        if (dsc.has_d) phase1_greedy_row<E>(stage_d(i), j, dsc.nv, dsc.e0, bd, id, nn);
        warp_argmax_redux(bt, it);
        warp_argmax_redux(bd, id);
        nanw = __any_sync(kFull, nn) ? 1.0f : 0.0f;
        part = make_float4(bt, __int_as_float(it), bd, __int_as_float(id));
      }
      // the control warp has read this slot's previous partials (task i - kSlots)
      if (i >= kSlots) pwait(smem_addr(&sm.p1free[slot]), par(i) ^ 1u, P, sm);
      if (lane == 0) {
        sm.wp1[slot][warp] = part;
        sm.wnan[slot][warp] = nanw;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&sm.p1done[slot]));
        if constexpr (kGreedy) mbar_arrive(smem_addr(&sm.empty[i % D]));
      }
    }
  } else if (warp < kCompWarps) {
    // ================= phase-2 warps (T > 0) =================
    const int w2 = warp - kP1Warps;
    const int j = w2 * 32 + lane;
    for (int jt = 0; jt < n; ++jt) {
      const int slot = jt % kSlots2;
      pwait(smem_addr(&sm.nrm_bar[slot]), par2(jt), P, sm);
      const Nrm nr = sm.nrm[slot];
      const StageDesc dsc = sm.desc[jt % D];  // the stage is held until these warps release it
      float A, R, Sm;
      uint32_t* segp = (P.seg != nullptr) ? P.seg + ((long long)dsc.u * P.C + dsc.c) * kMaxSegs : nullptr;
      phase2_sample<E, MODE>(stage_t(jt), stage_d(jt), j, w2, lane, dsc.nv, nr.mode, s, nr.c1t, nr.cd2, segp, A, R,
                             Sm);
      A = warp_sum(A);
      if constexpr (MODE == kE2E) Sm = warp_sum(Sm);
      if (lane == 0) sm.wp2[slot][w2] = make_float4(A, R, Sm, 0.0f);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&sm.p2done[slot]));
        mbar_arrive(smem_addr(&sm.empty[jt % D]));
      }
    }
  } else if (warp == kProducerWarp) {
    // ================= producer warp =================
    const bool bulk = P.aligned != 0;
    for (int i = 0; i < n; ++i) {
      const int st = i % D;
      if (i >= D) pwait(smem_addr(&sm.empty[st]), (uint32_t)((i / D) + 1) & 1u, P, sm);
      const TaskInfo tk = task_of(i);
      const UnitInfo<E> ui = unit_info<E, MODE>(P, tk.u);
      uint8_t* dst = stage_mem + (size_t)st * P.stage;
      const uint32_t bar = smem_addr(&sm.full[st]);
      if (lane == 0) {
        StageDesc dd;
        dd.u = tk.u;
        dd.c = tk.c;
        dd.e0 = tk.e0;
        dd.nv = tk.nv;
        dd.has_d = ui.has_d ? 1 : 0;
        dd.pad[0] = dd.pad[1] = dd.pad[2] = 0;
        sm.desc[st] = dd;  // published by the arrival below (release), read after the full wait
      }
      if (bulk) {
        // 4 copies per stage (2 per row when both rows are loaded): a few
        // copies of several KB each keep the memory pipe full, while copies
        // of 1 KB or less cost more in per-copy overhead than they gain
        const uint32_t bytes = (uint32_t)tk.len * (uint32_t)E::ES;
        const int rows = ui.has_d ? 2 : 1;
        const int per_row = 4 / rows;
        const uint32_t piece = ((bytes + per_row - 1) / per_row + 15u) & ~15u;
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar, (uint32_t)rows * bytes);
        }
        __syncwarp();
        const int row = lane / per_row;
        const uint32_t off = (uint32_t)(lane % per_row) * piece;
        if (row < rows && off < bytes) {
          const uint32_t len = min(piece, bytes - off);
          const char* src = reinterpret_cast<const char*>((row == 0 ? ui.tg : ui.dg) + tk.e0) + off;
          bulk_load_plain(smem_addr(dst + (row ? P.doff : 0) + off), src, len, bar);
        }
      } else {
        // element-wise staging for rows off 16-byte boundaries (-inf padding)
        Raw* rt = reinterpret_cast<Raw*>(dst);
        Raw* rd = reinterpret_cast<Raw*>(dst + P.doff);
        const int padded = tk.nv * PV;
        for (int e = lane; e < padded; e += 32) {
          const bool in = e < tk.len;
          rt[e] = in ? ui.tg[tk.e0 + e] : E::kNegInf;
          if (ui.has_d) rd[e] = in ? ui.dg[tk.e0 + e] : E::kNegInf;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
      }
    }
    // no CTA may leave with bulk copies still landing in its shared memory
    if (bulk && lane == 0) {
      for (int i = (n > D ? n - D : 0); i < n; ++i) pwait(smem_addr(&sm.full[i % D]), (uint32_t)(i / D) & 1u, P, sm);
    }
  } else if (warp < kFinalWarp) {
    // ================= control warps =================
    const int r = warp - kControlWarp0;
    // one ticket per job; the finaliser takes them in ticket order
    auto push_job = [&](const Job& jb) {
      int kc = 0;
      if (lane == 0) kc = atomicAdd(&sm.job_tail, 1);
      kc = __shfl_sync(kFull, kc, 0);
      const int q = kc % kJobSlots;
      if (kc >= kJobSlots) pwait(smem_addr(&sm.job_empty[q]), (uint32_t)((kc / kJobSlots) + 1) & 1u, P, sm);
      if (lane == 0) sm.job[q] = jb;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.job_full[q]));
    };
    // tagged words of every chunk of unit u, lanes over chunks in groups of 32,
    // once all are written
    auto read_unit = [&](int u, int nwords, uint64_t (&a)[3], const uint64_t* base_ptr, int stride, int base) {
      const int c = base + lane;
      const uint64_t* w = base_ptr + ((long long)u * P.C + c) * stride;
      auto load = [&]() {
#pragma unroll
        for (int k = 0; k < 3; ++k) a[k] = (c < P.C && k < nwords) ? ld_relaxed_u64(w + k) : ~0ull;
      };
      auto ok = [&]() { return tag_ok(a[0]) && tag_ok(a[1]) && tag_ok(a[2]); };
      load();
      poll_words(P, lane, ok, load);
    };
    // phase-1 partials of task i from the compute warps' slot
    auto read_wp1 = [&](int i, float& x, float& y, float& z, float& w, float& nn) {
      const int slot = i % kSlots;
      pwait(smem_addr(&sm.p1done[slot]), par(i), P, sm);
      x = y = z = w = nn = 0.0f;
      if (lane < kP1Count) {
        const float4 q = sm.wp1[slot][lane];
        x = q.x;
        y = q.y;
        z = q.z;
        w = q.w;
        nn = sm.wnan[slot][lane];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.p1free[slot]));  // the slot may be reused
    };

    if constexpr (kGreedy) {
      for (int i = r; i < n; i += kCtlWarps) {
        float v1, v2, fi1, fi2, nn;
        read_wp1(i, v1, fi1, v2, fi2, nn);
        int i1 = (lane < kP1Count) ? __float_as_int(fi1) : 0x7FFFFFFF;
        int i2 = (lane < kP1Count) ? __float_as_int(fi2) : 0x7FFFFFFF;
        if (lane >= kP1Count) v1 = v2 = -INFINITY;
        warp_argmax_redux(v1, i1);
        warp_argmax_redux(v2, i2);
        nn = redux_max_f32(nn);
        const TaskInfo tk = task_of(i);
        if (lane == 0) {
          uint64_t* w = P.part1 + ((long long)tk.u * P.C + tk.c) * 4;
          st_relaxed_u64(w + 0, tag2i(v1, i1));
          st_relaxed_u64(w + 1, tag2i(v2, i2));
          st_relaxed_u64(w + 2, tag2(nn, 0.0f));
        }
        // the CTA holding the unit's finalising chunk hands the unit to its
        // finaliser, which waits for the other chunks' partials
        if (tk.c == fin_chunk(P, tk.u)) {
          Job jb{};
          jb.unit = tk.u;
          push_job(jb);
        }
      }
    } else {
      for (int i = r; i < n + kLag; i += kCtlWarps) {
        // ---- task i: publish its phase-1 partials, read back the unit's, decide
        if (i < n) {
          float mt, zt, md, zd, nn;
          read_wp1(i, mt, zt, md, zd, nn);
          if (lane >= kP1Count) {
            mt = md = -INFINITY;
            zt = zd = 0.0f;
          }
          warp_combine_mz2(mt, zt, md, zd, s);
          const TaskInfo tk = task_of(i);
          const UnitInfo<E> ui = unit_info<E, MODE>(P, tk.u);
          int y = -1;
          float ua = 0.0f, uf = 0.0f;
          if constexpr (MODE == kVerify) {
            if (lane == 0) {
              y = ui.bonus ? -1 : __ldg(P.draft_tokens + ui.b * P.K + ui.k);
              ua = ui.bonus ? 0.0f : __ldg(P.u_accept + ui.b * P.K + ui.k);
              uf = __ldg(P.u_final + ui.b);
            }
          }
          if (lane == 0) {
            float gt = 0.0f, gd = 0.0f;
            if (MODE == kVerify && !ui.bonus && y >= tk.e0 && y < tk.e0 + tk.len) {
              // the stage of task i is held until its phase 2, which needs this decision
              gt = E::to_f32(reinterpret_cast<const Raw*>(stage_t(i))[y - tk.e0]);
              gd = E::to_f32(reinterpret_cast<const Raw*>(stage_d(i))[y - tk.e0]);
            }
            uint64_t* w = P.part1 + ((long long)tk.u * P.C + tk.c) * 4;
            st_relaxed_u64(w + 0, tag2(mt, zt));
            if (ui.has_d) {
              st_relaxed_u64(w + 1, tag2(md, zd));
              st_relaxed_u64(w + 2, tag2(gt, gd));
            }
          }
          const bool need_g = (MODE == kVerify) && !ui.bonus;
          const int yb = __shfl_sync(kFull, y, 0);
          const int cy = (need_g && yb >= 0 && yb < P.V) ? yb / P.Lc : -1;
          const int nwords = need_g ? 3 : (ui.has_d ? 2 : 1);
          float cm_t = -INFINITY, cz_t = 0.0f, cm_d = -INFINITY, cz_d = 0.0f, gt = 0.0f, gd = 0.0f;
          auto merge = [&](float& m, float& z, float m2, float z2) {
            if (!(m2 > -INFINITY)) {
              if (m2 != m2) m = m2;  // NaN propagates
              return;
            }
            if (!(m > -INFINITY)) {
              if (m == m) {
                m = m2;
                z = z2;
              }
              return;
            }
            const float M = fmaxf(m, m2);
            const float cM = __fmul_rn(M, s);
            z = __fadd_rn(__fmul_rn(z, ex2(__fadd_rn(__fmul_rn(m, s), -cM))),
                          __fmul_rn(z2, ex2(__fadd_rn(__fmul_rn(m2, s), -cM))));
            m = M;
          };
          for (int base = 0; base < P.C; base += 32) {
            uint64_t a[3];
            read_unit(tk.u, nwords, a, P.part1, 4, base);
            if (base + lane < P.C) {
              if (base == 0) {
                cm_t = tag_lo(a[0]);
                cz_t = tag_hi(a[0]);
                if (ui.has_d) {
                  cm_d = tag_lo(a[1]);
                  cz_d = tag_hi(a[1]);
                }
              } else {
                merge(cm_t, cz_t, tag_lo(a[0]), tag_hi(a[0]));
                if (ui.has_d) merge(cm_d, cz_d, tag_lo(a[1]), tag_hi(a[1]));
              }
              if (base + lane == cy) {
                gt = tag_lo(a[2]);
                gd = tag_hi(a[2]);
              }
            }
          }
          warp_combine_mz2(cm_t, cz_t, cm_d, cz_d, s);
          if (cy >= 0) {
            gt = __shfl_sync(kFull, gt, cy & 31);
            gd = __shfl_sync(kFull, gd, cy & 31);
          }
          const int slot2 = i % kSlots2;
          if (lane == 0) {
            const float Zt = cz_t, Zd = cz_d;
            const float c1t = __fmul_rn(cm_t, s), c1d = __fmul_rn(cm_d, s);
            const bool valid = (Zt > 0.0f && Zt < INFINITY) && (!ui.has_d || (Zd > 0.0f && Zd < INFINITY));
            const float izt = __frcp_rn(Zt), izd = __frcp_rn(Zd);
            uint32_t flags = 0;
            int mode = 0, acc = 1;
            if constexpr (MODE == kVerify) {
              if (ui.bonus) {
                mode = 2;
                acc = 0;
              } else {
                const bool tok_ok = y >= 0 && y < P.V;
                // u * q(y) <= p(y), with p(y), q(y) formed like the per-element values
                const float pyv = __fmul_rn(ex2(fmaf(gt, s, -c1t)), izt);
                const float qyv = __fmul_rn(ex2(fmaf(gd, s, -c1d)), izd);
                acc = (tok_ok && __fmul_rn(ua, qyv) <= pyv) ? 1 : 0;
                mode = acc ? 0 : 1;
                if (!(ua >= 0.0f && ua < 1.0f)) flags |= kBadUniform;
                if (!tok_ok) flags |= kBadToken;
              }
              if (!(uf >= 0.0f && uf < 1.0f)) flags |= kBadUniform;
            }
            if (!valid) {
              flags |= kBadLogits;
              mode = 3;
              acc = 0;
            }
            if (flags && tk.c == 0 && P.status) atomicOr(P.status, flags);
            Nrm& nr = sm.nrm[slot2];  // its previous content (task i - 8) was consumed at task i - 4
            nr.c1t = c1t;
            nr.c1d = c1d;
            nr.cd2 = (ui.has_d && valid) ? c1d + __log2f(__fmul_rn(Zd, izt)) : 0.0f;
            nr.izt = izt;
            nr.uf = uf;
            nr.mode = mode;
            nr.acc = acc;
            nr.unit = tk.u;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.nrm_bar[slot2]));
        }
        // ---- task i - kLag: publish its phase-2 partials; the CTA holding the
        // unit's finalising chunk waits for the others' and hands the unit on
        if (i >= kLag && i - kLag < n) {
          const int i4 = i - kLag;
          const int slot2 = i4 % kSlots2;
          pwait(smem_addr(&sm.p2done[slot2]), par2(i4), P, sm);
          float A = 0.0f, R = 0.0f, Sm = 0.0f;
          if (lane < kP2Warps) {
            const float4 q = sm.wp2[slot2][lane];
            A = q.x;
            R = q.y;
            Sm = q.z;
          }
          A = warp_sum(A);
          R = warp_sum(R);
          Sm = warp_sum(Sm);
          const TaskInfo t4 = task_of(i4);
          const Nrm nr = sm.nrm[slot2];
          if (lane == 0) {
            const float nanv = __int_as_float(0x7FC00000);
            const float ac = (nr.mode == 3) ? nanv : __fmul_rn(A, nr.izt);
            const float second = (MODE == kE2E) ? ((nr.mode == 3) ? nanv : __fmul_rn(Sm, nr.izt)) : R;
            st_relaxed_u64(P.part2 + (long long)t4.u * P.C + t4.c, tag2(ac, second));
          }
          if (t4.c == fin_chunk(P, t4.u)) {
            Job jb{};
            jb.unit = t4.u;
            jb.mode = nr.mode;
            jb.acc = nr.acc;
            jb.c1t = nr.c1t;
            jb.cd2 = nr.cd2;
            jb.izt = nr.izt;
            jb.uf = nr.uf;
            push_job(jb);
          }
        }
      }
    }
    // one stop job per control warp
    Job stop{};
    stop.stop = 1;
    push_job(stop);
  } else {
    // ================= finaliser warp =================
    int stops = 0;
    for (int k = 0;; ++k) {
      const int q = k % kJobSlots;
      if (!pwait(smem_addr(&sm.job_full[q]), (uint32_t)(k / kJobSlots) & 1u, P, sm)) break;
      const Job jb = sm.job[q];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.job_empty[q]));
      if (jb.stop) {
        if (++stops == kCtlWarps) break;
        continue;
      }
      finalize_unit<E, MODE>(P, jb, lane);
    }
  }

  // ---- exit: the last CTA resets the control words (and, after an abort,
  // the whole workspace, whose contents are then undefined)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(P.ctl + kCtlExit, 1u);
    if (old == (uint32_t)G - 1) {
      __threadfence();
      sm.wipe = (ld_relaxed_u32(P.ctl + kCtlAbort) != 0u) ? 2 : 1;
    }
  }
  __syncthreads();
  if (sm.wipe == 2) {
    uint32_t* w = reinterpret_cast<uint32_t*>(P.ws);
    for (size_t i = threadIdx.x; i < P.ws_bytes / 4; i += blockDim.x) w[i] = 0u;
  } else if (sm.wipe == 1 && threadIdx.x == 0) {
    P.ctl[kCtlExit] = 0u;
  }
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
