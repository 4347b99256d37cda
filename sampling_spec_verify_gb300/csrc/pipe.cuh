// Two-pass vocabulary sweep for sm_103a: pass A streams the logits from HBM,
// pass C reads them again from L2.
//
// A (row b, position k) "unit" is one target row (and, for drafted positions,
// one draft row) of V logits.  A thread-block cluster of S CTAs (one CTA per
// SM) works through its units in order; CTA r owns the slice r of every
// row, and the slice is cut into chunks of at most CV 16-byte vectors.  Each
// CTA has
//   * a producer warp, whose elected lane streams chunks into a ring of NS
//     shared-memory stages with 1-D bulk (TMA) copies, each stage completing
//     on its own mbarrier;
//   * sixteen consumer warps, which share every chunk (warp w takes a
//     contiguous sub-segment, lane l every 32nd vector of it) and touch
//     nothing but shared memory on their hot path;
//   * a decision warp, which combines the cluster's per-warp pass-A
//     partials of each unit once per CTA and publishes the unit's decision
//     (normalisers, acceptance, what pass C computes) in shared memory;
//   * a completion warp, which takes each finished unit from an in-order job
//     ring in shared memory and does all of the unit's global-memory work:
//     per-CTA partials, records, arrivals on the row counters, the row's
//     completion, and the inverse-CDF draws of rejected and bonus positions.
// A unit's chunks are loaded twice: once for pass A (softmax normalisers,
// from HBM) and once more for pass C (overlap, residual weights; the second
// copy hits L2, because it comes a few chunks after the first).  The ring
// interleaves the pass-A chunks of unit u+1 with the pass-C chunks of unit
// u, so a stage is never held while the cluster exchanges unit u's
// normalisers: every consumer warp pushes its (max, sum) pairs with st.async
// into every CTA's mailbox, completing on that CTA's mbarrier, and each CTA's
// decision warp combines all the cluster's pairs in one fixed order, so every
// CTA of the cluster takes the same decision with no cluster barrier.
//
// Draws: every consumer warp's residual (or target) total of its
// sub-segment of each chunk goes to the workspace, in (CTA, chunk, warp)
// order; the CTA whose completion warp brings a drawing unit's counter to S
// does the draw: it sums those totals, locates the sub-segment holding
// u' * total, copies that sub-segment into shared memory with one round of
// loads, recomputes its weights in the consumers' order and arithmetic, and
// walks to the token.
#pragma once

#include "sweep.cuh"

namespace ssv {

constexpr int kPNC = 16;                    // consumer warps
constexpr int kPProd = kPNC;                // producer warp
constexpr int kPDone = kPNC + 1;            // completion warp
constexpr int kPDec = kPNC + 2;             // decision warp
constexpr int kPThreads = (kPNC + 3) * 32;  // 608
constexpr int kPNX = 4;                     // exchange slots (units in flight)
constexpr int kPMaxS = 16;
constexpr int kPMaxNS = 8;
constexpr int kPMaxCh = 32;     // chunks per slice
constexpr int kPMaxParts = 32;  // S x chunks per slice
constexpr int kPSegs = kPMaxParts * 16;  // draw totals per unit: one per (CTA, chunk, consumer warp)
constexpr int kPQ = 8;          // units between the consumers and the completion warp
constexpr int kPSegV = 128;     // vectors per row of a warp sub-segment, at most (32 lanes x 4)
// Unit-scalar slots: the producer may run up to a full ring (kPMaxNS items,
// one phase per item at worst) ahead of the consumers, which read a unit's
// slot until the phase after it.
constexpr int kPUS = 16;

enum PMode : int { kPSample = 0, kPGreedy = 1, kPOverlap = 2, kPE2E = 3 };

struct PipeParams {
  const void* target;
  const void* draft;
  int B, K, KT, V;
  int units;
  int S, G;     // CTAs per cluster, clusters
  int NV;       // vectors per CTA slice
  int CV;       // vectors per chunk (per row)
  int NCH;      // chunks per slice
  int WV;       // vectors per consumer warp per chunk
  int NS;       // ring stages
  int rows;     // rows per stage: 2 (target and draft) or 1 (target only)
  int grouped;  // sampling: rows in groups of G, position-major
  float s;      // log2(e) / T
  float inv_t;
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
  float* part;     // [units][kPartStride] overlap partials, one per CTA
  float* part2;    // [units][kPartStride] E2E S-mass partials
  float* dtot;     // [units][kPSegs] draw totals per (CTA, chunk, consumer warp)
  uint32_t* dcnt;  // [units] CTAs done with a drawing unit
  float* row_loss;
  uint32_t* row_cnt;
  uint32_t* rej;  // [B] kRejBase - (earliest rejected position seen), 0 if none
  uint32_t* glob_cnt;
  uint32_t* status;
};

// Dynamic shared memory of a launch: the ring, then the mailbox, then the
// per-chunk draw totals of the units between the consumers and the
// completion warp.
__host__ __device__ constexpr size_t pipe_stage_bytes(int rows, int CV) { return (size_t)rows * CV * 16; }
__host__ __device__ constexpr size_t pipe_mbox_bytes(int S) { return (size_t)kPNX * S * (kPNC + 1) * 16; }
__host__ __device__ constexpr size_t pipe_wt_bytes(int NCH) { return (size_t)kPQ * NCH * kPNC * 4; }
__host__ __device__ constexpr size_t pipe_dyn_bytes(int NS, int rows, int CV, int S, int NCH) {
  return NS * pipe_stage_bytes(rows, CV) + pipe_mbox_bytes(S) + pipe_wt_bytes(NCH);
}

struct PUnit {
  int b, k, rec;
  bool bonus, has_draft;
  long long trow, drow;  // row indices into target / draft
};

template <int MODE>
__device__ __forceinline__ PUnit pdecode(const PipeParams& P, int u) {
  PUnit x;
  const int K = P.K;
  if constexpr (MODE == kPSample) {
    if (P.grouped) {
      // rows in groups of G, position-major inside a group: with full
      // groups, cluster c takes row c of the group at positions 0..K in turn
      const int G = P.G;
      const int gsz = G * (K + 1);
      const int g = u / gsz;
      const int j = u - g * gsz;
      const int r0 = g * G;
      const int rg = min(G, P.B - r0);
      x.k = j / rg;
      x.b = r0 + (j - x.k * rg);
    } else {
      // drafted positions row-major, then every row's bonus
      const int nd = P.B * K;
      if (u < nd) {
        x.b = u / K;
        x.k = u - x.b * K;
      } else {
        x.b = u - nd;
        x.k = K;
      }
    }
    x.bonus = (x.k == K);
    x.has_draft = !x.bonus;
    x.rec = x.b * (K + 1) + x.k;
  } else if constexpr (MODE == kPGreedy) {
    x.b = u / (K + 1);
    x.k = u - x.b * (K + 1);
    x.bonus = (x.k == K);
    x.has_draft = !x.bonus && P.rows == 2;
    x.rec = u;
  } else {
    x.b = u / K;
    x.k = u - x.b * K;
    x.bonus = false;
    x.has_draft = true;
    x.rec = u;
  }
  x.trow = (long long)x.b * P.KT + x.k;
  x.drow = (long long)x.b * K + x.k;
  return x;
}

// A unit's decision, handed from the consumers to the completion warp.
struct UnitJob {
  int mode_c;  // 0 overlap only, 1 residual draw, 2 target draw, 3 invalid logits
  int acc;     // accepted (verify), or the greedy decision
  int draw;    // this unit draws (it may still be unused)
  int need_a;  // pass C sums the overlap
  int am_t, am_d;  // greedy: target / draft arg-maxima
  float c1t, c1d, cd2, izt, ratio, ufin;
};

// Per-unit inputs of the decision, loaded by the producer warp so that the
// consumer warps issue no global-memory operation.
struct UnitScalars {
  int y;          // drafted token
  float ua, uf;   // acceptance and final uniforms
  uint32_t rejw;  // rank 0: the row's earliest-rejection word when the unit started
  float zty, zdy; // target and draft logits of the drafted token
};

struct PipeSmem {
  uint64_t full[kPMaxNS];
  uint64_t empty[kPMaxNS];
  uint64_t xbar[kPNX];
  float wa[kPQ][kPNC];  // warp overlap partials
  float wg[kPQ][kPNC];  // warp E2E S-mass partials
  uint32_t cnt[kPQ];    // warps done with a unit
  UnitJob job[kPQ];
  uint32_t ticket[kPQ];    // p + 1 once unit p's job is in slot p % kPQ
  uint32_t done_head;      // units the completion warp has finished
  uint32_t us_done;        // units whose scalars (gathered logits included) are in `us`
  UnitScalars us[kPUS];    // written by the producer at the start of a unit's phase
  uint64_t dbar[kPNX];     // a unit's decision is in `dec`
  UnitJob dec[kPNX];       // written by the decision warp, read by the consumer warps
  uint4 dseg[2 * kPSegV];  // the completion warp's copy of the sub-segment a draw walks
};

__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}
__device__ __forceinline__ void st_volatile_u32(uint32_t* p, uint32_t v) {
  *reinterpret_cast<volatile uint32_t*>(p) = v;
}

// Waits (lane 0 polling, the warp following) until *ctr >= want; gives up
// after the wait limit and reports it.
__device__ __forceinline__ void wait_counter(const uint32_t* ctr, uint32_t want, int lane, uint32_t* status) {
  int ok = 1;
  if (lane == 0) {
    if (ld_volatile_u32(ctr) < want) {
      const uint64_t t0 = global_timer_ns();
      while (ld_volatile_u32(ctr) < want) {
        __nanosleep(32);
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          ok = 0;
          break;
        }
      }
    }
    __threadfence_block();
  }
  ok = __shfl_sync(kFull, ok, 0);
  if (!ok && lane == 0 && status) atomicOr(status, kTimeout);
}

// (m, z) stands for z * 2^fl(m s).  Merges (mi, zi) into (m, z) with the same
// rescaling as the warp combine.
__device__ __forceinline__ void mz_merge(float& m, float& z, float mi, float zi, float s) {
  if (!(mi > -INFINITY)) return;
  if (!(m > -INFINITY)) {
    m = mi;
    z = zi;
  } else if (mi > m) {
    z = __fadd_rn(__fmul_rn(z, ex2(__fadd_rn(__fmul_rn(m, s), -__fmul_rn(mi, s)))), zi);
    m = mi;
  } else {
    z = __fadd_rn(z, __fmul_rn(zi, ex2(__fadd_rn(__fmul_rn(mi, s), -__fmul_rn(m, s)))));
  }
}

// The values of a 16-byte vector as float2 pairs in element order (exact
// widening of bf16; fp32 as is).
template <class E>
__device__ __forceinline__ void pairs2(const uint4& w, float2 (&p)[E::PV / 2]) {
  if constexpr (E::ES == 2) {
    p[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
    p[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
    p[2] = make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
    p[3] = make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
  } else {
    p[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
    p[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
}

// A lane's VPL vectors idx0, idx0+32, ... of a chunk of cv vectors, loaded
// at once; vectors past the chunk read as -inf (they add nothing).
template <class E, int VPL>
__device__ __forceinline__ bool load_lane(const uint4* base, int idx0, int cv, uint4 (&w)[VPL]) {
  if (idx0 + 32 * (VPL - 1) < cv) {  // every vector present: all but a slice's last chunk
#pragma unroll
    for (int v = 0; v < VPL; ++v) w[v] = base[idx0 + 32 * v];
    return true;
  }
  const uint32_t ninf = (E::ES == 2) ? 0xFF80FF80u : 0xFF800000u;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int i = idx0 + 32 * v;
    w[v] = (i < cv) ? base[i] : make_uint4(ninf, ninf, ninf, ninf);
  }
  return idx0 < cv;
}

// Adds a lane's vectors of one chunk to its running pair (m, z) of the unit:
// the offset fl(m s) is fixed by the lane's first vector of the unit and
// later chunks add 2^(x s - fl(m s)) to z.  A chunk whose sum is not below
// 2^100 (a value far above the offset, an infinity or a NaN) is summed again
// with a running maximum and merged with rescaling.
template <class E, int VPL>
__device__ __forceinline__ void lane_item_add(const uint4 (&w)[VPL], float s, float& m, float& z) {
  constexpr int PV = E::PV;
  float m0 = m, z0 = z;
  if (!(m0 > -INFINITY)) {
    m0 = E::vmax(w[0]);
    z0 = 0.0f;
  }
  if (m0 > -INFINITY) {
    const float c = __fmul_rn(m0, s);
    const float2 S2 = make_float2(s, s), C2 = make_float2(-c, -c);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float2 p[PV / 2];
      pairs2<E>(w[v], p);
#pragma unroll
      for (int h = 0; h < PV / 2; ++h) {
        const float2 x = __ffma2_rn(p[h], S2, C2);
        acc = __fadd2_rn(acc, make_float2(ex2(x.x), ex2(x.y)));
      }
    }
    const float zc = __fadd_rn(acc.x, acc.y);
    if (zc < 0x1p100f) {  // false for NaN and infinities
      m = m0;
      z = __fadd_rn(z0, zc);
      return;
    }
  }
  const f32x2 S2 = f2(s, s);
  float mc = -INFINITY, zc = 0.0f, cm = 0.0f;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const float vm = E::vmax(w[v]);
    if (vm > mc) {
      const float cn = __fmul_rn(vm, s);
      zc = (mc > -INFINITY) ? __fmul_rn(zc, ex2(__fadd_rn(cm, -cn))) : 0.0f;
      cm = cn;
      mc = vm;
    }
    if (mc > -INFINITY) {
      f32x2 ep[PV / 2];
      exp_pairs<E>(w[v], S2, f2(-cm, -cm), ep);
      zc = __fadd_rn(zc, f2_hsum(psum(ep)));
    }
  }
  mz_merge(m, z, mc, zc, s);
}

// Overlap terms of a lane's vector pairs of one chunk: the sum of
// 2^min(x_t, x_d') (and, for E2E-TV, of the terms with x_d' < x_t).
template <class E, int VPL, bool kE2EM>
__device__ __forceinline__ void lane_item_overlap(const uint4 (&wt)[VPL], const uint4 (&wd)[VPL], float s, float ct,
                                                  float cd, float2& a2, float2& g2) {
  constexpr int PV = E::PV;
  const float2 S2 = make_float2(s, s), CT = make_float2(-ct, -ct), CD = make_float2(-cd, -cd);
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    float2 pt[PV / 2], pd[PV / 2];
    pairs2<E>(wt[v], pt);
    pairs2<E>(wd[v], pd);
#pragma unroll
    for (int h = 0; h < PV / 2; ++h) {
      const float2 x = __ffma2_rn(pt[h], S2, CT), y = __ffma2_rn(pd[h], S2, CD);
      const float e0 = ex2(fminf(x.x, y.x)), e1 = ex2(fminf(x.y, y.y));
      a2 = __fadd2_rn(a2, make_float2(e0, e1));
      if constexpr (kE2EM) g2 = __fadd2_rn(g2, make_float2(y.x < x.x ? e0 : 0.0f, y.y < x.y ? e1 : 0.0f));
    }
  }
}

// Total of the draw weights of one warp sub-segment [v0, v1) of a chunk
// (vector indices into `tv` / `dv`), one vector per lane per step, steps
// summed in order: the arithmetic of pass C' and of the draw.  With pick
// non-null it also walks to the first element whose running sum exceeds thr
// (returned as a vector * PV + element offset from v0's first element, or
// the last positive weight if none does).
template <class E, bool kResid>
__device__ __forceinline__ float seg_weights(const uint4* tv, const uint4* dv, int v0, int v1, f32x2 S2, f32x2 CT,
                                             f32x2 CD, f32x2 NR, int lane, float thr, int* pick,
                                             f32x2* min_mass = nullptr) {
  constexpr int PV = E::PV;
  float R = 0.0f;
  int found = -1, ilast = -1;
  f32x2 mm = f2(0.0f, 0.0f);
  for (int base = v0; base < v1; base += 32) {
    const int i = base + lane;
    float w[PV];
    float ws = 0.0f;
    if (i < v1) {
      ws = draw_weights<E, kResid>(tv[i], kResid ? dv[i] : tv[i], S2, CT, CD, NR, w, mm);
    } else {
#pragma unroll
      for (int e = 0; e < PV; ++e) w[e] = 0.0f;
    }
    const float incl = warp_incl_scan(ws, lane);
    const float run = __fadd_rn(R, incl);
    if (pick != nullptr && found < 0) {
      const float up = __shfl_up_sync(kFull, run, 1);
      const float before = (lane == 0) ? R : up;
      const unsigned pos = __ballot_sync(kFull, ws > 0.0f);
      if (pos) ilast = base + 31 - __clz(pos);
      const unsigned hit = __ballot_sync(kFull, ws > 0.0f && run > thr);
      if (hit) {
        const int k = __ffs(hit) - 1;
        int pk = -1;
        if (lane == k) {
          float a = before;
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < PV; ++e) {
            a = __fadd_rn(a, w[e]);
            if (w[e] > 0.0f) {
              lastp = e;
              if (pk < 0 && a > thr) pk = e;
            }
          }
          if (pk < 0) pk = lastp;  // the vector crosses but no element does (rounding)
          pk = (i - v0) * PV + pk;
        }
        found = __shfl_sync(kFull, pk, k);
      }
    }
    R = __shfl_sync(kFull, run, 31);
  }
  if (min_mass) *min_mass = f2_add(*min_mass, mm);
  if (pick != nullptr) {
    if (found < 0 && ilast >= 0) {  // no crossing (rounding): the last positive weight
      int pk = -1;
      if (lane == 0) {
        float w[PV];
        f32x2 dummy = f2(0.0f, 0.0f);
        draw_weights<E, kResid>(tv[ilast], kResid ? dv[ilast] : tv[ilast], S2, CT, CD, NR, w, dummy);
#pragma unroll
        for (int e = 0; e < PV; ++e)
          if (w[e] > 0.0f) pk = (ilast - v0) * PV + e;
      }
      found = __shfl_sync(kFull, pk, 0);
    }
    *pick = found;
  }
  return R;
}

// ---- per-row completion (one warp) ---------------------------------------------

template <int MODE>
__device__ __forceinline__ void pcomplete_row(const PipeParams& P, int b, int lane) {
  constexpr bool kVer = (MODE == kPSample || MODE == kPGreedy);
  const int K = P.K;
  const int per_row = kVer ? K + 1 : K;
  const int base = b * per_row;
  const int nparts = (MODE == kPGreedy) ? 1 : P.S;
  const float* pp0 = P.part + (long long)base * kPartStride;
  auto alpha_of = [&](int kk) {
    const float* pp = pp0 + kk * kPartStride;
    float a = 0.0f;
    for (int r = 0; r < nparts; ++r) a = __fadd_rn(a, __ldcg(pp + r));
    return a;
  };
  float* pw = P.part + (long long)base * kPartStride;
  if constexpr (kVer) {
    const VerifyRecord* rr = P.rec + base;
    int nacc = K;
    for (int k0 = 0; k0 < K; k0 += 32) {
      const int kk = k0 + lane;
      const int a = (kk < K) ? __ldcg(&rr[kk].acc) : 1;
      const unsigned m = __ballot_sync(kFull, a == 0);
      if (m) {
        nacc = k0 + __ffs(m) - 1;
        break;
      }
    }
    const int corr = __ldcg(&rr[nacc].token);
    const uint32_t emptied = __ldcg(&rr[nacc].pad0);
    if (lane == 0 && emptied && P.status) atomicOr(P.status, kEmptyResidual);
    for (int kk = lane; kk <= K; kk += 32) {
      int tokv = -1;
      if (kk < nacc) tokv = P.draft_tokens[(long long)b * K + kk];
      else if (kk == nacc) tokv = corr;
      P.out_tokens[base + kk] = tokv;
      if (kk < K && P.alpha) P.alpha[(long long)b * K + kk] = alpha_of(kk);
    }
    __syncwarp();
    VerifyRecord* rw = P.rec + base;
    for (int kk = lane; kk <= K; kk += 32) rw[kk] = VerifyRecord{0, 0, 0u, 0u};
    for (int i = lane; i < per_row * kPartStride; i += 32) pw[i] = 0.0f;
    if (lane == 0) {
      P.n_accepted[b] = nacc;
      P.row_cnt[b] = 0;
      if (P.rej) P.rej[b] = 0;
    }
  } else if constexpr (MODE == kPOverlap) {
    float al[2];
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      al[h] = (kk < K) ? alpha_of(kk) : 0.0f;
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
    __syncwarp();
    for (int i = lane; i < per_row * kPartStride; i += 32) pw[i] = 0.0f;
    if (lane == 0) {
      if (P.exp_acc) P.exp_acc[b] = sum;
      P.row_cnt[b] = 0;
    }
  } else {  // kPE2E
    E2EStats* sr = P.stats + (long long)b * K;
    const float* qq0 = P.part2 + (long long)base * kPartStride;
    float al[2], sm2[2];
    for (int h = 0; h < 2; ++h) {
      const int kk = lane + 32 * h;
      al[h] = 0.0f;
      sm2[h] = 0.0f;
      if (kk < K) {
        al[h] = alpha_of(kk);
        const float* qq = qq0 + kk * kPartStride;
        for (int r = 0; r < nparts; ++r) sm2[h] = __fadd_rn(sm2[h], __ldcg(qq + r));
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
    float* pw2 = P.part2 + (long long)base * kPartStride;
    for (int i = lane; i < per_row * kPartStride; i += 32) {
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

// One arrival of a CTA for row b (whole warp, converged); the arrival that
// completes the row finishes it.
template <int MODE>
__device__ __forceinline__ void parrive_row(const PipeParams& P, int b, int lane) {
  constexpr bool kVer = (MODE == kPSample || MODE == kPGreedy);
  const int per_row = kVer ? P.K + 1 : P.K;
  const uint32_t need = (uint32_t)(per_row * ((MODE == kPGreedy) ? 1 : P.S));
  int last = 0;
  if (lane == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&P.row_cnt[b], 1u);
    last = (old + 1u == need) ? 1 : 0;
    if (last) __threadfence();
  }
  last = __shfl_sync(kFull, last, 0);
  if (last) pcomplete_row<MODE>(P, b, lane);
}

// ---- the draw of one unit (completion warp) ------------------------------------------

template <class E, int MODE>
__device__ void pdraw(const PipeParams& P, const PUnit& x, const UnitJob& J, uint4* stage, int lane) {
  constexpr int PV = E::PV;
  const int S = P.S, NCH = P.NCH, CV = P.CV, WV = P.WV;
  const int nvec_row = P.V / PV;
  const int nseg = S * NCH * kPNC;  // warp sub-segments in prefix order (CTA, chunk, warp)
  const uint4* tv = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::Raw*>(P.target) + x.trow * P.V);
  const uint4* dv = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::Raw*>(P.draft) + x.drow * P.V);
  const f32x2 S2 = f2(P.s, P.s);
  const f32x2 CT = f2(-J.c1t, -J.c1t);
  const f32x2 CD = f2(-J.c1d, -J.c1d);
  const f32x2 NR = f2(-J.ratio, -J.ratio);
  float* dt = P.dtot + (long long)x.rec * kPSegs;
  // vectors [v0, v1) of sub-segment j of the row
  auto seg_range = [&](int j, int& v0, int& v1) {
    const int w = j % kPNC, rc = j / kPNC;
    const int r = rc / NCH, c = rc - r * NCH;
    const int s0 = min(r * P.NV, nvec_row);
    const int s1 = min(s0 + P.NV, nvec_row);
    const int c0 = min(s0 + c * CV, s1);
    const int cv = min(c0 + CV, s1) - c0;
    v0 = c0 + min(w * WV, cv);
    v1 = c0 + min(w * WV + WV, cv);
  };
  bool resid = (J.mode_c == 1);
  bool emptied = false;
  // lane l takes the contiguous block [l * E, (l + 1) * E) of the totals
  const int E_ = (nseg + 31) / 32;
  auto block_sum = [&]() {
    float t = 0.0f;
    for (int i = 0; i < E_; ++i) {
      const int j = lane * E_ + i;
      if (j < nseg) t = __fadd_rn(t, __ldcg(dt + j));
    }
    return t;
  };
  float bt = block_sum();
  float incl = warp_incl_scan(bt, lane);
  float total = __shfl_sync(kFull, incl, 31);
  if (!(total > 0.0f) && resid) {
    // no residual mass (rounding only): draw from p, recomputing every
    // sub-segment's target-weight total with the consumers' arithmetic
    resid = false;
    emptied = true;
    for (int j = 0; j < nseg; ++j) {
      int v0, v1;
      seg_range(j, v0, v1);
      const float t = seg_weights<E, false>(tv, dv, v0, v1, S2, CT, CD, NR, lane, -1.0f, nullptr);
      if (lane == 0) dt[j] = t;
    }
    __syncwarp();
    __threadfence();
    bt = block_sum();
    incl = warp_incl_scan(bt, lane);
    total = __shfl_sync(kFull, incl, 31);
  }
  int token = -1;
  if (total > 0.0f) {
    const float thr = __fmul_rn(J.ufin, total);
    // first positive sub-segment whose running total passes thr
    const float up = __shfl_up_sync(kFull, incl, 1);
    float cum = (lane == 0) ? 0.0f : up;
    int hit = -1, lastp = -1;
    float before = 0.0f;
    for (int i = 0; i < E_; ++i) {
      const int j = lane * E_ + i;
      const float t = (j < nseg) ? __ldcg(dt + j) : 0.0f;
      const float nc = __fadd_rn(cum, t);
      if (t > 0.0f) {
        lastp = j;
        if (hit < 0 && nc > thr) {
          hit = j;
          before = cum;
        }
      }
      cum = nc;
    }
    const unsigned hm = __ballot_sync(kFull, hit >= 0);
    int jsel;
    float thr_w = INFINITY;
    if (hm) {
      const int l = __ffs(hm) - 1;
      jsel = __shfl_sync(kFull, hit, l);
      thr_w = __fadd_rn(thr, -__shfl_sync(kFull, before, l));
    } else {  // no crossing (rounding): the last positive weight
      const unsigned pm = __ballot_sync(kFull, lastp >= 0);
      jsel = pm ? __shfl_sync(kFull, lastp, 31 - __clz(pm)) : -1;
    }
    if (jsel >= 0) {
      int v0, v1, pk = -1;
      seg_range(jsel, v0, v1);
      // the sub-segment's vectors into shared memory with one round of loads,
      // then the walk in the consumers' order and arithmetic
      const int nv = v1 - v0;
      uint4* st_t = stage;
      uint4* st_d = stage + kPSegV;
      uint4 rt[kPSegV / 32], rd[kPSegV / 32];
#pragma unroll
      for (int k = 0; k < kPSegV / 32; ++k) {
        const int i = lane + 32 * k;
        if (i < nv) {
          rt[k] = __ldcg(tv + v0 + i);
          if (resid) rd[k] = __ldcg(dv + v0 + i);
        }
      }
#pragma unroll
      for (int k = 0; k < kPSegV / 32; ++k) {
        const int i = lane + 32 * k;
        if (i < nv) {
          st_t[i] = rt[k];
          if (resid) st_d[i] = rd[k];
        }
      }
      __syncwarp();
      if (resid)
        seg_weights<E, true>(st_t, st_d, 0, nv, S2, CT, CD, NR, lane, thr_w, &pk);
      else
        seg_weights<E, false>(st_t, st_t, 0, nv, S2, CT, CD, NR, lane, thr_w, &pk);
      if (pk >= 0) token = v0 * PV + pk;
      __syncwarp();
    }
  }
  if (lane == 0) {
    P.rec[x.rec].token = token;
    if (emptied) P.rec[x.rec].pad0 = 1u;
    P.dcnt[x.rec] = 0u;
  }
  for (int i = lane; i < nseg; i += 32) dt[i] = 0.0f;
  __syncwarp();
  parrive_row<MODE>(P, x.b, lane);
}

// The completion warp's work for unit p: the CTA's partials, the record, the
// draw and the arrival.
template <class E, int MODE>
__device__ void pfinish_unit(const PipeParams& P, PipeSmem& sm, const float* wt, int p, int cl, uint32_t rank,
                             int lane) {
  const int slot = p % kPQ;
  const UnitJob J = sm.job[slot];
  const PUnit x = pdecode<MODE>(P, cl + p * P.G);
  const float nanv = __int_as_float(0x7FC00000);
  if constexpr (MODE == kPGreedy) {
    if (rank == 0) {
      if (lane == 0) {
        VerifyRecord r;
        r.acc = J.acc;
        r.token = J.am_t;
        r.pad0 = r.pad1 = 0u;
        P.rec[x.rec] = r;
        if (x.has_draft) P.part[(long long)x.rec * kPartStride] = (J.am_t >= 0 && J.am_t == J.am_d) ? 1.0f : 0.0f;
      }
      __syncwarp();
      parrive_row<MODE>(P, x.b, lane);
    }
    return;
  } else {
    if (lane == 0) {
      if (x.has_draft && (MODE != kPSample || P.alpha != nullptr)) {
        float A = 0.0f;
        for (int w = 0; w < kPNC; ++w) A = __fadd_rn(A, sm.wa[slot][w]);
        P.part[(long long)x.rec * kPartStride + rank] = (J.mode_c == 3) ? nanv : __fmul_rn(A, J.izt);
      }
      if constexpr (MODE == kPE2E) {
        float M2 = 0.0f;
        for (int w = 0; w < kPNC; ++w) M2 = __fadd_rn(M2, sm.wg[slot][w]);
        P.part2[(long long)x.rec * kPartStride + rank] = (J.mode_c == 3) ? nanv : __fmul_rn(M2, J.izt);
        if (rank == 0) {
          E2EStats e2;
          e2.c1t = J.c1t;
          e2.cd = J.cd2;
          e2.izt = J.izt;
          e2.smass = e2.alpha = e2.b1 = e2.b0 = e2.pad = 0.0f;
          P.stats[x.rec] = e2;
        }
      }
      if constexpr (MODE == kPSample) {
        if (rank == 0) {
          P.rec[x.rec].acc = x.bonus ? 1 : J.acc;
          if (!J.draw) P.rec[x.rec].token = -1;
        }
      }
    }
    if constexpr (MODE == kPSample) {
      if (J.draw) {
        // this CTA's per-warp totals, (chunk, warp) order
        const int NCH = P.NCH;
        float* dt = P.dtot + (long long)x.rec * kPSegs + (long long)rank * NCH * kPNC;
        for (int i = lane; i < NCH * kPNC; i += 32) dt[i] = wt[slot * NCH * kPNC + i];
        __syncwarp();
        int drawer = 0;
        if (lane == 0) {
          __threadfence();
          drawer = (atomicAdd(&P.dcnt[x.rec], 1u) == (uint32_t)(P.S - 1)) ? 1 : 0;
          if (drawer) __threadfence();
        }
        drawer = __shfl_sync(kFull, drawer, 0);
        if (drawer) {
          pdraw<E, MODE>(P, x, J, sm.dseg, lane);  // writes the token, then arrives
          return;
        }
      }
    }
    __syncwarp();
    parrive_row<MODE>(P, x.b, lane);
  }
}

// ---- the kernel ------------------------------------------------------------------

template <class E, int MODE, int VPL>
__global__ void __launch_bounds__(kPThreads, 1) pipe_kernel(const PipeParams P) {
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ __align__(16) PipeSmem sm;

  constexpr int PV = E::PV;
  using Raw = typename E::Raw;
  constexpr bool kSampleM = (MODE == kPSample);
  constexpr bool kGreedyM = (MODE == kPGreedy);
  constexpr bool kHasC = !kGreedyM;  // units are read a second time (pass C)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = P.S;
  const uint32_t rank = cluster_rank();
  const int cl = blockIdx.x / S;
  const int G = P.G;
  const int nit = (P.units > cl) ? (P.units - cl + G - 1) / G : 0;
  constexpr int WV = 32 * VPL;    // vectors per consumer warp per chunk
  constexpr int CV = kPNC * WV;   // vectors per chunk (per row)
  const int NS = P.NS, NCH = P.NCH;
  const int nvec_row = P.V / PV;
  const int sv0 = min((int)rank * P.NV, nvec_row);
  const int sv1 = min(sv0 + P.NV, nvec_row);
  const size_t stage_bytes = pipe_stage_bytes(P.rows, CV);
  auto stage_t = [&](int st) { return reinterpret_cast<uint4*>(dyn_smem + st * stage_bytes); };
  // mailbox [slot][sender CTA][sender warp | aux][4] and per-chunk draw totals [job slot][chunk][warp]
  float* mbox = reinterpret_cast<float*>(dyn_smem + NS * stage_bytes);
  float* wt = reinterpret_cast<float*>(dyn_smem + NS * stage_bytes + pipe_mbox_bytes(S));
  auto mb_at = [&](int slot, int r, int w) { return mbox + ((slot * S + r) * (kPNC + 1) + w) * 4; };
  const uint32_t xbytes = (uint32_t)(S * (kPNC + 1) * 16);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_addr(&sm.full[i]), 1);
      mbar_init(smem_addr(&sm.empty[i]), kPNC);
    }
    for (int i = 0; i < kPNX; ++i) {
      mbar_init(smem_addr(&sm.xbar[i]), 1);
      mbar_init(smem_addr(&sm.dbar[i]), 1);
    }
    for (int i = 0; i < kPQ; ++i) {
      sm.cnt[i] = 0;
      sm.ticket[i] = 0;
    }
    sm.done_head = 0;
    sm.us_done = 0;
    fence_mbar_init();
    // arm the first exchange slots
    for (int i = 0; i < kPNX && i < nit; ++i) mbar_arrive_expect_tx(smem_addr(&sm.xbar[i]), xbytes);
  }
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before any peer pushes into them

  if (warp == kPProd) {
    // ===================== producer =====================
    if (lane == 0) {
      const uint64_t polA = kHasC ? l2_evict_normal_policy() : l2_evict_first_policy();
      const uint64_t polC = l2_evict_first_policy();
      int j = 0;             // items issued
      int st = 0;            // ring stage of item j
      uint32_t epar = 0u;    // phase parity of empty[st] to wait for (from item NS on)
      auto issue = [&](const PUnit& x, int c, bool second) {
        if (j >= NS) {
          if (!mbar_wait_bounded(smem_addr(&sm.empty[st]), epar, kWaitLimitNs) && P.status)
            atomicOr(P.status, kTimeout);
        }
        const int v0 = min(sv0 + c * CV, sv1);
        const int v1 = min(v0 + CV, sv1);
        const uint32_t nb = (uint32_t)(v1 - v0) * 16u;
        const uint32_t bar = smem_addr(&sm.full[st]);
        fence_proxy_async_smem();  // the consumers' reads of this stage come first
        mbar_arrive_expect_tx(bar, x.has_draft ? 2u * nb : nb);
        if (nb) {
          uint4* dst = stage_t(st);
          const Raw* tg = reinterpret_cast<const Raw*>(P.target) + x.trow * P.V;
          bulk_load(smem_addr(dst), tg + (long long)v0 * PV, nb, bar, second ? polC : polA);
          if (x.has_draft) {
            const Raw* dg = reinterpret_cast<const Raw*>(P.draft) + x.drow * P.V;
            bulk_load(smem_addr(dst + CV), dg + (long long)v0 * PV, nb, bar, second ? polC : polA);
          }
        }
        ++j;
        if (++st == NS) {
          st = 0;
          if (j > NS) epar ^= 1u;
        }
      };
      // Unit scalars, one phase ahead: loads issued in phase q-1 are stored
      // in shared memory early in phase q (after the phase's first chunk is
      // issued, so that no copy waits on a scalar load) and published to the
      // decision warp through us_done.
      constexpr bool kScal = (kSampleM || kGreedyM);
      int ny = -1;
      float nua = 0.0f, nuf = 0.0f;
      Raw pzt = E::kNegInf, pzd = E::kNegInf;  // raw logits, converted a phase later
      uint32_t nrej = 0u;
      auto load_scalars = [&](int q) {  // issue the loads of unit q (no wait)
        const PUnit x = pdecode<MODE>(P, cl + q * G);
        const long long di = (long long)x.b * P.K + x.k;
        ny = x.bonus ? -1 : __ldg(P.draft_tokens + di);
        if constexpr (kSampleM) {
          nua = x.bonus ? 0.0f : __ldg(P.u_accept + di);
          nuf = __ldg(P.u_final + x.b);
          nrej = (rank == 0) ? __ldcg(P.rej + x.b) : 0u;
        }
      };
      if constexpr (kScal) {
        if (nit > 0) load_scalars(0);
      }
      PUnit xa = {}, xc = {};
      for (int p = 0; p <= nit; ++p) {
        xc = xa;
        if (p < nit) xa = pdecode<MODE>(P, cl + p * G);
        // the phase's first chunk, then the scalars (whose loads it may wait on)
        if (p < nit) issue(xa, 0, false);
        if (kHasC && p >= 1) issue(xc, 0, true);
        if constexpr (kScal) {
          if (p >= 1) {  // gathered logits of unit p-1 (loaded during phase p-1)
            sm.us[(p - 1) % kPUS].zty = E::to_f32(pzt);
            sm.us[(p - 1) % kPUS].zdy = E::to_f32(pzd);
            __threadfence_block();
            st_volatile_u32(&sm.us_done, (uint32_t)p);
          }
          if (p < nit) {
            UnitScalars u;
            u.y = ny;
            u.ua = nua;
            u.uf = nuf;
            u.rejw = nrej;
            u.zty = 0.0f;
            u.zdy = 0.0f;
            sm.us[p % kPUS] = u;
            // this unit's gathered logits, then the next unit's scalars
            pzt = E::kNegInf;
            pzd = E::kNegInf;
            if constexpr (kSampleM) {
              if (!xa.bonus && ny >= 0 && ny < P.V) {
                pzt = __ldg(reinterpret_cast<const Raw*>(P.target) + xa.trow * P.V + ny);
                pzd = __ldg(reinterpret_cast<const Raw*>(P.draft) + xa.drow * P.V + ny);
              }
            }
            if (p + 1 < nit) load_scalars(p + 1);
          }
        }
        for (int c = 1; c < NCH; ++c) {
          if (p < nit) issue(xa, c, false);
          if (kHasC && p >= 1) issue(xc, c, true);
        }
      }
      // no copy may still be in flight when the CTA exits
      for (int jj = max(0, j - NS); jj < j; ++jj)
        mbar_wait_bounded(smem_addr(&sm.full[jj % NS]), (uint32_t)(jj / NS) & 1u, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == kPDec) {
    // ===================== decision warp =====================
    // Takes each unit's decision once for the CTA, as soon as the cluster's
    // pass-A partials are in: the combined normalisers, the acceptance test
    // and what pass C does.  Every CTA of the cluster combines the same
    // partials in the same order, so all take the same decision.
    constexpr bool kScal = (kSampleM || kGreedyM);
    const float s = P.s;
    int lrow = -1;  // rejection seen earlier in the current row (this cluster's own decisions)
    bool lrej = false;
    for (int p = 0; p < nit; ++p) {
      const PUnit cx = pdecode<MODE>(P, cl + p * G);
      const int slot = p % kPNX;
      const uint32_t xpar = (uint32_t)(p / kPNX) & 1u;
      const bool xok = mbar_wait_bounded(smem_addr(&sm.xbar[slot]), xpar, kWaitLimitNs);
      if (lane == 0 && p + kPNX < nit) mbar_arrive_expect_tx(smem_addr(&sm.xbar[slot]), xbytes);
      if constexpr (kScal) wait_counter(&sm.us_done, (uint32_t)p + 1u, lane, P.status);
      const int ne = S * (kPNC + 1);
      // the unit's scalars
      int c_y = -1;
      float c_ua = 0.0f, c_uf = 0.0f, c_zty = 0.0f, c_zdy = 0.0f;
      if constexpr (kSampleM || kGreedyM) {
        const UnitScalars u = sm.us[p % kPUS];
        c_y = u.y;
        c_ua = u.ua;
        c_uf = u.uf;
        c_zty = u.zty;
        c_zdy = u.zdy;
      }
      const bool tok_ok = cx.bonus || (c_y >= 0 && c_y < P.V);
      uint32_t flags = 0;
      int mode_c = 0, acc = 1, am_t = -1, am_d = -1;
      bool draw = false, need_a = false;
      float c1t = 0.0f, c1d = 0.0f, cd2 = 0.0f, izt = 0.0f, ratio = 0.0f;
      if constexpr (kGreedyM) {
        float v1 = -INFINITY, v2 = -INFINITY;
        int i1 = 0x7FFFFFFF, i2 = 0x7FFFFFFF;
        bool nn = false;
        for (int e = lane; e < ne; e += 32) {
          const int r = e / (kPNC + 1), w = e - r * (kPNC + 1);
          if (w == kPNC) continue;
          const float* mm = mb_at(slot, r, w);
          const float a = mm[0], d = mm[2];
          const int ia = __float_as_int(mm[1]), id = __float_as_int(mm[3]);
          nn |= (a != a) || (d != d);
          if (a > v1 || (a == v1 && ia < i1)) {
            v1 = a;
            i1 = ia;
          }
          if (d > v2 || (d == v2 && id < i2)) {
            v2 = d;
            i2 = id;
          }
        }
        warp_argmax_redux(v1, i1);
        warp_argmax_redux(v2, i2);
        nn = __any_sync(kFull, nn);
        const bool bad = nn || !(v1 < INFINITY) || i1 == 0x7FFFFFFF ||
                         (cx.has_draft && (!(v2 < INFINITY) || i2 == 0x7FFFFFFF));
        if (bad) flags |= kBadLogits;
        am_t = bad ? -1 : i1;
        am_d = i2;
        acc = (!cx.bonus && tok_ok && c_y == am_t) ? 1 : 0;
        if (!cx.bonus && !tok_ok) flags |= kBadToken;
      } else {
        float mt = -INFINITY, zt = 0.0f, md = -INFINITY, zd = 0.0f;
        for (int e = lane; e < ne; e += 32) {
          const int r = e / (kPNC + 1), w = e - r * (kPNC + 1);
          if (w == kPNC) continue;
          const float* mm = mb_at(slot, r, w);
          mz_merge(mt, zt, mm[0], mm[1], s);
          mz_merge(md, zd, mm[2], mm[3], s);
        }
        warp_combine_mz2(mt, zt, md, zd, s);
        const float Zt = zt, Zd = zd;
        c1t = __fmul_rn(mt, s);
        c1d = __fmul_rn(md, s);
        const bool valid = (Zt > 0.0f && Zt < INFINITY) && (!cx.has_draft || (Zd > 0.0f && Zd < INFINITY));
        izt = __frcp_rn(Zt);
        const float izd = __frcp_rn(Zd);
        cd2 = (cx.has_draft && valid) ? __fadd_rn(c1d, __log2f(__fmul_rn(Zd, izt))) : 0.0f;
        ratio = __fmul_rn(Zt, izd);
        mode_c = 0;
        acc = 1;
        if constexpr (kSampleM) {
          const uint32_t seen = __float_as_uint(mb_at(slot, 0, kPNC)[0]);
          if (cx.b != lrow) {
            lrow = cx.b;
            lrej = false;
          }
          const bool earlier = lrej || (seen > kRejBase - (uint32_t)cx.k);
          if (cx.bonus) {
            mode_c = 2;
          } else {
            // u * q(y) <= p(y), with p(y), q(y) formed like the per-element values
            const float zty = c_zty, zdy = c_zdy;
            const float py = __fmul_rn(ex2(fmaf(zty, s, -c1t)), izt);
            const float qy = __fmul_rn(ex2(fmaf(zdy, s, -c1d)), izd);
            acc = (tok_ok && __fmul_rn(c_ua, qy) <= py) ? 1 : 0;
            mode_c = acc ? 0 : 1;
            if (!(c_ua >= 0.0f && c_ua < 1.0f)) flags |= kBadUniform;
            if (!tok_ok) flags |= kBadToken;
          }
          if (!(c_uf >= 0.0f && c_uf < 1.0f)) flags |= kBadUniform;
          if (!valid) {
            flags |= kBadLogits;
            mode_c = 3;
            acc = 0;
          }
          if (!cx.bonus && (mode_c == 1 || mode_c == 3)) {
            if (rank == 0 && lane == 0) atomicMax(&P.rej[cx.b], kRejBase - (uint32_t)cx.k);
            lrej = true;
          }
          draw = (mode_c == 1 || mode_c == 2) && !earlier;
          need_a = cx.has_draft && P.alpha != nullptr && mode_c != 3;
        } else {
          if (!valid) {
            flags |= kBadLogits;
            mode_c = 3;
          }
          need_a = (mode_c == 0);
        }
      }
      if (!xok) flags |= kTimeout;
      if (flags && rank == 0 && lane == 0 && P.status) atomicOr(P.status, flags);
      UnitJob J;
      J.mode_c = mode_c;
      J.acc = acc;
      J.draw = draw ? 1 : 0;
      J.need_a = need_a ? 1 : 0;
      J.am_t = am_t;
      J.am_d = am_d;
      J.c1t = c1t;
      J.c1d = c1d;
      J.cd2 = cd2;
      J.izt = izt;
      J.ratio = ratio;
      J.ufin = c_uf;
      if constexpr (kGreedyM) {
        // no pass C: the unit goes straight to the completion warp, once it
        // is done with the unit whose job slot this one takes
        const int qs = p % kPQ;
        if (p >= kPQ) wait_counter(&sm.done_head, (uint32_t)(p - kPQ + 1), lane, P.status);
        if (lane == 0) {
          sm.job[qs] = J;
          __threadfence_block();
          st_volatile_u32(&sm.ticket[qs], (uint32_t)p + 1u);
          mbar_arrive_cta(smem_addr(&sm.dbar[slot]));
        }
      } else {
        if (lane == 0) {
          sm.dec[slot] = J;
          mbar_arrive_cta(smem_addr(&sm.dbar[slot]));
        }
      }
      __syncwarp();
    }
  } else if (warp == kPDone) {
    // ===================== completion warp =====================
    for (int p = 0; p < nit; ++p) {
      const uint32_t slot = (uint32_t)(p % kPQ);
      wait_counter(&sm.ticket[slot], (uint32_t)p + 1u, lane, P.status);
      pfinish_unit<E, MODE>(P, sm, wt, p, cl, rank, lane);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        st_volatile_u32(&sm.done_head, (uint32_t)p + 1u);
      }
    }
    __syncwarp();
  } else {
    // ===================== consumer warps =====================
    const f32x2 S2 = f2(P.s, P.s);
    const float s = P.s;
    int st = 0;           // ring stage of the next item
    uint32_t fpar = 0u;   // phase parity of full[st]
    auto advance = [&]() {
      if (++st == NS) {
        st = 0;
        fpar ^= 1u;
      }
    };

    // pass-A state of the unit being read
    PUnit ax = {};
    float amt = -INFINITY, azt = 0.0f, amd = -INFINITY, azd = 0.0f;  // sampling: (m, z) pairs
    float gbt = -INFINITY, gbd = -INFINITY;                          // greedy: best values
    int git = 0x7FFFFFFF, gid = 0x7FFFFFFF;                          // greedy: their indices
    bool gnan = false;
    bool a_ok = true;
    // a unit whose pass A has ended, until the end of the phase
    bool t_okA = true;
    // the unit in pass C
    bool c_okA = true;
    // its decision, as the decision warp took it
    int mode_c = 0;  // 0: overlap only, 1: residual, 2: target draw, 3: invalid
    bool draw = false, need_a = false;
    float c1t = 0.0f, c1d = 0.0f, cd2 = 0.0f, ratio = 0.0f;
    f32x2 a2 = f2(0.0f, 0.0f);                                // draw-path overlap terms
    float2 ao = make_float2(0.0f, 0.0f), go = make_float2(0.0f, 0.0f);  // overlap path (and E2E S-mass)

    auto A_item = [&](int p, int c) {
      if (c == 0) {
        ax = pdecode<MODE>(P, cl + p * G);
        amt = -INFINITY;
        azt = 0.0f;
        amd = -INFINITY;
        azd = 0.0f;
        gbt = gbd = -INFINITY;
        git = gid = 0x7FFFFFFF;
        gnan = false;
        a_ok = true;
      }
      const bool ok = mbar_wait_bounded(smem_addr(&sm.full[st]), fpar, kWaitLimitNs);
      if (!ok) {
        a_ok = false;
        if (lane == 0 && P.status) atomicOr(P.status, kTimeout);
      }
      const int v0 = min(sv0 + c * CV, sv1);
      const int cv = min(v0 + CV, sv1) - v0;
      const int idx0 = warp * WV + lane;
      const uint4* stt = stage_t(st);
      const uint4* sdd = stt + CV;
      if (ok) {
        if constexpr (kGreedyM) {
          // packed maxima per vector; the winning vector is unpacked below
          uint4 w[VPL];
          load_lane<E, VPL>(stt, idx0, cv, w);
          float bt = -INFINITY;
          uint4 wb = w[0];
          int jt = -1;
#pragma unroll
          for (int v = 0; v < VPL; ++v) {
            bool nn;
            const float vm = E::vmax_nan(w[v], nn);
            gnan |= nn;
            if (vm > bt) {
              bt = vm;
              jt = idx0 + 32 * v;
              wb = w[v];
            }
          }
          // earlier chunks hold smaller indices: a later chunk wins only if larger
          if (jt >= 0 && bt > gbt) {
            float xv[PV];
            E::unpack(wb, xv);
            int e = PV - 1;
            for (int q = PV - 1; q >= 0; --q)
              if (xv[q] == bt) e = q;
            gbt = bt;
            git = (v0 + jt) * PV + e;
          }
          if (ax.has_draft) {
            load_lane<E, VPL>(sdd, idx0, cv, w);
            float bd = -INFINITY;
            int jd = -1;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
              bool nn;
              const float vm = E::vmax_nan(w[v], nn);
              gnan |= nn;
              if (vm > bd) {
                bd = vm;
                jd = idx0 + 32 * v;
                wb = w[v];
              }
            }
            if (jd >= 0 && bd > gbd) {
              float xv[PV];
              E::unpack(wb, xv);
              int e = PV - 1;
              for (int q = PV - 1; q >= 0; --q)
                if (xv[q] == bd) e = q;
              gbd = bd;
              gid = (v0 + jd) * PV + e;
            }
          }
        } else {
          uint4 w[VPL];
          if (load_lane<E, VPL>(stt, idx0, cv, w)) {
            lane_item_add<E, VPL>(w, s, amt, azt);
            if (ax.has_draft) {
              load_lane<E, VPL>(sdd, idx0, cv, w);
              lane_item_add<E, VPL>(w, s, amd, azd);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.empty[st]));
      advance();
      if (c == NCH - 1) {
        // this warp's share of the unit: to every CTA of the cluster
        const int slot = p % kPNX;
        float f0, f1, f2_, f3;
        if constexpr (kGreedyM) {
          warp_argmax_redux(gbt, git);
          warp_argmax_redux(gbd, gid);
          const bool nn = __any_sync(kFull, gnan);
          f0 = nn ? __int_as_float(0x7FC00000) : gbt;  // a NaN anywhere poisons the unit
          f1 = __int_as_float(git);
          f2_ = nn ? __int_as_float(0x7FC00000) : gbd;
          f3 = __int_as_float(gid);
        } else {
          warp_combine_mz2(amt, azt, amd, azd, s);
          f0 = amt;
          f1 = azt;
          f2_ = amd;
          f3 = azd;
        }
        const uint32_t rjw = sm.us[p % kPUS].rejw;  // published by the first chunk's full barrier
        const float aok = __all_sync(kFull, a_ok) ? 0.0f : 1.0f;
        if (lane < S) {
          const uint32_t a = map_rank(smem_addr(mb_at(slot, (int)rank, warp)), (uint32_t)lane);
          const uint32_t bar = map_rank(smem_addr(&sm.xbar[slot]), (uint32_t)lane);
          st_async_v4(a, f0, f1, f2_, f3, bar);
          if (warp == 0) {
            const uint32_t ax_ = map_rank(smem_addr(mb_at(slot, (int)rank, kPNC)), (uint32_t)lane);
            st_async_v4(ax_, __uint_as_float(rjw), aok, 0.0f, 0.0f, bar);
          }
        }
        // hand the unit over; pass C takes it at the end of this phase
        t_okA = __all_sync(kFull, a_ok);
      }
    };

    auto C_begin = [&](int p) {
      const int slot = p % kPNX;
      if (!mbar_wait_bounded(smem_addr(&sm.dbar[slot]), (uint32_t)(p / kPNX) & 1u, kWaitLimitNs)) {
        if (lane == 0 && P.status) atomicOr(P.status, kTimeout);
      }
      // the completion warp must be done with the unit whose job slot this one takes
      if (p >= kPQ) wait_counter(&sm.done_head, (uint32_t)(p - kPQ + 1), lane, P.status);
      const UnitJob& D = sm.dec[slot];
      mode_c = D.mode_c;
      draw = D.draw != 0;
      need_a = D.need_a != 0;
      c1t = D.c1t;
      c1d = D.c1d;
      cd2 = D.cd2;
      ratio = D.ratio;
      a2 = f2(0.0f, 0.0f);
      ao = make_float2(0.0f, 0.0f);
      go = make_float2(0.0f, 0.0f);
      if (!c_okA && lane == 0 && P.status) atomicOr(P.status, kTimeout);
    };

    auto C_item = [&](int p, int c) {
      const int qs = p % kPQ;
      const bool ok = mbar_wait_bounded(smem_addr(&sm.full[st]), fpar, kWaitLimitNs);
      if (!ok && lane == 0 && P.status) atomicOr(P.status, kTimeout);
      const int v0 = min(sv0 + c * CV, sv1);
      const int cv = min(v0 + CV, sv1) - v0;
      const int w0 = min(warp * WV, cv), w1 = min(w0 + WV, cv);
      const uint4* stt = stage_t(st);
      const uint4* sdd = stt + CV;
      const f32x2 CT = f2(-c1t, -c1t);
      float R = 0.0f;
      if (ok) {
        if (mode_c == 0 && need_a) {
          // overlap (and E2E S-mass) terms: one exp per element of min(log p, log q)
          uint4 wt_[VPL], wd_[VPL];
          if (load_lane<E, VPL>(stt, w0 + lane, w1, wt_)) {
            load_lane<E, VPL>(sdd, w0 + lane, w1, wd_);
            lane_item_overlap<E, VPL, MODE == kPE2E>(wt_, wd_, s, c1t, cd2, ao, go);
          }
        } else if constexpr (kSampleM) {
          if (mode_c == 1 && (draw || need_a)) {
            // residual weights; the overlap from the same arithmetic
            const f32x2 CDd = f2(-c1d, -c1d);
            const f32x2 NR = f2(-ratio, -ratio);
            if (draw) {
              R = seg_weights<E, true>(stt, sdd, w0, w1, S2, CT, CDd, NR, lane, -1.0f, nullptr, &a2);
            } else {
              // the same per-chunk association as the drawing branch, so
              // that alpha does not depend on whether the draw was skipped
              f32x2 mm = f2(0.0f, 0.0f);
              for (int i = w0 + lane; i < w1; i += 32) {
                float w[PV];
                draw_weights<E, true>(stt[i], sdd[i], S2, CT, CDd, NR, w, mm);
              }
              a2 = f2_add(a2, mm);
            }
          } else if (mode_c == 2 && draw) {
            const f32x2 Z2 = f2(0.0f, 0.0f);
            R = seg_weights<E, false>(stt, stt, w0, w1, S2, CT, CT, Z2, lane, -1.0f, nullptr);
          }
        }
      }
      if (draw && lane == 0) wt[(qs * NCH + c) * kPNC + warp] = R;
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.empty[st]));
      advance();
    };

    auto C_end = [&](int p) {
      const int qs = p % kPQ;
      // this warp's overlap (and E2E S-mass) terms of the unit: one path or the other
      const float a = warp_sum(__fadd_rn(__fadd_rn(ao.x, ao.y), f2_hsum(a2)));
      float g = 0.0f;
      if constexpr (MODE == kPE2E) g = warp_sum(__fadd_rn(go.x, go.y));
      if (lane == 0) {
        sm.wa[qs][warp] = a;
        sm.wg[qs][warp] = g;
        __threadfence_block();
        if (atomicAdd(&sm.cnt[qs], 1u) == (uint32_t)(kPNC - 1)) {
          // the last warp of the CTA hands the unit to the completion warp
          // (the decision slot is not reused before every warp has pushed
          // the pass-A partials of unit p + kPNX)
          __threadfence_block();
          sm.cnt[qs] = 0u;
          sm.job[qs] = sm.dec[p % kPNX];
          __threadfence_block();
          st_volatile_u32(&sm.ticket[qs], (uint32_t)p + 1u);
        }
      }
    };

    for (int p = 0; p <= nit; ++p) {
      if constexpr (!kHasC) {
        // Unit p's partials go to mailbox slot p % kPNX of every CTA, which
        // must have read unit p - kPNX from it.  A CTA that decided unit
        // p - 2 had every CTA's partials of p - 2, each pushed after that
        // CTA saw its own decision of p - 4 (this same wait).  (With pass C
        // the wait for each decision before pass C gives the same order.)
        if (p >= 2 && p < nit) {
          const int q = p - 2;
          if (!mbar_wait_bounded(smem_addr(&sm.dbar[q % kPNX]), (uint32_t)(q / kPNX) & 1u, kWaitLimitNs)) {
            if (lane == 0 && P.status) atomicOr(P.status, kTimeout);
          }
        }
      }
      for (int c = 0; c < NCH; ++c) {
        if (p < nit) A_item(p, c);
        if constexpr (kHasC) {
          if (p >= 1) {
            if (c == 0) C_begin(p - 1);
            C_item(p - 1, c);
          }
        }
      }
      if constexpr (kHasC) {
        if (p >= 1) C_end(p - 1);
      }
      // unit p goes on to pass C in the next phase
      c_okA = t_okA;
    }
    __syncwarp();
  }
  __syncthreads();
  cluster_sync();  // no CTA leaves while a peer may still read or write its shared memory
}

}  // namespace ssv
