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
//   * eight consumer warps, which share every chunk (warp w takes a
//     contiguous sub-segment, lane l every 32nd vector of it);
//   * a draw warp, which runs the inverse-CDF draws of rejected and bonus
//     positions from L2-resident data, off the consumers' path.
// A unit's chunks are loaded twice: once for pass A (softmax normalisers,
// from HBM) and once more for pass C (overlap, residual weights; the copy
// hits L2, because the second load comes a few chunks after the first).  The
// ring interleaves the pass-A chunks of unit u+1 with the pass-C chunks of
// unit u, so a stage is never held while the cluster exchanges unit u's
// normalisers: every consumer warp pushes its (max, sum) pairs with st.async
// into every CTA's mailbox, completing on that CTA's mbarrier, and every warp
// combines all S x 8 pairs itself in one fixed order, so every warp of the
// cluster takes the same decision with no block or cluster barrier.
//
// Draws: each warp's per-chunk residual totals are summed per (CTA, chunk);
// the CTA whose arrival completes a drawing unit hands it to its draw warp,
// which locates the (CTA, chunk) holding u' * total, recomputes that
// chunk's weights from global memory in the same order and with the same
// arithmetic, and walks to the token.
#pragma once

#include "sweep.cuh"

namespace ssv {

constexpr int kPNC = 8;                     // consumer warps
constexpr int kPProd = kPNC;                // producer warp
constexpr int kPDraw = kPNC + 1;            // draw warp
constexpr int kPThreads = (kPNC + 2) * 32;  // 320
constexpr int kPNX = 4;                     // exchange slots (units in flight)
constexpr int kPMaxS = 16;
constexpr int kPMaxNS = 8;
constexpr int kPMaxCh = 32;     // chunks per slice
constexpr int kPMaxParts = 64;  // S x chunks per slice: draw totals per unit
constexpr int kPQ = 16;         // draw job ring

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
  float* dtot;     // [units][kPMaxParts] draw totals per (CTA, chunk)
  uint32_t* dcnt;  // [units] CTAs done with a drawing unit
  float* row_loss;
  uint32_t* row_cnt;
  uint32_t* rej;  // [B] kRejBase - (earliest rejected position seen), 0 if none
  uint32_t* glob_cnt;
  uint32_t* status;
};

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

struct DrawJob {
  int rec;
  int b;
  int resid;  // 1: residual max(0, p - q); 0: target p
  int pad;
  long long trow, drow;
  float c1t, c1d, ratio, ufin;
};

struct PipeSmem {
  uint64_t full[kPMaxNS];
  uint64_t empty[kPMaxNS];
  uint64_t xbar[kPNX];
  alignas(16) float mbox[kPNX][kPMaxS][kPNC + 1][4];  // [slot][sender CTA][sender warp | aux][field]
  float wa[kPNX][kPNC];           // warp overlap partials
  float wg[kPNX][kPNC];           // warp E2E S-mass partials
  float wt[kPNX][kPMaxCh][kPNC];  // warp draw totals per chunk
  uint32_t cnt[kPNX];             // warps done with a unit
  DrawJob q[kPQ];
  uint32_t q_ticket[kPQ];  // ticket t + 1 once job t is in its slot
  uint32_t q_res;          // jobs reserved
  uint32_t q_head;         // jobs taken by the draw warp
  uint32_t finished;       // consumer warps done
  float dsum[kPMaxParts];  // draw warp: recomputed totals (empty residual)
};

static_assert(offsetof(PipeSmem, mbox) % 16 == 0, "mailbox must be 16-byte aligned");

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

// (m, z) of one lane's vectors of a chunk: m the maximum of its first vector,
// z the sum of 2^(x s - fl(m s)); a sum not below 2^100 (a value far above
// the offset, an infinity or a NaN) is summed again with a running maximum.
template <class E>
__device__ __forceinline__ void lane_chunk_mz(const uint4* base, int i0, int i1, float s, float& m, float& z) {
  constexpr int PV = E::PV;
  m = -INFINITY;
  z = 0.0f;
  if (i0 >= i1) return;
  const f32x2 S2 = f2(s, s);
  m = E::vmax(base[i0]);
  const float c = __fmul_rn(m, s);
  const f32x2 C2 = f2(-c, -c);
  f32x2 acc = f2(0.0f, 0.0f);
  for (int i = i0; i < i1; i += 32) {
    f32x2 ep[PV / 2];
    exp_pairs<E>(base[i], S2, C2, ep);
    acc = f2_add(acc, psum(ep));
  }
  z = f2_hsum(acc);
  if (!(z < 0x1p100f) || !(c > -INFINITY)) {
    m = -INFINITY;
    z = 0.0f;
    float cm = 0.0f;
    for (int i = i0; i < i1; i += 32) {
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
}

// Total of the draw weights of one warp sub-segment [v0, v1) of a chunk
// (vector indices into `tv` / `dv`), one vector per lane per step, steps
// summed in order: the arithmetic pass C' and the draw warp both use.
// With thr >= 0 it also walks to the first element whose running sum
// exceeds thr (returned in *pick as a vector * PV + element offset from
// v0's element, or the last positive weight if none does).
template <class E, bool kResid>
__device__ __forceinline__ float seg_weights(const uint4* tv, const uint4* dv, int v0, int v1, f32x2 S2, f32x2 CT,
                                             f32x2 CD, f32x2 NR, int lane, float thr, int* pick) {
  constexpr int PV = E::PV;
  float R = 0.0f;
  int found = -1, ilast = -1;
  for (int base = v0; base < v1; base += 32) {
    const int i = base + lane;
    float w[PV];
    float ws = 0.0f;
    if (i < v1) {
      f32x2 dummy = f2(0.0f, 0.0f);
      ws = draw_weights<E, kResid>(tv[i], kResid ? dv[i] : tv[i], S2, CT, CD, NR, w, dummy);
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

// ---- the draw warp's work: one inverse-CDF draw of a unit ------------------------

template <class E, int MODE>
__device__ void pdraw(const PipeParams& P, PipeSmem& sm, const DrawJob& J, int lane) {
  constexpr int PV = E::PV;
  const int S = P.S, NCH = P.NCH, CV = P.CV, WV = P.WV;
  const int nvec_row = P.V / PV;
  const int nparts = S * NCH;
  const uint4* tv = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::Raw*>(P.target) + J.trow * P.V);
  const uint4* dv = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::Raw*>(P.draft) + J.drow * P.V);
  const f32x2 S2 = f2(P.s, P.s);
  const f32x2 CT = f2(-J.c1t, -J.c1t);
  const f32x2 CD = f2(-J.c1d, -J.c1d);
  const f32x2 NR = f2(-J.ratio, -J.ratio);
  float* dt = P.dtot + (long long)J.rec * kPMaxParts;
  auto chunk_range = [&](int jj, int& c0, int& cv) {
    const int r = jj / NCH, c = jj - r * NCH;
    const int s0 = min(r * P.NV, nvec_row);
    const int s1 = min(s0 + P.NV, nvec_row);
    c0 = min(s0 + c * CV, s1);
    cv = min(c0 + CV, s1) - c0;
  };
  bool resid = J.resid != 0;
  bool emptied = false;
  // per-(CTA, chunk) totals in prefix order, summed in order by lane 0
  for (int i = lane; i < nparts; i += 32) sm.dsum[i] = __ldcg(dt + i);
  __syncwarp();
  float total = 0.0f;
  for (int i = 0; i < nparts; ++i) total = __fadd_rn(total, sm.dsum[i]);
  if (!(total > 0.0f) && resid) {
    // no residual mass (rounding only): draw from p, recomputing every
    // chunk's target-weight total in the consumers' order
    resid = false;
    emptied = true;
    for (int jj = 0; jj < nparts; ++jj) {
      int c0, cv;
      chunk_range(jj, c0, cv);
      float t = 0.0f;
      for (int w = 0; w < kPNC; ++w) {
        const int a0 = min(w * WV, cv), a1 = min(a0 + WV, cv);
        t = __fadd_rn(t, seg_weights<E, false>(tv, dv, c0 + a0, c0 + a1, S2, CT, CD, NR, lane, -1.0f, nullptr));
      }
      if (lane == 0) sm.dsum[jj] = t;
    }
    __syncwarp();
    total = 0.0f;
    for (int i = 0; i < nparts; ++i) total = __fadd_rn(total, sm.dsum[i]);
  }
  int token = -1;
  if (total > 0.0f) {
    const float thr = __fmul_rn(J.ufin, total);
    int jsel = -1, jlast = -1;
    float cum = 0.0f, before = 0.0f;
    for (int i = 0; i < nparts; ++i) {
      const float t = sm.dsum[i];
      const float nc = __fadd_rn(cum, t);
      if (t > 0.0f) {
        jlast = i;
        if (jsel < 0 && nc > thr) {
          jsel = i;
          before = cum;
        }
      }
      cum = nc;
    }
    float thr_c = INFINITY;
    if (jsel >= 0) {
      thr_c = __fadd_rn(thr, -before);
    } else {
      jsel = jlast;
    }
    int c0, cv;
    chunk_range(jsel, c0, cv);
    // the consumers' warp order inside the chunk
    float cw = 0.0f;
    int wsel = -1, wlast = -1;
    float thr_w = INFINITY;
    for (int w = 0; w < kPNC && wsel < 0; ++w) {
      const int a0 = min(w * WV, cv), a1 = min(a0 + WV, cv);
      const float t = resid ? seg_weights<E, true>(tv, dv, c0 + a0, c0 + a1, S2, CT, CD, NR, lane, -1.0f, nullptr)
                            : seg_weights<E, false>(tv, dv, c0 + a0, c0 + a1, S2, CT, CD, NR, lane, -1.0f, nullptr);
      const float nc = __fadd_rn(cw, t);
      if (t > 0.0f) {
        wlast = w;
        if (nc > thr_c) {
          wsel = w;
          thr_w = __fadd_rn(thr_c, -cw);
        }
      }
      cw = nc;
    }
    if (wsel < 0) wsel = wlast;  // no crossing (rounding): the last positive weight
    if (wsel >= 0) {
      const int a0 = min(wsel * WV, cv), a1 = min(a0 + WV, cv);
      int pk = -1;
      if (resid)
        seg_weights<E, true>(tv, dv, c0 + a0, c0 + a1, S2, CT, CD, NR, lane, thr_w, &pk);
      else
        seg_weights<E, false>(tv, dv, c0 + a0, c0 + a1, S2, CT, CD, NR, lane, thr_w, &pk);
      if (pk >= 0) token = (c0 + a0) * PV + pk;
    }
  }
  if (lane == 0) {
    P.rec[J.rec].token = token;
    if (emptied) P.rec[J.rec].pad0 = 1u;
    P.dcnt[J.rec] = 0u;
  }
  for (int i = lane; i < nparts; i += 32) dt[i] = 0.0f;
  __syncwarp();
  parrive_row<MODE>(P, J.b, lane);
}

// ---- the kernel ------------------------------------------------------------------

template <class E, int MODE>
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
  const int NS = P.NS, NCH = P.NCH, CV = P.CV, WV = P.WV;
  const int nvec_row = P.V / PV;
  const int sv0 = min((int)rank * P.NV, nvec_row);
  const int sv1 = min(sv0 + P.NV, nvec_row);
  const size_t stage_bytes = (size_t)P.rows * (size_t)CV * 16u;
  auto stage_t = [&](int st) { return reinterpret_cast<uint4*>(dyn_smem + st * stage_bytes); };
  const uint32_t xbytes = (uint32_t)(S * (kPNC + 1) * 16);
  const int per_row = (kSampleM || kGreedyM) ? P.K + 1 : P.K;
  (void)per_row;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_addr(&sm.full[i]), 1);
      mbar_init(smem_addr(&sm.empty[i]), kPNC);
    }
    for (int i = 0; i < kPNX; ++i) {
      mbar_init(smem_addr(&sm.xbar[i]), 1);
      sm.cnt[i] = 0;
    }
    for (int i = 0; i < kPQ; ++i) sm.q_ticket[i] = 0;
    sm.q_res = 0;
    sm.q_head = 0;
    sm.finished = 0;
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
      int j = 0;
      auto issue = [&](int it, int c, bool second) {
        const int st = j % NS;
        if (j >= NS) {
          if (!mbar_wait_bounded(smem_addr(&sm.empty[st]), (uint32_t)((j / NS) - 1) & 1u, kWaitLimitNs) && P.status)
            atomicOr(P.status, kTimeout);
        }
        const PUnit x = pdecode<MODE>(P, cl + it * G);
        const int v0 = min(sv0 + c * CV, sv1);
        const int v1 = min(v0 + CV, sv1);
        const uint32_t nb = (uint32_t)(v1 - v0) * 16u;
        const uint32_t bar = smem_addr(&sm.full[st]);
        fence_proxy_async_smem();
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
      };
      for (int p = 0; p <= nit; ++p) {
        for (int c = 0; c < NCH; ++c) {
          if (p < nit) issue(p, c, false);
          if (kHasC && p >= 1) issue(p - 1, c, true);
        }
      }
      // no copy may still be in flight when the CTA exits
      for (int jj = max(0, j - NS); jj < j; ++jj)
        mbar_wait_bounded(smem_addr(&sm.full[jj % NS]), (uint32_t)(jj / NS) & 1u, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == kPDraw) {
    // ===================== draw warp =====================
    if constexpr (kSampleM) {
      uint32_t h = 0;
      uint64_t t0 = global_timer_ns();
      for (;;) {
        // lane 0 polls; the warp follows its reading
        int state = 0;  // 1: a job is ready, 2: no more jobs, 3: gave up
        if (lane == 0) {
          if (ld_volatile_u32(&sm.q_ticket[h % kPQ]) == h + 1u) {
            state = 1;
          } else if (ld_volatile_u32(&sm.finished) == (uint32_t)kPNC && ld_volatile_u32(&sm.q_res) == h) {
            state = 2;
          } else if (global_timer_ns() - t0 > kWaitLimitNs) {
            state = 3;
          }
          __threadfence_block();
        }
        state = __shfl_sync(kFull, state, 0);
        if (state == 0) {
          __nanosleep(64);
          continue;
        }
        if (state != 1) {
          if (state == 3 && lane == 0 && P.status) atomicOr(P.status, kTimeout);
          break;
        }
        const DrawJob J = sm.q[h % kPQ];
        __syncwarp();
        if (lane == 0) {
          st_volatile_u32(&sm.q_ticket[h % kPQ], 0u);
          __threadfence_block();
          st_volatile_u32(&sm.q_head, h + 1u);
        }
        ++h;
        pdraw<E, MODE>(P, sm, J, lane);
        t0 = global_timer_ns();
      }
    }
    __syncwarp();
  } else {
    // ===================== consumer warps =====================
    const f32x2 S2 = f2(P.s, P.s);
    const float s = P.s;
    int j = 0;  // ring position

    // pass-A state of the unit being read
    PUnit ax = {};
    float amt = -INFINITY, azt = 0.0f, amd = -INFINITY, azd = 0.0f;  // sampling: (m, z) pairs
    float gbt = -INFINITY, gbd = -INFINITY;                          // greedy: best values
    int git = 0x7FFFFFFF, gid = 0x7FFFFFFF;                          // greedy: their indices
    bool gnan = false;
    int a_y = -1;
    float a_ua = 0.0f, a_uf = 0.0f;
    uint32_t a_rejw = 0;
    bool a_ok = true;
    // a unit whose pass A has ended, until the end of the phase
    PUnit tx = {};
    int t_y = -1;
    float t_ua = 0.0f, t_uf = 0.0f, t_zty = 0.0f, t_zdy = 0.0f;
    bool t_okA = true;
    // the unit waiting for its exchange and pass C
    PUnit cx = {};
    int c_y = -1;
    float c_ua = 0.0f, c_uf = 0.0f, c_zty = 0.0f, c_zdy = 0.0f;
    bool c_okA = true;
    // decision of that unit
    int mode_c = 0;  // 0: overlap only, 1: residual, 2: target draw, 3: invalid
    bool draw = false, need_a = false;
    int acc = 1, am_t = -1, am_d = -1;
    float c1t = 0.0f, c1d = 0.0f, cd2 = 0.0f, izt = 0.0f, ratio = 0.0f;
    f32x2 a2 = f2(0.0f, 0.0f), g2 = f2(0.0f, 0.0f);
    // rejection seen earlier in the current row (this cluster's own decisions)
    int lrow = -1;
    bool lrej = false;

    auto A_item = [&](int p, int c) {
      const int st = j % NS;
      const uint32_t par = (uint32_t)(j / NS) & 1u;
      ++j;
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
        if (lane == 0) {
          const long long di = (long long)ax.b * P.K + ax.k;
          if constexpr (kSampleM || kGreedyM) a_y = ax.bonus ? -1 : __ldg(P.draft_tokens + di);
          if constexpr (kSampleM) {
            a_ua = ax.bonus ? 0.0f : __ldg(P.u_accept + di);
            a_uf = __ldg(P.u_final + ax.b);
            a_rejw = (rank == 0 && warp == 0) ? __ldcg(P.rej + ax.b) : 0u;
          }
        }
      }
      const bool ok = mbar_wait_bounded(smem_addr(&sm.full[st]), par, kWaitLimitNs);
      if (!ok) {
        a_ok = false;
        if (lane == 0 && P.status) atomicOr(P.status, kTimeout);
      }
      const int v0 = min(sv0 + c * CV, sv1);
      const int cv = min(v0 + CV, sv1) - v0;
      const int w0 = min(warp * WV, cv), w1 = min(w0 + WV, cv);
      const uint4* stt = stage_t(st);
      const uint4* sdd = stt + CV;
      if (ok) {
        if constexpr (kGreedyM) {
          // packed maxima per vector; the winning vector is unpacked below
          float bt = -INFINITY, bd = -INFINITY;
          int jt = -1, jd = -1;
          for (int i = w0 + lane; i < w1; i += 32) {
            bool nn;
            float vm = E::vmax_nan(stt[i], nn);
            gnan |= nn;
            if (vm > bt) {
              bt = vm;
              jt = i;
            }
            if (ax.has_draft) {
              vm = E::vmax_nan(sdd[i], nn);
              gnan |= nn;
              if (vm > bd) {
                bd = vm;
                jd = i;
              }
            }
          }
          // earlier chunks hold smaller indices: a later chunk wins only if larger
          if (jt >= 0 && bt > gbt) {
            float xv[PV];
            E::unpack(stt[jt], xv);
            int e = PV - 1;
            for (int q = PV - 1; q >= 0; --q)
              if (xv[q] == bt) e = q;
            gbt = bt;
            git = (v0 + jt) * PV + e;
          }
          if (jd >= 0 && bd > gbd) {
            float xv[PV];
            E::unpack(sdd[jd], xv);
            int e = PV - 1;
            for (int q = PV - 1; q >= 0; --q)
              if (xv[q] == bd) e = q;
            gbd = bd;
            gid = (v0 + jd) * PV + e;
          }
        } else {
          float m, z;
          lane_chunk_mz<E>(stt, w0 + lane, w1, s, m, z);
          mz_merge(amt, azt, m, z, s);
          if (ax.has_draft) {
            lane_chunk_mz<E>(sdd, w0 + lane, w1, s, m, z);
            mz_merge(amd, azd, m, z, s);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.empty[st]));
      if (c == NCH - 1) {
        // this warp's share of the unit: to every CTA of the cluster
        const int slot = p % kPNX;
        float f0, f1, f2_, f3;
        if constexpr (kGreedyM) {
          warp_argmax_redux(gbt, git);
          warp_argmax_redux(gbd, gid);
          const bool nn = __any_sync(kFull, gnan);
          f0 = gbt;
          f1 = __int_as_float(git);
          f2_ = nn ? __int_as_float(0x7FC00000) : gbd;  // a NaN anywhere poisons the draft value
          f3 = __int_as_float(gid);
          if (nn) f0 = __int_as_float(0x7FC00000);
        } else {
          warp_combine_mz2(amt, azt, amd, azd, s);
          f0 = amt;
          f1 = azt;
          f2_ = amd;
          f3 = azd;
        }
        const uint32_t rjw = __shfl_sync(kFull, a_rejw, 0);
        const float aok = __all_sync(kFull, a_ok) ? 0.0f : 1.0f;
        if (lane < S) {
          const uint32_t a = map_rank(smem_addr(&sm.mbox[slot][rank][warp][0]), (uint32_t)lane);
          const uint32_t bar = map_rank(smem_addr(&sm.xbar[slot]), (uint32_t)lane);
          st_async_v4(a, f0, f1, f2_, f3, bar);
          if (warp == 0) {
            const uint32_t ax_ = map_rank(smem_addr(&sm.mbox[slot][rank][kPNC][0]), (uint32_t)lane);
            st_async_v4(ax_, __uint_as_float(rjw), aok, 0.0f, 0.0f, bar);
          }
        }
        // hand the unit over; pass C takes it at the end of this phase
        tx = ax;
        t_okA = __all_sync(kFull, a_ok);
        t_y = __shfl_sync(kFull, a_y, 0);
        t_ua = __shfl_sync(kFull, a_ua, 0);
        t_uf = __shfl_sync(kFull, a_uf, 0);
        t_zty = 0.0f;
        t_zdy = 0.0f;
        if constexpr (kSampleM) {
          // gathered logits of the drafted token (read from L2 while pass C of
          // the previous unit runs)
          if (lane == 0 && !tx.bonus && t_y >= 0 && t_y < P.V) {
            t_zty = E::to_f32(__ldg(reinterpret_cast<const Raw*>(P.target) + tx.trow * P.V + t_y));
            t_zdy = E::to_f32(__ldg(reinterpret_cast<const Raw*>(P.draft) + tx.drow * P.V + t_y));
          }
        }
      }
    };

    auto C_begin = [&](int p) {
      const int slot = p % kPNX;
      const uint32_t xpar = (uint32_t)(p / kPNX) & 1u;
      if (!mbar_wait_bounded(smem_addr(&sm.xbar[slot]), xpar, kWaitLimitNs)) {
        if (lane == 0 && P.status) atomicOr(P.status, kTimeout);
      }
      if (warp == 0 && lane == 0 && p + kPNX < nit) mbar_arrive_expect_tx(smem_addr(&sm.xbar[slot]), xbytes);
      const int ne = S * (kPNC + 1);
      const bool tok_ok = cx.bonus || (c_y >= 0 && c_y < P.V);
      uint32_t flags = 0;
      a2 = f2(0.0f, 0.0f);
      g2 = f2(0.0f, 0.0f);
      draw = false;
      need_a = false;
      if constexpr (kGreedyM) {
        float v1 = -INFINITY, v2 = -INFINITY;
        int i1 = 0x7FFFFFFF, i2 = 0x7FFFFFFF;
        bool nn = false;
        for (int e = lane; e < ne; e += 32) {
          const int r = e / (kPNC + 1), w = e - r * (kPNC + 1);
          if (w == kPNC) continue;
          const float* mm = sm.mbox[slot][r][w];
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
          const float* mm = sm.mbox[slot][r][w];
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
          const uint32_t seen = __float_as_uint(sm.mbox[slot][0][kPNC][0]);
          if (cx.b != lrow) {
            lrow = cx.b;
            lrej = false;
          }
          const bool earlier = lrej || (seen > kRejBase - (uint32_t)cx.k);
          if (cx.bonus) {
            mode_c = 2;
          } else {
            // u * q(y) <= p(y), with p(y), q(y) formed like the per-element values
            const float zty = __shfl_sync(kFull, c_zty, 0), zdy = __shfl_sync(kFull, c_zdy, 0);
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
            if (rank == 0 && warp == 0 && lane == 0) atomicMax(&P.rej[cx.b], kRejBase - (uint32_t)cx.k);
            lrej = true;
          }
          if (mode_c == 2) {
            draw = !earlier;
          } else if (mode_c == 1) {
            draw = !earlier;
          }
          need_a = cx.has_draft && P.alpha != nullptr && mode_c != 3;
        } else {
          if (!valid) {
            flags |= kBadLogits;
            mode_c = 3;
          }
          need_a = (mode_c == 0);
        }
      }
      if (!c_okA) flags |= kTimeout;
      if (flags && rank == 0 && warp == 0 && lane == 0 && P.status) atomicOr(P.status, flags);
    };

    auto C_item = [&](int p, int c) {
      const int st = j % NS;
      const uint32_t par = (uint32_t)(j / NS) & 1u;
      ++j;
      const int slot = p % kPNX;
      const bool ok = mbar_wait_bounded(smem_addr(&sm.full[st]), par, kWaitLimitNs);
      if (!ok && lane == 0 && P.status) atomicOr(P.status, kTimeout);
      const int v0 = min(sv0 + c * CV, sv1);
      const int cv = min(v0 + CV, sv1) - v0;
      const int w0 = min(warp * WV, cv), w1 = min(w0 + WV, cv);
      const uint4* stt = stage_t(st);
      const uint4* sdd = stt + CV;
      const f32x2 CT = f2(-c1t, -c1t);
      if (ok) {
        if (mode_c == 0 && need_a) {
          // overlap (and E2E S-mass) terms: one exp per element of min(log p, log q)
          const f32x2 CD = f2(-cd2, -cd2);
          for (int i = w0 + lane; i < w1; i += 32) {
            f32x2 pt[PV / 2], pd[PV / 2], ep[PV / 2], gp[PV / 2];
            E::pairs(stt[i], pt);
            E::pairs(sdd[i], pd);
#pragma unroll
            for (int h = 0; h < PV / 2; ++h) {
              float t0, t1, d0, d1;
              f2_split(f2_fma(pt[h], S2, CT), t0, t1);
              f2_split(f2_fma(pd[h], S2, CD), d0, d1);
              const float e0 = ex2(fminf(t0, d0)), e1 = ex2(fminf(t1, d1));
              ep[h] = f2(e0, e1);
              if constexpr (MODE == kPE2E) gp[h] = f2(d0 < t0 ? e0 : 0.0f, d1 < t1 ? e1 : 0.0f);
            }
            a2 = f2_add(a2, psum(ep));
            if constexpr (MODE == kPE2E) g2 = f2_add(g2, psum(gp));
          }
        } else if constexpr (kSampleM) {
          if (mode_c == 1 && (draw || need_a)) {
            // residual weights; the overlap from the same arithmetic
            const f32x2 CDd = f2(-c1d, -c1d);
            const f32x2 NR = f2(-ratio, -ratio);
            if (draw) {
              float R = 0.0f;
              for (int base = w0; base < w1; base += 32) {
                const int i = base + lane;
                float w[PV];
                float ws = 0.0f;
                if (i < w1) ws = draw_weights<E, true>(stt[i], sdd[i], S2, CT, CDd, NR, w, a2);
                R = __fadd_rn(R, __shfl_sync(kFull, warp_incl_scan(ws, lane), 31));
              }
              if (lane == 0) sm.wt[slot][c][warp] = R;
            } else {
              for (int i = w0 + lane; i < w1; i += 32) {
                float w[PV];
                draw_weights<E, true>(stt[i], sdd[i], S2, CT, CDd, NR, w, a2);
              }
            }
          } else if (mode_c == 2 && draw) {
            float R = 0.0f;
            const f32x2 Z2 = f2(0.0f, 0.0f);
            for (int base = w0; base < w1; base += 32) {
              const int i = base + lane;
              float w[PV];
              float ws = 0.0f;
              f32x2 dummy = Z2;
              if (i < w1) ws = draw_weights<E, false>(stt[i], stt[i], S2, CT, CT, Z2, w, dummy);
              R = __fadd_rn(R, __shfl_sync(kFull, warp_incl_scan(ws, lane), 31));
            }
            if (lane == 0) sm.wt[slot][c][warp] = R;
          }
        }
      } else if (draw && lane == 0) {
        sm.wt[slot][c][warp] = 0.0f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.empty[st]));
    };

    auto C_end = [&](int p) {
      const int slot = p % kPNX;
      if constexpr (kGreedyM) {
        if (rank == 0 && warp == 0) {
          if (lane == 0) {
            VerifyRecord r;
            r.acc = acc;
            r.token = am_t;
            r.pad0 = r.pad1 = 0u;
            P.rec[cx.rec] = r;
            if (cx.has_draft)
              P.part[(long long)cx.rec * kPartStride] = (am_t >= 0 && am_t == am_d) ? 1.0f : 0.0f;
          }
          __syncwarp();
          parrive_row<MODE>(P, cx.b, lane);
        }
        return;
      } else {
        const float a = warp_sum(f2_hsum(a2));
        float g = 0.0f;
        if constexpr (MODE == kPE2E) g = warp_sum(f2_hsum(g2));
        int last = 0;
        if (lane == 0) {
          sm.wa[slot][warp] = a;
          sm.wg[slot][warp] = g;
          __threadfence_block();
          last = (atomicAdd(&sm.cnt[slot], 1u) == (uint32_t)(kPNC - 1)) ? 1 : 0;
          if (last) {
            __threadfence_block();
            sm.cnt[slot] = 0u;
          }
        }
        last = __shfl_sync(kFull, last, 0);
        if (!last) return;
        // this warp finishes the CTA's share of the unit
        const float nanv = __int_as_float(0x7FC00000);
        if (lane == 0) {
          if (cx.has_draft && (!kSampleM || P.alpha != nullptr)) {
            float A = 0.0f;
            for (int w = 0; w < kPNC; ++w) A = __fadd_rn(A, sm.wa[slot][w]);
            P.part[(long long)cx.rec * kPartStride + rank] = (mode_c == 3) ? nanv : __fmul_rn(A, izt);
          }
          if constexpr (MODE == kPE2E) {
            float M2 = 0.0f;
            for (int w = 0; w < kPNC; ++w) M2 = __fadd_rn(M2, sm.wg[slot][w]);
            P.part2[(long long)cx.rec * kPartStride + rank] = (mode_c == 3) ? nanv : __fmul_rn(M2, izt);
            if (rank == 0) {
              E2EStats e2;
              e2.c1t = c1t;
              e2.cd = cd2;
              e2.izt = izt;
              e2.smass = e2.alpha = e2.b1 = e2.b0 = e2.pad = 0.0f;
              P.stats[cx.rec] = e2;
            }
          }
          if constexpr (kSampleM) {
            if (rank == 0) {
              P.rec[cx.rec].acc = cx.bonus ? 1 : acc;
              if (!draw) P.rec[cx.rec].token = -1;
            }
          }
        }
        if constexpr (kSampleM) {
          if (draw) {
            // per-chunk totals of this CTA, warps in order
            float* dt = P.dtot + (long long)cx.rec * kPMaxParts + (long long)rank * NCH;
            for (int c = lane; c < NCH; c += 32) {
              float t = 0.0f;
              for (int w = 0; w < kPNC; ++w) t = __fadd_rn(t, sm.wt[slot][c][w]);
              dt[c] = t;
            }
            __syncwarp();
            int drawer = 0;
            if (lane == 0) {
              __threadfence();
              drawer = (atomicAdd(&P.dcnt[cx.rec], 1u) == (uint32_t)(S - 1)) ? 1 : 0;
              if (drawer) {
                __threadfence();
                // hand the draw to this CTA's draw warp
                const uint32_t t = atomicAdd(&sm.q_res, 1u);
                const uint64_t w0t = global_timer_ns();
                while (t - ld_volatile_u32(&sm.q_head) >= (uint32_t)kPQ) {
                  __nanosleep(64);
                  if (global_timer_ns() - w0t > kWaitLimitNs) {
                    if (P.status) atomicOr(P.status, kTimeout);
                    break;
                  }
                }
                DrawJob J;
                J.rec = cx.rec;
                J.b = cx.b;
                J.resid = (mode_c == 1) ? 1 : 0;
                J.pad = 0;
                J.trow = cx.trow;
                J.drow = cx.drow;
                J.c1t = c1t;
                J.c1d = c1d;
                J.ratio = ratio;
                J.ufin = c_uf;
                sm.q[t % kPQ] = J;
                __threadfence_block();
                st_volatile_u32(&sm.q_ticket[t % kPQ], t + 1u);
              }
            }
            drawer = __shfl_sync(kFull, drawer, 0);
            if (drawer) return;  // the draw warp arrives for this CTA once the token is written
          }
        }
        __syncwarp();
        parrive_row<MODE>(P, cx.b, lane);
      }
    };

    for (int p = 0; p <= nit; ++p) {
      for (int c = 0; c < NCH; ++c) {
        if (p < nit) A_item(p, c);
        if constexpr (kHasC) {
          if (p >= 1) {
            if (c == 0) C_begin(p - 1);
            C_item(p - 1, c);
          }
        }
      }
      if (p >= 1) {
        if constexpr (!kHasC) C_begin(p - 1);
        C_end(p - 1);
      }
      // unit p goes on to pass C in the next phase
      cx = tx;
      c_y = t_y;
      c_ua = t_ua;
      c_uf = t_uf;
      c_zty = t_zty;
      c_zdy = t_zdy;
      c_okA = t_okA;
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      atomicAdd(&sm.finished, 1u);
    }
  }
  __syncthreads();
  cluster_sync();  // no CTA leaves while a peer may still read or write its shared memory
}

}  // namespace ssv
