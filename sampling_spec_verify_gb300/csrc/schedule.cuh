// Verify-length scheduling: the lengths l_1..l_R that maximise the expected
// throughput Theta = tau * SPS(B), with B = sum_r (1 + l_r) target tokens and
// tau = sum_r (1 + sum_{j<=l_r} a_{r,j}) expected produced tokens, a_{r,j} the
// prefix survival of request r at drafted position j and SPS(B) the decode
// steps per second of the serving engine at batch B ("读 Qwen Bebop 与 DeepSeek
// DSpark", section "DSpark 的第二块拼图：置信度调度验证长度").
//
// For a fixed B the best tau takes the B - R largest survivals; a row's
// survivals are non-increasing (products of acceptances), so the taken ones
// form a prefix of every row.  The whole table is put in one order (survival
// descending, ties in (row, position) order), Theta is formed for every
// prefix of that order, and the argmax (smaller B on ties) fixes the lengths.
//
// One cluster of 16 CTAs, all in distributed shared memory:
//   1. CTA c takes rows [c * rpc, (c + 1) * rpc) and sorts their survivals
//      (after the running minimum along each row) with a bitonic network;
//   2. every CTA copies its sorted run into every CTA (DSMEM stores);
//   3. each element's place in the whole order is its place in its own run
//      plus, for every other run, the number of that run's elements ahead of
//      it (a binary search);
//   4. each element's survival, in fixed point (units of 2^-48, exact integer
//      sums in any order), goes to the CTA that owns its place (places split
//      evenly over the CTAs);
//   5. every CTA sums its places' survivals, the CTAs exchange their totals,
//      and each forms Theta in fp64 for its places; the CTAs exchange their
//      best (Theta, B) and all take the same argmax;
//   6. each CTA counts its own rows' elements placed before the argmax.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace ssv {

constexpr int kSThreads = 1024;
constexpr int kSCtas = 16;             // CTAs of the cluster
constexpr int kSchedMaxItems = 16384;  // R * L
constexpr int kSchedMaxL = 64;
// Elements of one CTA's rows: ceil(R / 16) * L <= R * L / 16 + 15 * 64 / 16 <= 1084.
constexpr int kSRunCap = 1088;
constexpr int kSCtaItems = 2048;  // bitonic network width (a power of two >= kSRunCap)
constexpr int kSPlaces = kSchedMaxItems / kSCtas;  // places of the order per CTA, at most
constexpr int kSMaxRows = kSRunCap;                // rows of one CTA, at most (L = 1)

struct SchedParams {
  const float* surv;  // [R, L]
  int R, L;
  const float* sps;  // SPS(B), B = 0 .. nsps - 1
  int nsps;
  int32_t* lengths;  // [R]
  float* objective;  // [2] {Theta, tau} or null
  uint32_t* status;
};

// Shared memory of one CTA (dynamic): every run of the cluster (survival and
// flat index), this CTA's own sort, the fixed-point survivals of its places,
// and the exchanged totals and maxima.
struct SchedSmem {
  int2 run[kSCtas][kSRunCap];    // run c: (survival bits, flat index r * L + j) in order
  float sv[kSCtaItems];          // own elements during the sort
  int si[kSCtaItems];
  int grank[kSRunCap];           // own sorted run: place in the whole order
  unsigned long long pv[kSPlaces];  // survivals (2^-48 units) of this CTA's places
  unsigned long long tot[kSCtas];   // place totals of every CTA
  unsigned long long best[kSCtas];  // best Theta of every CTA (fp64 bits)
  int bestm[kSCtas];                // its B - R
  unsigned long long wsum[kSThreads / 32];
  unsigned long long wbest[kSThreads / 32];
  int wbestm[kSThreads / 32];
  int len[kSMaxRows];               // own rows' counts
  int bad;
};

// A survival in [0, 1] as an integer number of 2^-48 units (exact scaling,
// one rounding); sums of up to 2^14 of them stay below 2^63.
__device__ __forceinline__ unsigned long long sched_fixed(float v) { return __float2ull_rn(__fmul_rn(v, 0x1p48f)); }

// (va, ia) comes before (vb, ib) in the order: survival descending, ties by index.
__device__ __forceinline__ bool sched_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ int sched_rpc(int R) { return (R + kSCtas - 1) / kSCtas; }

__device__ __forceinline__ int sched_run_len(int R, int L, int c) {
  const int rpc = sched_rpc(R);
  const int r0 = min(R, c * rpc), r1 = min(R, r0 + rpc);
  return (r1 - r0) * L;
}

// Elements of a sorted run of length n before (v, i): lower bound by binary search.
__device__ __forceinline__ int sched_count_before(const int2* run, int n, float v, int i) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int2 e = run[mid];
    if (sched_before(__int_as_float(e.x), e.y, v, i))
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// One compare-exchange of the bitonic network for the element a thread
// holds, against its partner's (pv, pi): the thread at the lower place of the
// pair keeps the earlier element when the block runs in order (`up`), the
// later one otherwise; the thread at the upper place the opposite.
__device__ __forceinline__ void sched_cx(float& v, int& ix, float pv, int pi, bool lower, bool up) {
  const bool mine_first = sched_before(v, ix, pv, pi);
  const bool take = (lower == up) ? !mine_first : mine_first;
  if (take) {
    v = pv;
    ix = pi;
  }
}

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
// (Theta, B - R) pairs: larger Theta first, smaller B on ties.  Theta >= 0
// is compared through its fp64 bit pattern, which orders non-negative doubles
// like their values, so the reductions run on the integer pipe.
__device__ __forceinline__ bool sched_better(unsigned long long ta, int ma, unsigned long long tb, int mb) {
  return ta > tb || (ta == tb && ma < mb);
}

// Launched as one cluster of kSCtas CTAs.
__global__ void __launch_bounds__(kSThreads, 1) schedule_kernel(const __grid_constant__ SchedParams P) {
  extern __shared__ __align__(16) unsigned char sched_smem[];
  SchedSmem& sm = *reinterpret_cast<SchedSmem*>(sched_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = (int)cluster_rank();
  const int R = P.R, L = P.L, n = R * L;
  const int rpc = sched_rpc(R);
  const int r0 = min(R, c * rpc), r1 = min(R, r0 + rpc);
  const int m = (r1 - r0) * L;  // own elements
  const int e0 = r0 * L;        // their first flat index
  const int ppc = (n + kSCtas - 1) / kSCtas;  // places per CTA
  const int p0 = min(n, c * ppc), p1 = min(n, p0 + ppc);

  if (tid == 0) sm.bad = 0;
  __syncthreads();

  // ---- own rows: running minimum along each row, then a bitonic sort ----
  for (int i = tid; i < m; i += kSThreads) {  // coalesced load
    const float a = P.surv[e0 + i];
    if (a != a) sm.bad = 1;
    sm.sv[i] = (a != a) ? 0.0f : fmaxf(a, 0.0f);
    sm.si[i] = e0 + i;
  }
  __syncthreads();
  for (int r = tid; r < r1 - r0; r += kSThreads) {
    float run = INFINITY;
    for (int j = 0; j < L; ++j) {
      run = fminf(run, sm.sv[r * L + j]);
      sm.sv[r * L + j] = run;
    }
  }
  int w2 = 1;  // network width: a power of two >= m
  while (w2 < m) w2 <<= 1;
  for (int i = m + tid; i < w2; i += kSThreads) {  // padding sorts last
    sm.sv[i] = -1.0f;
    sm.si[i] = 0x7FFFFFFF;
  }
  __syncthreads();
  if (w2 <= kSThreads) {
    // thread t holds place t; partners closer than a warp by shuffles, the
    // others through shared memory (two buffers, one barrier per step)
    float v = (tid < w2) ? sm.sv[tid] : -1.0f;
    int ix = (tid < w2) ? sm.si[tid] : 0x7FFFFFFF;
    int buf = 0;
    for (int k = 2; k <= w2; k <<= 1) {
      const bool up = (tid & k) == 0;
      for (int j = k >> 1; j > 0; j >>= 1) {
        const bool lower = (tid & j) == 0;
        float pv;
        int pi;
        if (j < 32) {
          pv = __shfl_xor_sync(kFull, v, j);
          pi = __shfl_xor_sync(kFull, ix, j);
        } else {
          float* bv = buf ? sm.sv + kSThreads : sm.sv;
          int* bi = buf ? sm.si + kSThreads : sm.si;
          bv[tid] = v;
          bi[tid] = ix;
          __syncthreads();
          pv = bv[tid ^ j];
          pi = bi[tid ^ j];
          buf ^= 1;
        }
        sched_cx(v, ix, pv, pi, lower, up);
      }
    }
    __syncthreads();
    if (tid < w2) {
      sm.sv[tid] = v;
      sm.si[tid] = ix;
    }
    __syncthreads();
  } else {
    for (int k = 2; k <= w2; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int t = tid; t < (w2 >> 1); t += kSThreads) {
          const int i = 2 * t - (t & (j - 1));  // lower element of the pair
          const int q = i + j;
          const bool up = (i & k) == 0;  // this block ends up in order (else reversed)
          const float va = sm.sv[i], vb = sm.sv[q];
          const int ia = sm.si[i], ib = sm.si[q];
          const bool swap = up ? sched_before(vb, ib, va, ia) : sched_before(va, ia, vb, ib);
          if (swap) {
            sm.sv[i] = vb;
            sm.sv[q] = va;
            sm.si[i] = ib;
            sm.si[q] = ia;
          }
        }
        __syncthreads();
      }
    }
  }

  // ---- every run to every CTA: 16-byte stores of two (survival, index) pairs ----
  cluster_sync();  // every CTA is running before any DSMEM store
  for (int i2 = tid; 2 * i2 < m; i2 += kSThreads) {
    const int i = 2 * i2;
    const float va = sm.sv[i], vb = (i + 1 < m) ? sm.sv[i + 1] : -1.0f;
    const int ia = sm.si[i], ib = (i + 1 < m) ? sm.si[i + 1] : 0x7FFFFFFF;
    const uint32_t a = smem_addr(&sm.run[c][i]);
#pragma unroll 4
    for (int d = 0; d < kSCtas; ++d)
      st_cluster_v4(map_rank(a, (uint32_t)d), va, __int_as_float(ia), vb, __int_as_float(ib));
  }
  cluster_sync();

  // ---- place of each own element in the whole order; its survival to the place's owner ----
  for (int i = tid; i < m; i += kSThreads) {
    const float v = sm.sv[i];
    const int ix = sm.si[i];
    int g = i;
    for (int d = 0; d < kSCtas; ++d)
      if (d != c) g += sched_count_before(sm.run[d], sched_run_len(R, L, d), v, ix);
    sm.grank[i] = g;
    const int owner = g / ppc;
    st_cluster_u64(map_rank(smem_addr(&sm.pv[g - owner * ppc]), (uint32_t)owner), sched_fixed(v));
  }
  cluster_sync();

  // ---- prefix sums over this CTA's places: thread t owns [t*C, (t+1)*C) ----
  const int np = p1 - p0;
  const int C = (np + kSThreads - 1) / kSThreads;
  const int lo = min(tid * C, np), hi = min(lo + C, np);
  unsigned long long part = 0;
  for (int i = lo; i < hi; ++i) part += sm.pv[i];
  unsigned long long incl = part;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long t = sm.wsum[lane];
    unsigned long long ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(kFull, ti, o);
      if (lane >= o) ti += u;
    }
    sm.wsum[lane] = ti - t;
    if (lane == 31) {  // this CTA's total to every CTA
#pragma unroll 4
      for (int d = 0; d < kSCtas; ++d) st_cluster_u64(map_rank(smem_addr(&sm.tot[c]), (uint32_t)d), ti);
    }
  }
  cluster_sync();
  unsigned long long before = (unsigned long long)R << 48;  // R + the survivals of earlier CTAs' places
  for (int d = 0; d < c; ++d) before += sm.tot[d];
  unsigned long long run = before + sm.wsum[warp] + (incl - part);

  // ---- Theta for every B - R = place + 1; best, smaller B on ties ----
  // Theta scaled by 2^48: the scale is common to every B, so the argmax is
  // unchanged.  A NaN Theta is never taken; (0, no B) loses to every other.
  unsigned long long best = 0ull;
  int best_m = 0x7FFFFFFF;
  if (c == 0 && tid == 0) {
    const double th = (double)((unsigned long long)R << 48) * (double)P.sps[R];
    if (th == th) {
      best = (unsigned long long)__double_as_longlong(th);
      best_m = 0;
    }
  }
  for (int i = lo; i < hi; ++i) {
    run += sm.pv[i];
    const int mm = p0 + i + 1;
    const double th = (double)run * (double)__ldg(P.sps + R + mm);
    const unsigned long long tb = (unsigned long long)__double_as_longlong(th);
    if (th == th && sched_better(tb, mm, best, best_m)) {
      best = tb;
      best_m = mm;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ob = __shfl_xor_sync(kFull, best, o);
    const int om = __shfl_xor_sync(kFull, best_m, o);
    if (sched_better(ob, om, best, best_m)) {
      best = ob;
      best_m = om;
    }
  }
  if (lane == 0) {
    sm.wbest[warp] = best;
    sm.wbestm[warp] = best_m;
  }
  __syncthreads();
  if (warp == 0) {
    best = sm.wbest[lane];
    best_m = sm.wbestm[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ob = __shfl_xor_sync(kFull, best, o);
      const int om = __shfl_xor_sync(kFull, best_m, o);
      if (sched_better(ob, om, best, best_m)) {
        best = ob;
        best_m = om;
      }
    }
    if (lane < kSCtas) {  // this CTA's best to CTA `lane`
      st_cluster_u64(map_rank(smem_addr(&sm.best[c]), (uint32_t)lane), best);
      st_cluster_u32(map_rank(smem_addr(&sm.bestm[c]), (uint32_t)lane), (uint32_t)best_m);
    }
  }
  cluster_sync();
  // every CTA takes the same argmax over the CTAs' bests
  unsigned long long tbest = sm.best[0];
  int mstar = sm.bestm[0];
  for (int d = 1; d < kSCtas; ++d) {
    if (sched_better(sm.best[d], sm.bestm[d], tbest, mstar)) {
      tbest = sm.best[d];
      mstar = sm.bestm[d];
    }
  }
  if (mstar == 0x7FFFFFFF) mstar = 0;  // every Theta NaN
  const double theta = __longlong_as_double((long long)tbest);

  // ---- lengths of the own rows: own elements placed before mstar ----
  for (int r = tid; r < r1 - r0; r += kSThreads) sm.len[r] = 0;
  __syncthreads();
  for (int i = tid; i < m; i += kSThreads)
    if (sm.grank[i] < mstar) atomicAdd(&sm.len[sm.si[i] / L - r0], 1);
  __syncthreads();
  for (int r = tid; r < r1 - r0; r += kSThreads) P.lengths[r0 + r] = sm.len[r];

  // ---- the objective: tau from the place mstar - 1's running sum ----
  if (P.objective) {
    const bool mine = (mstar == 0) ? (c == 0 && tid == 0) : (mstar - 1 >= p0 + lo && mstar - 1 < p0 + hi);
    if (mine) {
      unsigned long long at = before + sm.wsum[warp] + (incl - part);
      for (int i = lo; i < mstar - p0; ++i) at += sm.pv[i];
      if (mstar == 0) at = (unsigned long long)R << 48;
      P.objective[0] = (float)(theta * 0x1p-48);
      P.objective[1] = (float)((double)at * 0x1p-48);
    }
  }
  if (tid == 0 && sm.bad && P.status) atomicOr(P.status, kBadLogits);
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace ssv
