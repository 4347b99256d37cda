// Verify-length scheduling: the lengths l_1..l_R that maximise the expected
// throughput Theta = tau * SPS(B), with B = sum_r (1 + l_r) target tokens and
// tau = sum_r (1 + sum_{j<=l_r} a_{r,j}) expected produced tokens, a_{r,j} the
// prefix survival of request r at drafted position j and SPS(B) the decode
// steps per second of the serving engine at batch B ("读 Qwen Bebop 与 DeepSeek
// DSpark", section "DSpark 的第二块拼图：置信度调度验证长度").
//
// For a fixed B the best tau takes the B - R largest survivals; a row's
// survivals are non-increasing (products of acceptances), so the taken ones
// form a prefix of every row.  One CTA: the rows are already sorted runs, so
// they are merged pairwise (log2 R rounds; every element finds its place by a
// binary search in the partner run) into one order, survival descending with
// ties in (row, position) order; prefix sums in fp64, Theta for every B, the
// argmax (smaller B on ties), and the per-row counts.
#pragma once

#include <cstdint>

namespace ssv {

constexpr int kSThreads = 1024;
constexpr int kSchedMaxItems = 16384;  // R * L held in shared memory

struct SchedParams {
  const float* surv;  // [R, L]
  int R, L;
  const float* sps;  // SPS(B), B = 0 .. nsps - 1
  int nsps;
  int32_t* lengths;  // [R]
  float* objective;  // [2] {Theta, tau} or null
  uint32_t* status;
};

// Element a precedes element b in the merged order.
__device__ __forceinline__ bool sched_before(const float* val, int a, int b) {
  const float va = val[a], vb = val[b];
  return va > vb || (va == vb && a < b);
}

__global__ void __launch_bounds__(kSThreads, 1) schedule_kernel(const __grid_constant__ SchedParams P) {
  extern __shared__ __align__(16) unsigned char sched_smem[];  // val[n], idx[2][n]
  __shared__ double wsum[kSThreads / 32];
  __shared__ double wbest[kSThreads / 32];
  __shared__ int wbestm[kSThreads / 32];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = P.R, L = P.L, n = R * L;
  float* val = reinterpret_cast<float*>(sched_smem);
  int* idx0 = reinterpret_cast<int*>(val + n);
  int* idx1 = idx0 + n;
  if (tid == 0) bad = 0;
  __syncthreads();

  // ---- running minimum along each row: every row is a sorted run ----
  for (int r = tid; r < R; r += kSThreads) {
    float run = INFINITY;
    int nan = 0;
    for (int j = 0; j < L; ++j) {
      float a = P.surv[(long long)r * L + j];
      if (a != a) {
        a = 0.0f;
        nan = 1;
      }
      run = fminf(run, fmaxf(a, 0.0f));
      val[r * L + j] = run;
      idx0[r * L + j] = r * L + j;
    }
    if (nan) bad = 1;
  }
  __syncthreads();

  // ---- pairwise merges of runs of width w: log2(R) rounds ----
  int* src = idx0;
  int* dst = idx1;
  for (int w = L; w < n; w <<= 1) {
    for (int p = tid; p < n; p += kSThreads) {
      const int run = p / w;
      const int start = run * w;
      const int e = src[p];
      const int pstart = (run & 1) ? start - w : start + w;  // the partner run
      int out = p;
      if (pstart < n) {
        const int plen = min(w, n - pstart);
        // elements of the partner run that precede e (all keys are distinct)
        int lo = 0, hi = plen;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (sched_before(val, src[pstart + mid], e))
            lo = mid + 1;
          else
            hi = mid;
        }
        out = min(start, pstart) + (p - start) + lo;
      }
      dst[out] = e;
    }
    __syncthreads();
    int* t = src;
    src = dst;
    dst = t;
  }
  const int* order = src;  // merged order: survival descending, ties in (row, position) order
  int* lens = dst;          // free now (R <= n): per-row counts of taken survivals
  for (int r = tid; r < R; r += kSThreads) lens[r] = 0;
  __syncthreads();

  // ---- prefix sums over sorted positions: thread t owns [t*C, (t+1)*C) ----
  const int C = (n + kSThreads - 1) / kSThreads;
  const int lo = min(tid * C, n), hi = min(lo + C, n);
  double part = 0.0;
  for (int i = lo; i < hi; ++i) part += (double)val[order[i]];
  // block exclusive scan of the thread sums
  double incl = part;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const double t = lane < kSThreads / 32 ? wsum[lane] : 0.0;
    double ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double u = __shfl_up_sync(kFull, ti, o);
      if (lane >= o) ti += u;
    }
    if (lane < kSThreads / 32) wsum[lane] = ti - t;
  }
  __syncthreads();
  double run = wsum[warp] + (incl - part);  // sum of the positions before lo

  // ---- Theta for every total m = B - R of taken survivals; best, smaller m on ties ----
  double best = -1.0;
  int best_m = 0x7FFFFFFF;
  if (tid == 0) {
    best = (double)R * (double)P.sps[R];
    best_m = 0;
  }
  for (int i = lo; i < hi; ++i) {
    run += (double)val[order[i]];
    const int m = i + 1;
    const double th = ((double)R + run) * (double)P.sps[R + m];
    if (th > best) {
      best = th;
      best_m = m;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ob = __shfl_xor_sync(kFull, best, o);
    const int om = __shfl_xor_sync(kFull, best_m, o);
    if (ob > best || (ob == best && om < best_m)) {
      best = ob;
      best_m = om;
    }
  }
  if (lane == 0) {
    wbest[warp] = best;
    wbestm[warp] = best_m;
  }
  __syncthreads();
  if (warp == 0) {
    best = lane < kSThreads / 32 ? wbest[lane] : -1.0;
    best_m = lane < kSThreads / 32 ? wbestm[lane] : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ob = __shfl_xor_sync(kFull, best, o);
      const int om = __shfl_xor_sync(kFull, best_m, o);
      if (ob > best || (ob == best && om < best_m)) {
        best = ob;
        best_m = om;
      }
    }
    if (lane == 0) {
      wbest[0] = best;
      wbestm[0] = best_m;
    }
  }
  __syncthreads();
  const int mstar = wbestm[0];
  const double theta = wbest[0];

  // ---- lengths: taken positions per row; tau ----
  double taken = 0.0;
  for (int i = tid; i < mstar; i += kSThreads) {
    const int e = order[i];
    atomicAdd(&lens[e / L], 1);
    taken += (double)val[e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) taken += __shfl_xor_sync(kFull, taken, o);
  __syncthreads();  // wsum reuse
  if (lane == 0) wsum[warp] = taken;
  __syncthreads();
  for (int r = tid; r < R; r += kSThreads) P.lengths[r] = lens[r];
  if (tid == 0) {
    double tau = (double)R;
    for (int w = 0; w < kSThreads / 32; ++w) tau += wsum[w];
    if (P.objective) {
      P.objective[0] = (float)theta;
      P.objective[1] = (float)tau;
    }
    if (bad && P.status) atomicOr(P.status, kBadLogits);
  }
}

}  // namespace ssv
