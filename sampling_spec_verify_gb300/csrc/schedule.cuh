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
// they are merged pairwise (log2 R rounds; every thread merges a fixed slice
// of the output from its merge-path split) into one order, survival
// descending with ties in (row, position) order; exact prefix sums of the
// survivals in 2^-48 fixed point, Theta for every B in fp64, the argmax
// (smaller B on ties), and the per-row counts.
#pragma once

#include <cstdint>

namespace ssv {

constexpr int kSThreads = 1024;
constexpr int kSchedMaxItems = 16384;  // R * L held in shared memory
static_assert(kSchedMaxItems % kSThreads == 0, "positions per thread");

// Shared arrays are padded by one word every 32, so that threads walking
// their own consecutive slots (stride T or L words) hit distinct banks.
__host__ __device__ constexpr int sched_pad(int i) { return i + (i >> 5); }
__host__ __device__ constexpr size_t sched_smem_bytes(int n) {
  return 3 * (size_t)(sched_pad(n) + 1) * sizeof(int);
}

struct SchedParams {
  const float* surv;  // [R, L]
  int R, L;
  const float* sps;  // SPS(B), B = 0 .. nsps - 1
  int nsps;
  int32_t* lengths;  // [R]
  float* objective;  // [2] {Theta, tau} or null
  uint32_t* status;
};

// A survival in [0, 1] as an integer number of 2^-48 units (exact scaling,
// one rounding); sums of up to 2^14 of them stay below 2^63.
__device__ __forceinline__ unsigned long long sched_fixed(float v) { return __float2ull_rn(__fmul_rn(v, 0x1p48f)); }

// Element a precedes element b in the merged order.
__device__ __forceinline__ bool sched_before(const float* val, int a, int b) {
  const float va = val[sched_pad(a)], vb = val[sched_pad(b)];
  return va > vb || (va == vb && a < b);
}

__global__ void __launch_bounds__(kSThreads, 1) schedule_kernel(const __grid_constant__ SchedParams P) {
  extern __shared__ __align__(16) unsigned char sched_smem[];  // val, idx0, idx1: padded slots
  __shared__ unsigned long long wsum[kSThreads / 32];
  __shared__ double wbest[kSThreads / 32];
  __shared__ int wbestm[kSThreads / 32];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = P.R, L = P.L, n = R * L;
  float* val = reinterpret_cast<float*>(sched_smem);  // by item, padded slots
  int* idx0 = reinterpret_cast<int*>(val + sched_pad(n) + 1);
  int* idx1 = idx0 + sched_pad(n) + 1;
  if (tid == 0) bad = 0;
  __syncthreads();

  // ---- running minimum along each row: every row is a sorted run ----
  for (int i = tid; i < n; i += kSThreads) {  // coalesced load
    const float a = P.surv[i];
    if (a != a) bad = 1;
    val[sched_pad(i)] = (a != a) ? 0.0f : fmaxf(a, 0.0f);
    idx0[sched_pad(i)] = i;
  }
  __syncthreads();
  for (int r = tid; r < R; r += kSThreads) {
    float run = INFINITY;
    for (int j = 0; j < L; ++j) {
      run = fminf(run, val[sched_pad(r * L + j)]);
      val[sched_pad(r * L + j)] = run;
    }
  }
  __syncthreads();

  // ---- pairwise merges of runs of width w: log2(R) rounds ----
  // Thread t writes the outputs [t*T, (t+1)*T) of each round.  Inside a pair
  // of runs A, B it finds where its first output splits A and B (the merge
  // path: the number of A elements among the first d outputs, by binary
  // search), then merges sequentially.
  int* src = idx0;
  int* dst = idx1;
  const int T = (n + kSThreads - 1) / kSThreads;
  for (int w = L; w < n; w <<= 1) {
    const int o1 = min((tid + 1) * T, n);
    int o = min(tid * T, n);
    while (o < o1) {
      const int seg = (o / (2 * w)) * (2 * w);
      const int la = min(w, n - seg);
      const int lb = max(0, min(w, n - seg - w));
      auto A = [&](int k) { return src[sched_pad(seg + k)]; };
      auto Bv = [&](int k) { return src[sched_pad(seg + la + k)]; };
      const int stop = min(seg + la + lb, o1);
      const int d = o - seg;
      int lo = max(0, d - lb), hi = min(d, la);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sched_before(val, A(mid), Bv(d - 1 - mid)))
          lo = mid + 1;
        else
          hi = mid;
      }
      int i = lo, j = d - lo;
      int ea = i < la ? A(i) : -1, eb = j < lb ? Bv(j) : -1;
      for (; o < stop; ++o) {
        if (eb < 0 || (ea >= 0 && sched_before(val, ea, eb))) {
          dst[sched_pad(o)] = ea;
          ++i;
          ea = i < la ? A(i) : -1;
        } else {
          dst[sched_pad(o)] = eb;
          ++j;
          eb = j < lb ? Bv(j) : -1;
        }
      }
    }
    __syncthreads();
    int* t = src;
    src = dst;
    dst = t;
  }
  const int* order = src;  // merged order (padded slots): survival descending, ties in (row, position) order
  int* lens = dst;          // free now (R <= n): per-row counts of taken survivals
  for (int r = tid; r < R; r += kSThreads) lens[r] = 0;
  __syncthreads();

  // ---- prefix sums over sorted positions: thread t owns [t*C, (t+1)*C) ----
  // Survivals in fixed point (units of 2^-48, exact integer sums in any order)
  constexpr int kCMax = kSchedMaxItems / kSThreads;  // positions per thread at most
  const int C = (n + kSThreads - 1) / kSThreads;
  const int lo = min(tid * C, n), hi = min(lo + C, n);
  unsigned long long part = 0;
  for (int i = lo; i < hi; ++i) part += sched_fixed(val[sched_pad(order[sched_pad(i)])]);
  // block exclusive scan of the thread sums
  unsigned long long incl = part;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long t = lane < kSThreads / 32 ? wsum[lane] : 0ull;
    unsigned long long ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(kFull, ti, o);
      if (lane >= o) ti += u;
    }
    if (lane < kSThreads / 32) wsum[lane] = ti - t;
  }
  __syncthreads();
  // R + (sum of the positions before lo), in the same units: R < 2^15, so no overflow
  unsigned long long run = ((unsigned long long)R << 48) + wsum[warp] + (incl - part);

  // ---- Theta for every total m = B - R of taken survivals; best, smaller m on ties ----
  // Theta scaled by 2^48: the scale is common to every B, so the argmax is unchanged
  double best = -1.0;
  int best_m = 0x7FFFFFFF;
  if (tid == 0) {
    best = (double)((unsigned long long)R << 48) * (double)P.sps[R];
    best_m = 0;
  }
  // SPS(R + m) of 8 positions at a time is loaded ahead of the loop that uses it
  for (int k0 = 0; k0 < kCMax; k0 += 8) {
    float spv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lo + k0 + k;
      spv[k] = i < hi ? __ldg(P.sps + R + i + 1) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lo + k0 + k;
      if (i >= hi) break;
      run += sched_fixed(val[sched_pad(order[sched_pad(i)])]);
      const int m = i + 1;
      const double th = (double)run * (double)spv[k];
      if (th > best) {
        best = th;
        best_m = m;
      }
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
  unsigned long long taken = 0;
  for (int i = tid; i < mstar; i += kSThreads) {
    const int e = order[sched_pad(i)];
    atomicAdd(&lens[e / L], 1);
    taken += sched_fixed(val[sched_pad(e)]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) taken += __shfl_xor_sync(kFull, taken, o);
  __syncthreads();  // wsum reuse
  if (lane == 0) wsum[warp] = taken;
  __syncthreads();
  for (int r = tid; r < R; r += kSThreads) P.lengths[r] = lens[r];
  if (tid == 0) {
    unsigned long long tw = 0;
    for (int w = 0; w < kSThreads / 32; ++w) tw += wsum[w];
    const double tau = (double)R + (double)tw * 0x1p-48;
    if (P.objective) {
      P.objective[0] = (float)(theta * 0x1p-48);
      P.objective[1] = (float)tau;
    }
    if (bad && P.status) atomicOr(P.status, kBadLogits);
  }
}

}  // namespace ssv
