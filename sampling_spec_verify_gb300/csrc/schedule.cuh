// Verify-length scheduling: the lengths l_1..l_R that maximise the expected
// throughput Theta = tau * SPS(B), with B = sum_r (1 + l_r) target tokens and
// tau = sum_r (1 + sum_{j<=l_r} a_{r,j}) expected produced tokens, a_{r,j} the
// prefix survival of request r at drafted position j and SPS(B) the decode
// steps per second of the serving engine at batch B ("读 Qwen Bebop 与 DeepSeek
// DSpark", section "DSpark 的第二块拼图：置信度调度验证长度").
//
// For a fixed B the best tau takes the B - R largest survivals; a row's
// survivals are non-increasing (products of acceptances), so the taken ones
// form a prefix of every row.  One CTA: sort all survivals (bitonic, in shared
// memory, descending, ties in (row, position) order), prefix sums in fp64,
// Theta for every B, the argmax (smaller B on ties), and the per-row counts.
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

__global__ void __launch_bounds__(kSThreads, 1) schedule_kernel(const __grid_constant__ SchedParams P) {
  extern __shared__ __align__(16) unsigned long long keys[];  // [N] then int lens[R]
  __shared__ double wsum[kSThreads / 32];
  __shared__ double wbest[kSThreads / 32];
  __shared__ int wbestm[kSThreads / 32];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = P.R, L = P.L, n = R * L;
  int N = 1;
  while (N < n) N <<= 1;
  int* lens = reinterpret_cast<int*>(keys + N);
  if (tid == 0) bad = 0;
  __syncthreads();

  // ---- keys: running minimum along each row (survival bits << 32 | ~index) ----
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
      const uint32_t idx = (uint32_t)(r * L + j);
      keys[idx] = ((unsigned long long)__float_as_uint(run) << 32) | (unsigned long long)(~idx);
    }
    lens[r] = 0;
    if (nan) bad = 1;
  }
  for (int i = n + tid; i < N; i += kSThreads) keys[i] = 0ull;  // below every real key
  __syncthreads();

  // ---- bitonic sort, descending; thread work is over pairs (i, i + j), i's bit j clear ----
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int q = tid; q < (N >> 1); q += kSThreads) {
        const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1));
        const int p = i + j;
        const unsigned long long a = keys[i], b = keys[p];
        const bool desc = (i & k) == 0;
        if (desc ? (a < b) : (a > b)) {
          keys[i] = b;
          keys[p] = a;
        }
      }
      __syncthreads();
    }
  }

  // ---- prefix sums over sorted positions: thread t owns [t*C, (t+1)*C) ----
  const int C = (n + kSThreads - 1) / kSThreads;
  const int lo = min(tid * C, n), hi = min(lo + C, n);
  double part = 0.0;
  for (int i = lo; i < hi; ++i) part += (double)__uint_as_float((uint32_t)(keys[i] >> 32));
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
    run += (double)__uint_as_float((uint32_t)(keys[i] >> 32));
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
    const uint32_t idx = ~(uint32_t)(keys[i] & 0xFFFFFFFFull);
    atomicAdd(&lens[idx / (uint32_t)L], 1);
    taken += (double)__uint_as_float((uint32_t)(keys[i] >> 32));
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
