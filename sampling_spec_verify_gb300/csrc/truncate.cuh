// Top-k / top-p truncation of logit rows, applied the same way to target and
// draft logits before a verify step.
//
// "Speculative Decoding 与 MTP", section 4: p and q must both be computed after
// the agreed temperature and top-k / top-p transforms; section 23: a mask that
// only one side applies breaks correctness.  The transform: rank tokens by
// logit (larger first, ties to the smaller index); top-k keeps the first
// top_k; top-p renormalises softmax(z / T) over what is left and keeps the
// shortest ranked prefix whose mass reaches top_p; dropped logits become -inf.
//
// One CTA per row; every pass streams the row through L2 (the first one from
// HBM).  Keys are order-preserving 16-bit (bf16) or 32-bit (fp32) images of
// the logits.  Warp w always walks the same contiguous chunk of the row, so
// per-warp counts give ordered compaction.
// bf16 rows take the value-histogram path first: the maximum pass also counts
// every bf16 value (one bin per value, three merged bins for the extremes);
// both cuts are read off the histogram, the top-p masses as count x mass of
// each value; the write pass keeps every element of the last cut's key, marks
// them in a bitmap and drops the ones past the kept count.  Two passes in
// all, unless a cut falls in a merged bin: then the row takes the radix path:
//  1. maximum and NaN check;
//  2. top-k: for bf16, per-warp counts of the 256 keys just below the
//     maximum's (one bin per key), which hold the top_k-th key in the usual
//     case; the tied tokens of the threshold key are compacted, in index
//     order, only when some of them are cut.  Otherwise (fp32, or a threshold
//     further down) per-warp counts of the first digit; the crossing digit's
//     elements are compacted, in index order, into shared memory, and the
//     remaining digits and the index-order tie are resolved on that list;
//  3. top-p: per-warp fixed-point masses (2^44 for the row maximum, summed as
//     integers, so every cut is independent of the order of the additions)
//     and counts of the first digit over the top-k set; the same compaction
//     and list selection by mass;
//  4. the write pass.
// A digit holding more than kTCap elements falls back to radix passes over
// the whole row.  Histograms are per warp, so atomics conflict only between
// the lanes of one warp.
#pragma once

#include <cstdint>

namespace ssv {

constexpr int kTThreads = 512;
constexpr int kTWarps = kTThreads / 32;
constexpr float kMassScale = 0x1p44f;  // fixed-point unit of the top-p masses
constexpr int kTCap = 6144;            // candidates held in shared memory after the first digit

struct TruncParams {
  const void* in;
  void* out;  // may equal in
  int rows, V;
  int aligned;  // in and out rows on 16-byte boundaries and V * elem a multiple of 16
  float s;      // log2(e) / T
  int top_k;    // active when 0 < top_k < V
  float top_p;  // active when top_p < 1
  uint32_t* status;
};

struct TruncSmem {
  unsigned long long ph[kTWarps][256];  // per-warp histograms of one radix pass
  uint32_t pc[kTWarps][256];            // per-warp counts of the first digit (compaction offsets)
  int cand_idx[kTCap];                  // candidates of the crossing first digit, in index order
  float cand_x[kTCap];
  unsigned long long hist[256];
  unsigned long long wtot[kTWarps];
  float wmax[kTWarps];
  int wnan[kTWarps];
  unsigned long long bc;
  int bin;
  int tie;
  uint32_t wc[kTWarps];           // per-warp counts of a tie walk
  int xbin;                       // crossing bin of the value histogram
  unsigned long long xabove;      // weight above it
};

// Per-warp 32-bit limb counters, kept in the candidate arrays' storage while a
// histogram pass runs (the list is not in use then): a weight w <= 2^44 adds
// its low 22 bits to lo[d] and the rest to hi[d] with native 32-bit shared
// atomics, and every 3 steps of 256 elements the limbs are folded into the
// warp's 64-bit histogram, before either could overflow.
struct Limbs {
  uint32_t* lo;
  uint32_t* hi;
  unsigned long long* ph;
  int steps;
  bool dirty;  // limbs may be nonzero
  __device__ __forceinline__ Limbs(TruncSmem& sm, int warp)
      : lo(reinterpret_cast<uint32_t*>(sm.cand_idx) + warp * 256),
        hi(reinterpret_cast<uint32_t*>(sm.cand_x) + warp * 256),
        ph(sm.ph[warp]),
        steps(0),
        dirty(false) {}
  __device__ __forceinline__ void zero(int lane) {
    for (int b = lane; b < 256; b += 32) {
      lo[b] = 0u;
      hi[b] = 0u;
      ph[b] = 0ull;
    }
    __syncwarp();
  }
  __device__ __forceinline__ void add(uint32_t d, unsigned long long w) {
    atomicAdd(lo + d, (uint32_t)(w & 0x3FFFFFull));
    const uint32_t h = (uint32_t)(w >> 22);
    if (h) atomicAdd(hi + d, h);
  }
  __device__ __forceinline__ void flush(int lane) {
    if (!dirty) return;
    dirty = false;
    __syncwarp();
    for (int b = lane; b < 256; b += 32) {
      ph[b] += (unsigned long long)lo[b] + ((unsigned long long)hi[b] << 22);
      lo[b] = 0u;
      hi[b] = 0u;
    }
    __syncwarp();
  }
  // once per 32 lanes x PV elements, warp-converged; added: this lane added a weight
  __device__ __forceinline__ void step(int lane, bool added) {
    dirty |= __any_sync(kFull, added);
    if (++steps == 3) {
      flush(lane);
      steps = 0;
    }
  }
};
static_assert(sizeof(int) * kTCap >= kTWarps * 256 * sizeof(uint32_t), "limbs fit in the candidate storage");

// Order-preserving key of a logit (larger value, larger key), -0 folded onto
// +0, keeping the top KB bits (16 for bf16 values, whose low bits are zero).
template <int KB>
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return k >> (32 - KB);
}

// The value whose key is k (inverse of order_key).
template <int KB>
__device__ __forceinline__ float key_value(uint32_t k) {
  uint32_t k32 = k << (32 - KB);
  if (KB < 32 && !(k32 & 0x80000000u)) k32 |= (1u << (32 - KB)) - 1u;  // negative: low bits were ones
  const uint32_t u = (k32 & 0x80000000u) ? (k32 & 0x7FFFFFFFu) : ~k32;
  return __uint_as_float(u);
}

// Fixed-point mass of a logit x against the row maximum M: round(2^((x - M) s) * 2^44).
__device__ __forceinline__ unsigned long long fixed_mass(float x, float M, float s) {
  return __float2ull_rn(__fmul_rn(ex2(__fmul_rn(__fsub_rn(x, M), s)), kMassScale));
}

// Calls f(v, x) for every element of the row: coalesced 16-byte loads when the
// row is aligned, element loads otherwise.
constexpr int kTUnroll = 4;  // independent 16-byte loads in flight per thread

template <class E, class F>
__device__ __forceinline__ void for_each_elem(const typename E::Raw* row, int V, bool aligned, F&& f) {
  if (aligned) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int nvec = V / E::PV;
    for (int i0 = threadIdx.x; i0 < nvec; i0 += kTThreads * kTUnroll) {
      uint4 w[kTUnroll];
#pragma unroll
      for (int u = 0; u < kTUnroll; ++u) {
        const int i = i0 + u * kTThreads;
        w[u] = i < nvec ? __ldcg(r4 + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kTUnroll; ++u) {
        const int i = i0 + u * kTThreads;
        if (i >= nvec) break;
        float x[E::PV];
        E::unpack(w[u], x);
#pragma unroll
        for (int k = 0; k < E::PV; ++k) f(i * E::PV + k, x[k]);
      }
    }
  } else {
    for (int v = threadIdx.x; v < V; v += kTThreads) f(v, E::to_f32(__ldcg(row + v)));
  }
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Block sum of a 64-bit value, returned to every thread.
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, TruncSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  __syncthreads();  // earlier readers of wtot / bc are done
  if (lane == 0) sm.wtot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = lane < kTWarps ? sm.wtot[lane] : 0ull;
    t = warp_sum_u64(t);
    if (lane == 0) sm.bc = t;
  }
  __syncthreads();
  return sm.bc;
}

// Block inclusive scan of a 64-bit value in thread order; *total gets the sum.
__device__ __forceinline__ unsigned long long block_incl_scan_u64(unsigned long long v, TruncSmem& sm,
                                                                  unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = warp_incl_scan_u64(v, lane);
  __syncthreads();
  if (lane == 31) sm.wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long t = lane < kTWarps ? sm.wtot[lane] : 0ull;
    const unsigned long long ti = warp_incl_scan_u64(t, lane);
    if (lane < kTWarps) sm.wtot[lane] = ti - t;  // exclusive offsets of the warps
    if (lane == kTWarps - 1) sm.bc = ti;
  }
  __syncthreads();
  *total = sm.bc;
  return incl + sm.wtot[warp];
}

// One radix pass: sm.hist[d] = total weight of the eligible elements whose key
// matches `prefix` under `pmask` and whose digit (key >> shift) & 255 is d.
// kCount: every weight is 1.
template <class E, bool kCount, class Elig, class Wt>
__device__ void hist_pass(const typename E::Raw* row, int V, bool aligned, uint32_t prefix, uint32_t pmask,
                          int shift, Elig elig, Wt wt, TruncSmem& sm) {
  constexpr int KB = 8 * E::ES;
  constexpr int PV = E::PV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // readers of the previous pass's histograms are done
  Limbs lb(sm, warp);
  lb.zero(lane);
  const int nitem = aligned ? V / PV : V;
  const int per = aligned ? PV : 1;
  for (int base = warp * 32; base < nitem; base += kTThreads * kTUnroll) {
    uint4 raw[kTUnroll];
#pragma unroll
    for (int u = 0; u < kTUnroll; ++u) {
      const int i = base + u * kTThreads + lane;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < nitem) {
        if (aligned)
          raw[u] = __ldcg(reinterpret_cast<const uint4*>(row) + i);
        else
          raw[u].x = (uint32_t)__ldcg(row + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kTUnroll; ++u) {
      const int i = base + u * kTThreads + lane;
      if (base + u * kTThreads >= nitem) break;  // warp-uniform
      const bool valid = i < nitem;
      bool added = false;
      float x[PV];
#pragma unroll
      for (int j = 0; j < PV; ++j) x[j] = -INFINITY;
      if (valid) {
        if (aligned)
          E::unpack(raw[u], x);
        else
          x[0] = E::to_f32((typename E::Raw)raw[u].x);
      }
#pragma unroll
      for (int j = 0; j < PV; ++j) {
        if (j >= per) break;  // warp-uniform
        const int v = aligned ? i * PV + j : i;
        const uint32_t key = order_key<KB>(x[j]);
        const bool on = valid && (key & pmask) == prefix && elig(v, key);
        const unsigned long long w = on ? (kCount ? 1ull : wt(x[j])) : 0ull;
        const uint32_t digit = (key >> shift) & 255u;
        if (w) lb.add(digit, w);  // the warp's own counters: conflicts only within the warp
        added |= (w != 0ull);
      }
      lb.step(lane, added);
    }
  }
  lb.flush(lane);
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += kTThreads) {
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < kTWarps; ++w) t += sm.ph[w][b];
    sm.hist[b] = t;
  }
  __syncthreads();
}

// Radix select, descending: the key thr of the element at which the running
// weight, in ranking order over the eligible elements, first reaches `need`
// (need >= 1).  *above gets the weight of eligible elements with larger keys
// (< need); the rest, need - *above, is still needed inside the key thr.
// Returns false if the eligible weight is below need.  first >= 0: the first
// digit is already known to be `first`, with weight `above0` above it.
template <class E, bool kCount, class Elig, class Wt>
__device__ bool radix_select(const typename E::Raw* row, int V, bool aligned, unsigned long long need, Elig elig,
                             Wt wt, TruncSmem& sm, uint32_t* thr, unsigned long long* above, int first = -1,
                             unsigned long long above0 = 0) {
  constexpr int KB = 8 * E::ES;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long abv = 0;
  int shift = KB - 8;
  if (first >= 0) {
    prefix = (uint32_t)first << shift;
    pmask = 0xFFu << shift;
    abv = above0;
    shift -= 8;
  }
  for (; shift >= 0; shift -= 8) {
    hist_pass<E, kCount>(row, V, aligned, prefix, pmask, shift, elig, wt, sm);
    if (warp == 0) {
      // lane l scans bins 255 - 8l down to 248 - 8l: lanes in descending key order
      unsigned long long c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.hist[255 - 8 * lane - j];
        tot += c[j];
      }
      const unsigned long long rem = need - abv;
      const unsigned long long incl = warp_incl_scan_u64(tot, lane);
      const unsigned long long excl = incl - tot;
      const bool mine = excl < rem && rem <= incl;
      if (mine) {
        unsigned long long run = excl;
        int b = 255 - 8 * lane - 7;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= rem) {
            b = 255 - 8 * lane - j;
            break;
          }
          run += c[j];
        }
        sm.bin = b;
        sm.bc = run;
      }
      if (__ballot_sync(kFull, mine) == 0u && lane == 0) sm.bin = -1;
    }
    __syncthreads();
    const int b = sm.bin;
    const unsigned long long run = sm.bc;
    if (b < 0) return false;
    abv += run;
    prefix |= (uint32_t)b << shift;
    pmask |= 0xFFu << shift;
  }
  *thr = prefix;
  *above = abv;
  return true;
}

// Index of the need-th (1-based) eligible element with key thr, in index
// order; V if there are fewer.
template <class E, class Elig>
__device__ int tie_index(const typename E::Raw* row, int V, bool aligned, uint32_t thr, unsigned long long need,
                         Elig elig, TruncSmem& sm) {
  constexpr int KB = 8 * E::ES;
  constexpr int PV = E::PV;
  const int per = aligned ? PV : 1;
  const int tile = kTThreads * per;
  unsigned long long running = 0;
  for (int base = 0; base < V; base += tile) {
    const int v0 = base + threadIdx.x * per;
    float x[PV];
#pragma unroll
    for (int j = 0; j < PV; ++j) x[j] = -INFINITY;
    if (aligned) {
      if (v0 < V) E::unpack(__ldcg(reinterpret_cast<const uint4*>(row + v0)), x);
    } else if (v0 < V) {
      x[0] = E::to_f32(__ldcg(row + v0));
    }
    unsigned long long c = 0;
#pragma unroll
    for (int j = 0; j < PV; ++j)
      if (j < per && v0 + j < V) {
        const uint32_t key = order_key<KB>(x[j]);
        if (key == thr && elig(v0 + j, key)) ++c;
      }
    unsigned long long total;
    const unsigned long long incl = block_incl_scan_u64(c, sm, &total);
    if (running + total >= need) {
      const unsigned long long before = running + incl - c;
      if (c > 0 && before < need && running + incl >= need) {
        unsigned long long k = need - before;
#pragma unroll
        for (int j = 0; j < PV; ++j)
          if (j < per && v0 + j < V) {
            const uint32_t key = order_key<KB>(x[j]);
            if (key == thr && elig(v0 + j, key) && --k == 0) sm.tie = v0 + j;
          }
      }
      __syncthreads();
      const int t = sm.tie;
      __syncthreads();
      return t;
    }
    running += total;
  }
  return V;
}

// Warp w walks its own contiguous chunk of the row, 32 consecutive vectors
// (elements, for unaligned rows) per step, kTUnroll steps of loads in flight;
// f(i, valid, x) runs warp-converged for every lane: vector i (element i if
// unaligned), x its PV values (-inf past the end; x[0] only if unaligned).
template <class E, class F>
__device__ __forceinline__ void chunk_walk(const typename E::Raw* row, int V, bool aligned, F&& f) {
  constexpr int PV = E::PV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nitem = aligned ? V / PV : V;
  const int cw = (nitem + kTWarps - 1) / kTWarps;
  const int lo = min(warp * cw, nitem), hi = min(lo + cw, nitem);
  for (int base = lo; base < hi; base += 32 * kTUnroll) {
    uint4 raw[kTUnroll];
#pragma unroll
    for (int u = 0; u < kTUnroll; ++u) {
      const int i = base + u * 32 + lane;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < hi) {
        if (aligned)
          raw[u] = __ldcg(reinterpret_cast<const uint4*>(row) + i);
        else
          raw[u].x = (uint32_t)__ldcg(row + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kTUnroll; ++u) {
      if (base + u * 32 >= hi) break;  // warp-uniform
      const int i = base + u * 32 + lane;
      const bool valid = i < hi;
      float x[PV];
#pragma unroll
      for (int j = 0; j < PV; ++j) x[j] = -INFINITY;
      if (valid) {
        if (aligned)
          E::unpack(raw[u], x);
        else
          x[0] = E::to_f32((typename E::Raw)raw[u].x);
      }
      f(i, valid, x);
    }
  }
}

// Ordered compaction: every element (index v, value x) with pick(v, x) goes
// to the candidate list in index order.  pc[w][digit] must hold, for warp
// w's chunk, the number of picked elements (they all have first digit d1).
template <class E, class Pick>
__device__ int compact(const typename E::Raw* row, int V, bool aligned, uint32_t d1, Pick pick, TruncSmem& sm) {
  constexpr int PV = E::PV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = aligned ? PV : 1;
  int off = 0, total = 0;
  for (int w = 0; w < kTWarps; ++w) {
    const int c = (int)sm.pc[w][d1];
    if (w < warp) off += c;
    total += c;
  }
  chunk_walk<E>(row, V, aligned, [&](int i, bool valid, const float (&x)[PV]) {
    unsigned m = 0;  // picked elements of this lane, bit j
#pragma unroll
    for (int j = 0; j < PV; ++j)
      if (j < per && valid && pick(aligned ? i * PV + j : i, x[j])) m |= 1u << j;
    const int c = __popc(m);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    int at = off + incl - c;
#pragma unroll
    for (int j = 0; j < PV; ++j)
      if ((m >> j) & 1u) {
        sm.cand_idx[at] = aligned ? i * PV + j : i;
        sm.cand_x[at] = x[j];
        ++at;
      }
    off += __shfl_sync(kFull, incl, 31);
  });
  __syncthreads();
  return total;
}

// Radix select over the candidate list for the digits below the first:
// prefix holds the first digit; need is the weight still needed inside it.
// Returns the full threshold key; *above gets the weight of candidates with
// larger keys.
template <class E, bool kCount, class Wt>
__device__ uint32_t list_select(int n, uint32_t prefix, unsigned long long need, Wt wt, TruncSmem& sm,
                                unsigned long long* above) {
  constexpr int KB = 8 * E::ES;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t pmask = 0xFFu << (KB - 8);
  unsigned long long abv = 0;
  for (int shift = KB - 16; shift >= 0; shift -= 8) {
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += kTThreads) sm.hist[i] = 0ull;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kTThreads) {
      const float x = sm.cand_x[i];
      const uint32_t key = order_key<KB>(x);
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], kCount ? 1ull : wt(x));
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.hist[255 - 8 * lane - j];
        tot += c[j];
      }
      const unsigned long long rem = need - abv;
      const unsigned long long incl = warp_incl_scan_u64(tot, lane);
      const unsigned long long excl = incl - tot;
      const bool mine = excl < rem && rem <= incl;
      if (mine) {
        unsigned long long run = excl;
        int b = 255 - 8 * lane - 7;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= rem) {
            b = 255 - 8 * lane - j;
            break;
          }
          run += c[j];
        }
        sm.bin = b;
        sm.bc = run;
      }
      if (__ballot_sync(kFull, mine) == 0u && lane == 0) {  // cannot happen for consistent weights
        sm.bin = 0;
        sm.bc = 0;
      }
    }
    __syncthreads();
    abv += sm.bc;
    prefix |= (uint32_t)sm.bin << shift;
    pmask |= 0xFFu << shift;
  }
  *above = abv;
  return prefix;
}

// Index of the need-th candidate (list order = index order) with key thr;
// V if there are fewer.
template <int KB>
__device__ int list_tie(int n, uint32_t thr, unsigned long long need, int V, TruncSmem& sm) {
  const int per = (n + kTThreads - 1) / kTThreads;
  const int lo = min((int)threadIdx.x * per, n), hi = min(lo + per, n);
  unsigned long long c = 0;
  for (int i = lo; i < hi; ++i) c += order_key<KB>(sm.cand_x[i]) == thr;
  unsigned long long total;
  const unsigned long long incl = block_incl_scan_u64(c, sm, &total);
  if (threadIdx.x == 0) sm.tie = V;
  __syncthreads();
  const unsigned long long before = incl - c;
  if (c > 0 && before < need && incl >= need) {
    unsigned long long k = need - before;
    for (int i = lo; i < hi; ++i)
      if (order_key<KB>(sm.cand_x[i]) == thr && --k == 0) {
        sm.tie = sm.cand_idx[i];
        break;
      }
  }
  __syncthreads();
  const int t = sm.tie;
  __syncthreads();
  return t;
}

// Reduces the per-warp first-digit histograms (counts pc or weights ph) into
// sm.hist; returns the total weight.
template <bool kFromCounts>
__device__ unsigned long long reduce_first(TruncSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += kTThreads) {
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < kTWarps; ++w) t += kFromCounts ? (unsigned long long)sm.pc[w][b] : sm.ph[w][b];
    sm.hist[b] = t;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) t += sm.hist[8 * lane + j];
    t = warp_sum_u64(t);
    if (lane == 0) sm.bc = t;
  }
  __syncthreads();
  const unsigned long long total = sm.bc;
  __syncthreads();
  return total;
}

// The first-digit bin, scanning sm.hist from the top, at which the running
// weight reaches need (>= 1); *above gets the weight of the bins above it.
// -1 if the total is below need.
__device__ int crossing_bin(unsigned long long need, TruncSmem& sm, unsigned long long* above) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == 0) {
    unsigned long long c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = sm.hist[255 - 8 * lane - j];
      tot += c[j];
    }
    const unsigned long long incl = warp_incl_scan_u64(tot, lane);
    const unsigned long long excl = incl - tot;
    const bool mine = excl < need && need <= incl;
    if (mine) {
      unsigned long long run = excl;
      int b = 255 - 8 * lane - 7;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + c[j] >= need) {
          b = 255 - 8 * lane - j;
          break;
        }
        run += c[j];
      }
      sm.bin = b;
      sm.bc = run;
    }
    if (__ballot_sync(kFull, mine) == 0u && lane == 0) sm.bin = -1;
  }
  __syncthreads();
  *above = sm.bc;
  const int bin = sm.bin;
  __syncthreads();
  return bin;
}

// ---- bf16 value histogram: both cuts from one counting pass ---------------------
// A bf16 row holds few distinct values, so the pass that finds the maximum
// also counts every value: one bin per bf16 value for 2^-24 <= |x| < 2^16
// (both signs, full 7-bit mantissa), plus three merged bins: x <= -2^16,
// |x| < 2^-24 (zeros included) and x >= 2^16.  Bins ascend with the value,
// so the ranking order is the bins' order, top down.  Every element of a
// one-value bin has the same fixed-point mass, so a bin's mass is count x
// mass, the same integer the per-element sums give.  The merged bins only
// take part while that stays exact: the small-magnitude bin when |M| >= 2
// (every x there then gives fl(x - M) = -M), the large negative bin when
// its masses are provably zero, and no cut may fall in a merged bin.
// Otherwise the row takes the radix path.
constexpr int kFLo = 103;                        // biased exponent of 2^-24
constexpr int kFHi = 142;                        // biased exponent of 2^15
constexpr int kNF = (kFHi - kFLo + 1) * 128;     // one-value bins per sign
constexpr int kNB = 2 * kNF + 3;                 // with the three merged bins
constexpr int kBinTiny = kNF + 1;                // |x| < 2^-24
constexpr int kTieSteps = 128;                   // per-warp step counts a tie walk keeps
static_assert(kNB * sizeof(uint32_t) <= sizeof(unsigned long long) * kTWarps * 256 + sizeof(uint32_t) * kTWarps * 256,
              "the value histogram fits in the radix histograms' storage");
static_assert(kTWarps * kTieSteps * sizeof(uint16_t) <= sizeof(int) * kTCap, "step counts fit in the candidate storage");

__device__ __forceinline__ uint32_t* value_hist(TruncSmem& sm) { return reinterpret_cast<uint32_t*>(&sm.ph[0][0]); }

// Bin of a bf16 value held in a float.
__device__ __forceinline__ int value_bin(float x) {
  const uint32_t u = __float_as_uint(x) >> 16;
  const uint32_t mag = u & 0x7FFFu;
  if (mag < (uint32_t)(kFLo << 7)) return kBinTiny;
  if (mag > (uint32_t)((kFHi << 7) | 0x7F)) return (u & 0x8000u) ? 0 : kNB - 1;
  const int f = (int)mag - (kFLo << 7);
  return (u & 0x8000u) ? kNF - f : kNF + 2 + f;
}

// The value of a one-value bin.
__device__ __forceinline__ float bin_value(int b) {
  const bool neg = b <= kNF;
  const int f = neg ? kNF - b : b - (kNF + 2);
  return __uint_as_float((((uint32_t)((kFLo << 7) + f)) | (neg ? 0x8000u : 0u)) << 16);
}

// Top-down crossing over the value histogram: thread t owns kNB / kTThreads
// consecutive bins, walked downward, and thread order is descending bin
// order.  wt(b) is bin b's weight; need_of(total) the weight to reach.
// Returns the bin where the running weight first reaches it (-1: never);
// *above gets the weight of the bins above, *need the target.
template <class Wt, class Need>
__device__ int value_crossing(Wt wt, Need need_of, TruncSmem& sm, unsigned long long* above,
                              unsigned long long* need) {
  constexpr int C = (kNB + kTThreads - 1) / kTThreads;
  const int hi = kNB - (int)threadIdx.x * C;  // exclusive
  const int lo = max(hi - C, 0);
  unsigned long long t = 0;
  for (int b = hi - 1; b >= lo; --b) t += wt(b);
  unsigned long long total;
  const unsigned long long incl = block_incl_scan_u64(t, sm, &total);
  const unsigned long long nd = need_of(total);
  if (threadIdx.x == 0) sm.xbin = -1;
  __syncthreads();
  const unsigned long long excl = incl - t;
  if (excl < nd && nd <= incl) {
    unsigned long long run = excl;
    for (int b = hi - 1; b >= lo; --b) {
      const unsigned long long w = wt(b);
      if (run + w >= nd) {
        sm.xbin = b;
        sm.xabove = run;
        break;
      }
      run += w;
    }
  }
  __syncthreads();
  const int b = sm.xbin;
  *above = b >= 0 ? sm.xabove : 0ull;
  *need = nd;
  __syncthreads();  // xbin / xabove reuse
  return b;
}

// Index of the need-th (1-based) eligible element of key thr, in index order;
// V if there are fewer.  Every warp counts the tied elements of its chunk,
// step by step (the chunk_walk order); the warp holding the need-th one
// reloads only the step that holds it.
template <class E, class Elig>
__device__ int tie_walk(const typename E::Raw* row, int V, bool aligned, uint32_t thr, unsigned long long need,
                        Elig elig, TruncSmem& sm) {
  constexpr int KB = 8 * E::ES;
  constexpr int PV = E::PV;
  constexpr int kStep = 32 * kTUnroll;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = aligned ? PV : 1;
  const int nitem = aligned ? V / PV : V;
  const int cw = (nitem + kTWarps - 1) / kTWarps;
  const int lo = min(warp * cw, nitem), hi = min(lo + cw, nitem);
  uint16_t* ws = reinterpret_cast<uint16_t*>(sm.cand_idx) + warp * kTieSteps;
  auto load = [&](int i, float (&x)[PV]) {
#pragma unroll
    for (int j = 0; j < PV; ++j) x[j] = -INFINITY;
    if (i < hi) {
      if (aligned)
        E::unpack(__ldcg(reinterpret_cast<const uint4*>(row) + i), x);
      else
        x[0] = E::to_f32(__ldcg(row + i));
    }
  };
  auto tied = [&](int i, const float (&x)[PV]) {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < PV; ++j) {
      if (j >= per) break;
      const uint32_t key = order_key<KB>(x[j]);
      if (i < hi && key == thr && elig(aligned ? i * PV + j : i, key)) m |= 1u << j;
    }
    return m;
  };
  uint32_t c = 0;
  int step = 0;
  for (int base = lo; base < hi; base += kStep, ++step) {
    float x[kTUnroll][PV];
#pragma unroll
    for (int u = 0; u < kTUnroll; ++u) load(base + u * 32 + lane, x[u]);
    uint32_t cs = 0;
#pragma unroll
    for (int u = 0; u < kTUnroll; ++u) cs += __popc(tied(base + u * 32 + lane, x[u]));
    cs = __reduce_add_sync(kFull, cs);
    if (lane == 0 && step < kTieSteps) ws[step] = (uint16_t)cs;
    c += cs;
  }
  if (lane == 0) sm.wc[warp] = c;
  if (threadIdx.x == 0) sm.tie = V;
  __syncthreads();
  unsigned long long run = 0;
  int cwarp = -1;
  for (int w = 0; w < kTWarps; ++w) {
    if (run + sm.wc[w] >= need) {
      cwarp = w;
      break;
    }
    run += sm.wc[w];
  }
  if (warp == cwarp) {
    unsigned long long k = need - run;  // rank inside this warp's chunk
    const int nsteps = (hi - lo + kStep - 1) / kStep;
    int s0 = 0;
    if (nsteps <= kTieSteps) {  // skip whole steps by their recorded counts
      while (s0 < nsteps && (unsigned long long)ws[s0] < k) {
        k -= ws[s0];
        ++s0;
      }
    }
    for (int base = lo + s0 * kStep; base < hi && k > 0; base += 32) {
      float x[PV];
      const int i = base + lane;
      load(i, x);
      const uint32_t m = tied(i, x);
      const int cc = __popc(m);
      int incl = cc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned long long tot = (unsigned long long)__shfl_sync(kFull, incl, 31);
      if (tot >= k) {
        const unsigned long long ex = (unsigned long long)(incl - cc);
        if (ex < k && k <= (unsigned long long)incl) {
          uint32_t mm = m;
          for (unsigned long long r = k - ex; r > 1; --r) mm &= mm - 1u;
          const int j = __ffs(mm) - 1;
          sm.tie = aligned ? i * PV + j : i;
        }
        break;
      }
      k -= tot;
    }
  }
  __syncthreads();
  const int t = sm.tie;
  __syncthreads();  // tie / wc / step counts reuse
  return t;
}

template <class E>
__global__ void __launch_bounds__(kTThreads, 2) truncate_kernel(const __grid_constant__ TruncParams P) {
  extern __shared__ __align__(16) unsigned char tsm_raw[];
  TruncSmem& sm = *reinterpret_cast<TruncSmem*>(tsm_raw);
  using Raw = typename E::Raw;
  constexpr int KB = 8 * E::ES;
  constexpr int PV = E::PV;
  const int V = P.V;
  const bool al = P.aligned != 0;
  const int per = al ? PV : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool do_k = P.top_k > 0 && P.top_k < V;
  const bool do_p = P.top_p < 1.0f;
  const float s = P.s;
  for (int row = blockIdx.x; row < P.rows; row += gridDim.x) {
    const Raw* zin = reinterpret_cast<const Raw*>(P.in) + (long long)row * V;
    Raw* zout = reinterpret_cast<Raw*>(P.out) + (long long)row * V;

    // ---- pass 1: maximum and NaN check (bf16: and the value histogram) ----
    constexpr bool kHist = KB == 16;
    const bool vh = kHist && (do_k || do_p);
    __syncthreads();  // the previous row is done with the shared state
    if (vh)
      for (int b = threadIdx.x; b < kNB; b += kTThreads) value_hist(sm)[b] = 0u;
    __syncthreads();
    float mx = -INFINITY;
    int nan = 0;
    chunk_walk<E>(zin, V, al, [&](int, bool valid, const float (&x)[PV]) {
#pragma unroll
      for (int j = 0; j < PV; ++j) {
        if (j >= per) break;
        mx = fmaxf(mx, x[j]);
        nan |= (x[j] != x[j]);
        if (kHist && vh && valid) atomicAdd(value_hist(sm) + value_bin(x[j]), 1u);
      }
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    nan = __any_sync(kFull, nan);
    if (lane == 0) {
      sm.wmax[warp] = mx;
      sm.wnan[warp] = nan;
    }
    __syncthreads();
    float M = -INFINITY;
    int bad = 0;
    for (int w = 0; w < kTWarps; ++w) {
      M = fmaxf(M, sm.wmax[w]);
      bad |= sm.wnan[w];
    }
    bad |= !(M > -INFINITY && M < INFINITY);

    // ---- top-k: key thr1, ties kept up to index tie1 ----
    uint32_t thr1 = 0;
    int tie1 = V;
    bool ok = !bad;
    bool done_k = !do_k;
    // ---- top-p over the top-k set: key thr2, ties kept up to index tie2 ----
    uint32_t thr2 = 0;
    int tie2 = V;
    bool done_p = !do_p;

    // ---- bf16: both cuts from the value histogram ----
    // The last active cut leaves one key thrF of which only the first nF
    // tied elements (index order) stay: the write pass keeps every element
    // of that key and marks them in a bitmap, then drops the ones after the
    // nF-th.  Rows too long for the bitmap find the index with a tie walk.
    uint32_t thrF = 0;
    unsigned long long nF = 0;
    bool fix = false;
    if constexpr (kHist) if (vh && ok) {
      const uint32_t* H = value_hist(sm);
      bool fast = H[kNB - 1] == 0u;  // no value at or above 2^16
      int b1 = -1;                   // the top-k cut's bin; bins below it are dropped
      unsigned long long keep1 = 0;  // kept elements of bin b1
      int bF = -1;
      if (fast && do_k) {
        unsigned long long above = 0, need = 0;
        const int b = value_crossing([&](int bb) { return (unsigned long long)H[bb]; },
                                     [&](unsigned long long) { return (unsigned long long)P.top_k; }, sm, &above,
                                     &need);
        if (b <= 0 || b == kBinTiny) {
          fast = false;  // a cut among merged values
        } else {
          thr1 = order_key<KB>(bin_value(b));
          const unsigned long long rem = need - above, nt = H[b];
          b1 = b;
          keep1 = rem < nt ? rem : nt;
          bF = b;
          thrF = thr1;
          nF = keep1;
        }
      }
      if (fast && do_p) {
        // merged bins with a mass: |x| < 2^-24 needs fl(x - M) = -M; x <= -2^16 needs zero mass
        if (H[kBinTiny] != 0u && !(fabsf(M) >= 2.0f)) fast = false;
        if (H[0] != 0u && !(__fmul_rn(__fsub_rn(-65536.0f, M), s) <= -60.0f)) fast = false;
      }
      if (fast && do_p) {
        auto mass = [&](int bb) -> unsigned long long {
          unsigned long long c = H[bb];
          if (do_k) {
            if (bb < b1) return 0ull;
            if (bb == b1) c = keep1;
          }
          if (c == 0ull || bb == 0) return 0ull;
          return c * fixed_mass(bb == kBinTiny ? 0.0f : bin_value(bb), M, s);
        };
        unsigned long long above = 0, tau = 0;
        const int c = value_crossing(mass,
                                     [&](unsigned long long z) {
                                       const unsigned long long t =
                                           (unsigned long long)ceil((double)P.top_p * (double)z);
                                       return t == 0ull ? 1ull : t;
                                     },
                                     sm, &above, &tau);
        if (c <= 0 || c == kBinTiny) {
          fast = false;
        } else {
          // c >= b1: the top-p cut lies inside the top-k set
          const float xc = bin_value(c);
          thr2 = order_key<KB>(xc);
          // tied tokens share one mass: keep the first ceil(rest / w) of them
          const unsigned long long w = fixed_mass(xc, M, s);
          const unsigned long long rest = tau - above;
          const unsigned long long nk = w ? (rest + w - 1) / w : 1ull;
          const unsigned long long avail = (do_k && c == b1) ? keep1 : (unsigned long long)H[c];
          bF = c;
          thrF = thr2;
          nF = nk < avail ? nk : avail;
        }
      }
      if (fast) {
        done_k = true;
        done_p = true;
        if (nF < (unsigned long long)H[bF]) {
          if ((V + 31) / 32 <= kTCap) {
            fix = true;
          } else {
            const int t = tie_walk<E>(zin, V, al, thrF, nF, [](int, uint32_t) { return true; }, sm);
            if (do_p) tie2 = t;
            else tie1 = t;
          }
        }
      } else {  // the radix path recomputes both cuts
        thr1 = 0;
        tie1 = V;
        thr2 = 0;
        tie2 = V;
        thrF = 0;
        nF = 0;
      }
    }
    if (ok && !done_k && KB == 16) {
      // bf16: per-warp counts of the 256 keys just below the maximum's, one
      // bin per key (bin 255 - d for key kM - d); the top_k-th key usually
      // lies among them, and elements further down cost no atomic
      const uint32_t kM = order_key<KB>(M);
      __syncthreads();
      for (int b = lane; b < 256; b += 32) sm.pc[warp][b] = 0u;
      __syncwarp();
      chunk_walk<E>(zin, V, al, [&](int, bool valid, const float (&x)[PV]) {
#pragma unroll
        for (int j = 0; j < PV; ++j) {
          if (j >= per) break;
          const uint32_t dk = kM - order_key<KB>(x[j]);
          if (valid && dk < 256u) atomicAdd(&sm.pc[warp][255u - dk], 1u);
        }
      });
      const unsigned long long inwin = reduce_first<true>(sm);
      if (inwin >= (unsigned long long)P.top_k) {
        unsigned long long above = 0;
        const int b = crossing_bin((unsigned long long)P.top_k, sm, &above);
        thr1 = kM - (255u - (uint32_t)b);
        const unsigned long long rem = (unsigned long long)P.top_k - above;
        const unsigned long long nt = sm.hist[b];
        if (rem >= nt) {
          tie1 = V;  // every token of the threshold key is kept
        } else if (nt <= (unsigned long long)kTCap) {
          const uint32_t t1 = thr1;
          const int n = compact<E>(zin, V, al, (uint32_t)b, [&](int, float x) { return order_key<KB>(x) == t1; },
                                   sm);
          tie1 = list_tie<KB>(n, thr1, rem, V, sm);
        } else {
          tie1 = tie_index<E>(zin, V, al, thr1, rem, [](int, uint32_t) { return true; }, sm);
        }
        done_k = true;
      }
    }
    if (ok && !done_k) {
      // first-digit counts, then the crossing digit's candidates
      __syncthreads();
      for (int b = lane; b < 256; b += 32) sm.pc[warp][b] = 0u;
      __syncwarp();
      chunk_walk<E>(zin, V, al, [&](int, bool valid, const float (&x)[PV]) {
#pragma unroll
        for (int j = 0; j < PV; ++j) {
          if (j >= per) break;
          const uint32_t d = order_key<KB>(x[j]) >> (KB - 8);
          if (valid) atomicAdd(&sm.pc[warp][d], 1u);  // the warp's own counters
        }
      });
      reduce_first<true>(sm);
      unsigned long long above = 0;
      const int b1 = crossing_bin((unsigned long long)P.top_k, sm, &above);
      const unsigned long long n1 = b1 >= 0 ? sm.hist[b1] : 0ull;
      if (b1 < 0) {
        ok = false;
      } else if (n1 <= (unsigned long long)kTCap) {
        // the candidates of the crossing digit, in index order; the rest of the key on them
        const int n = compact<E>(zin, V, al, (uint32_t)b1,
                                 [&](int, float x) { return (order_key<KB>(x) >> (KB - 8)) == (uint32_t)b1; }, sm);
        unsigned long long above2 = 0;
        thr1 = list_select<E, true>(n, (uint32_t)b1 << (KB - 8), (unsigned long long)P.top_k - above,
                                    [](float) { return 1ull; }, sm, &above2);
        tie1 = list_tie<KB>(n, thr1, (unsigned long long)P.top_k - above - above2, V, sm);
      } else {  // a crowded digit: select its lower digits over the whole row
        ok = radix_select<E, true>(
            zin, V, al, (unsigned long long)P.top_k, [](int, uint32_t) { return true; },
            [](float) { return 1ull; }, sm, &thr1, &above, b1, above);
        if (ok) tie1 = tie_index<E>(zin, V, al, thr1, (unsigned long long)P.top_k - above,
                                    [](int, uint32_t) { return true; }, sm);
      }
    }
    auto kept1 = [&](int v, uint32_t key) { return key > thr1 || (key == thr1 && v <= tie1); };

    if (ok && !done_p) {
      // pass: fixed-point masses and counts of the first digit over the top-k set
      __syncthreads();
      for (int b = lane; b < 256; b += 32) sm.pc[warp][b] = 0u;
      Limbs lb(sm, warp);
      lb.zero(lane);
      chunk_walk<E>(zin, V, al, [&](int i, bool valid, const float (&x)[PV]) {
        bool added = false;
#pragma unroll
        for (int j = 0; j < PV; ++j) {
          if (j >= per) break;
          const uint32_t key = order_key<KB>(x[j]);
          const bool on = valid && kept1(al ? i * PV + j : i, key);
          const uint32_t d = key >> (KB - 8);
          if (on) {
            atomicAdd(&sm.pc[warp][d], 1u);
            const unsigned long long w = fixed_mass(x[j], M, s);
            if (w) {
              lb.add(d, w);
              added = true;
            }
          }
        }
        lb.step(lane, added);
      });
      lb.flush(lane);
      const unsigned long long z = reduce_first<false>(sm);
      unsigned long long tau = (unsigned long long)ceil((double)P.top_p * (double)z);
      if (tau == 0ull) tau = 1ull;
      unsigned long long above = 0;
      const int c1 = crossing_bin(tau, sm, &above);
      unsigned long long n2 = 0;
      if (c1 >= 0)
        for (int w = 0; w < kTWarps; ++w) n2 += sm.pc[w][c1];
      if (c1 < 0) {
        ok = false;
      } else if (n2 <= (unsigned long long)kTCap) {
        const int n = compact<E>(zin, V, al, (uint32_t)c1,
                                 [&](int v, float x) {
                                   const uint32_t key = order_key<KB>(x);
                                   return (key >> (KB - 8)) == (uint32_t)c1 && kept1(v, key);
                                 },
                                 sm);
        unsigned long long above2 = 0;
        thr2 = list_select<E, false>(n, (uint32_t)c1 << (KB - 8), tau - above,
                                     [&](float x) { return fixed_mass(x, M, s); }, sm, &above2);
        // tied tokens share one mass: keep the first ceil(rest / w) of them
        const unsigned long long w = fixed_mass(key_value<KB>(thr2), M, s);
        const unsigned long long rest = tau - above - above2;
        const unsigned long long nk = w ? (rest + w - 1) / w : 1ull;
        tie2 = list_tie<KB>(n, thr2, nk, V, sm);
      } else {  // a crowded digit: select its lower digits over the whole row
        ok = radix_select<E, false>(zin, V, al, tau, kept1, [&](float x) { return fixed_mass(x, M, s); }, sm,
                                    &thr2, &above, c1, above);
        if (ok) {
          const unsigned long long w = fixed_mass(key_value<KB>(thr2), M, s);
          const unsigned long long rest = tau - above;
          const unsigned long long nk = w ? (rest + w - 1) / w : 1ull;
          tie2 = tie_index<E>(zin, V, al, thr2, nk, kept1, sm);
        }
      }
    }
    // a row with NaN or infinite logits (or none finite) is copied unchanged
    if ((bad || !ok) && threadIdx.x == 0 && P.status) atomicOr(P.status, kBadLogits);
    const bool cut = ok && (do_k || do_p);
    uint32_t* tie_bits = reinterpret_cast<uint32_t*>(sm.cand_idx);  // one bit per index of the row
    auto keep = [&](int v, float x) {
      if (!cut) return true;
      const uint32_t key = order_key<KB>(x);
      const bool k = kept1(v, key) && (!do_p || key > thr2 || (key == thr2 && v <= tie2));
      if (fix && k && key == thrF) atomicOr(tie_bits + (v >> 5), 1u << (v & 31));
      return k;
    };
    if (fix) {
      for (int w = threadIdx.x; w < (V + 31) / 32; w += kTThreads) tie_bits[w] = 0u;
      __syncthreads();
    }

    // ---- write pass ----
    if (al) {
      const uint4* r4 = reinterpret_cast<const uint4*>(zin);
      uint4* o4 = reinterpret_cast<uint4*>(zout);
      const int nvec = V / PV;
      for (int i0 = threadIdx.x; i0 < nvec; i0 += kTThreads * kTUnroll) {
        uint4 raw[kTUnroll];
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
          const int i = i0 + u * kTThreads;
          raw[u] = i < nvec ? __ldcg(r4 + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
          const int i = i0 + u * kTThreads;
          if (i >= nvec) break;
          const uint4 w = raw[u];
          float x[PV];
          E::unpack(w, x);
          uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < PV; ++k) {
            if (keep(i * PV + k, x[k])) continue;
            if constexpr (PV == 8) {  // bf16: element 2j in the low half of word j
              wd[k >> 1] = (k & 1) ? ((wd[k >> 1] & 0x0000FFFFu) | 0xFF800000u) : ((wd[k >> 1] & 0xFFFF0000u) | 0xFF80u);
            } else {
              wd[k] = 0xFF800000u;
            }
          }
          __stcs(o4 + i, make_uint4(wd[0], wd[1], wd[2], wd[3]));
        }
      }
    } else {
      for (int v = threadIdx.x; v < V; v += kTThreads) {
        const Raw r = __ldcg(zin + v);
        zout[v] = keep(v, E::to_f32(r)) ? r : E::kNegInf;
      }
    }
    if (fix) {
      // the nF-th marked index in index order; every later marked element is dropped
      __syncthreads();
      const int nw = (V + 31) / 32;
      const int per_t = (nw + kTThreads - 1) / kTThreads;
      const int w0 = min((int)threadIdx.x * per_t, nw), w1 = min(w0 + per_t, nw);
      unsigned long long c = 0;
      for (int w = w0; w < w1; ++w) c += __popc(tie_bits[w]);
      unsigned long long total;
      const unsigned long long incl = block_incl_scan_u64(c, sm, &total);
      if (threadIdx.x == 0) sm.tie = V;
      __syncthreads();
      const unsigned long long ex = incl - c;
      if (ex < nF && nF <= incl) {
        unsigned long long k = nF - ex;
        for (int w = w0; w < w1; ++w) {
          const uint32_t m = tie_bits[w];
          const unsigned long long pc = (unsigned long long)__popc(m);
          if (pc >= k) {
            uint32_t mm = m;
            for (unsigned long long r = k; r > 1; --r) mm &= mm - 1u;
            sm.tie = w * 32 + __ffs(mm) - 1;
            break;
          }
          k -= pc;
        }
      }
      __syncthreads();
      const int tF = sm.tie;
      for (int w = w0; w < w1; ++w) {
        uint32_t m = tie_bits[w];
        while (m) {
          const int v = w * 32 + __ffs(m) - 1;
          m &= m - 1u;
          if (v > tF) zout[v] = E::kNegInf;
        }
      }
    }
    __syncthreads();  // shared state is reused by the next row
  }
}

}  // namespace ssv
