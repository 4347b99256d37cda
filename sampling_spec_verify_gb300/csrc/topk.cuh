// Top-k (k <= 256) truncation by candidate filtering, with top-p over the
// top-k set when both are asked for: the same transform as truncate.cuh
// ("Speculative Decoding 与 MTP", sections 4 and 23) — rank tokens by logit,
// larger first, ties to the smaller index; keep the first top_k; top-p
// renormalises softmax(z / T) over them and keeps the shortest ranked prefix
// whose mass reaches top_p; dropped logits become -inf.
//
// One CTA per row, two passes:
//  1. every warp walks its own contiguous chunk of the row and keeps, in
//     shared memory and in index order, the elements above its running
//     threshold; when the list grows past a bound the warp selects its k-th
//     largest key (radix select over the list), keeps the top k (ties to the
//     smaller index) and raises the threshold to that key.  After a few
//     hundred elements almost nothing passes the threshold, so the pass costs
//     about one compare per logit.  The CTA then selects the k-th largest key
//     over all warps' lists (each holds its chunk's top k, so the union holds
//     the row's), resolves the tie by index across the warps in chunk order,
//     and, for top-p, sorts the k kept tokens and cuts them by fixed-point
//     mass (units of 2^-44 of the row maximum's, as on the general path);
//  2. the write pass keeps key > thr and (key == thr, index <= tie).
#pragma once

#include <cstdint>

#include "truncate.cuh"

namespace ssv {

constexpr int kKMax = 256;                 // largest top_k on this path
constexpr int kKBuf = 640;                 // list capacity per warp
constexpr int kKTrig = kKBuf - 32 * 8;     // select when a vector step could overflow the list

struct TopkSmem {
  uint32_t key[kTWarps][kKBuf];  // per-warp lists, index order
  int idx[kTWarps][kKBuf];
  uint32_t hist[kTWarps][256];   // per-warp radix histograms
  uint32_t chist[256];           // the CTA's histogram
  int cnt[kTWarps];              // list lengths
  int tiec[kTWarps];             // per-warp counts of the threshold key
  uint32_t skey[kKMax];          // the top-k set, sorted (top-p)
  int sidx[kKMax];
  unsigned long long wtot[kTWarps];
  float wmax[kTWarps];
  int wnan[kTWarps];
  uint32_t thr;
  int tie;
  int cut;
  unsigned long long need;
  uint32_t gkey;  // the largest per-warp threshold key so far (0: none)
};

// Warp radix select over the warp's list (n entries): the key thr of the
// k-th largest (k <= n) and the number of entries with key thr among the top
// k (the rest have larger keys).
template <int KB>
__device__ __forceinline__ uint32_t warp_list_select(const uint32_t* key, int n, int k, uint32_t* hist, int lane,
                                                     int* need_out) {
  uint32_t prefix = 0, pmask = 0;
  int need = k;
#pragma unroll 1
  for (int shift = KB - 8; shift >= 0; shift -= 8) {
#pragma unroll
    for (int b = lane; b < 256; b += 32) hist[b] = 0u;
    __syncwarp();
    for (int e = lane; e < n; e += 32) {
      const uint32_t kk = key[e];
      if ((kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l holds bins 255 - 8l .. 248 - 8l, walked downward
    uint32_t c = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) c += hist[255 - 8 * lane - q];
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(kFull, incl >= (uint32_t)need);
    const int l = __ffs(hit) - 1;  // need <= total, so some lane crosses
    uint32_t run = __shfl_sync(kFull, incl - c, l);
    int d = 0;
    for (int q = 0; q < 8; ++q) {  // every lane walks lane l's bins alike
      const int b = 255 - 8 * l - q;
      const uint32_t h = hist[b];
      if (run + h >= (uint32_t)need) {
        d = b;
        break;
      }
      run += h;
    }
    need -= (int)run;
    prefix |= (uint32_t)d << shift;
    pmask |= 255u << shift;
    __syncwarp();
  }
  *need_out = need;
  return prefix;
}

// Keeps the entries with key > thr and the first `need` with key == thr, in
// list order (in place); returns the new length.
__device__ __forceinline__ int warp_list_keep(uint32_t* key, int* idx, int n, uint32_t thr, int need, int lane) {
  int out = 0, ties = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < n; base += 32) {
    const int e = base + lane;
    const uint32_t kk = e < n ? key[e] : 0u;
    const int ii = e < n ? idx[e] : 0;
    const bool eq = e < n && kk == thr;
    const unsigned te = __ballot_sync(kFull, eq);
    const bool keep = e < n && (kk > thr || (eq && ties + __popc(te & lt) < need));
    const unsigned ke = __ballot_sync(kFull, keep);
    __syncwarp();  // every lane has read its entry
    if (keep) {
      const int p = out + __popc(ke & lt);
      key[p] = kk;
      idx[p] = ii;
    }
    out += __popc(ke);
    ties += __popc(te);
    __syncwarp();
  }
  return out;
}

// Radix select of the k-th largest key over the union of every warp's list
// (warp w's list is wkey[0, n) in its threads; the union holds >= k entries),
// the whole CTA; *need_out gets how many of the union's entries with that key
// are among the top k.
template <int KB>
__device__ uint32_t cta_list_select(TopkSmem& sm, const uint32_t* wkey, int n, int k, unsigned long long* need_out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long need = (unsigned long long)k;
#pragma unroll 1
  for (int shift = KB - 8; shift >= 0; shift -= 8) {
    if (threadIdx.x < 256) sm.chist[threadIdx.x] = 0u;
    __syncthreads();
    for (int e = lane; e < n; e += 32) {
      const uint32_t kk = wkey[e];
      if ((kk & pmask) == prefix) atomicAdd(&sm.chist[(kk >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t c = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) c += sm.chist[255 - 8 * lane - q];
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned hit = __ballot_sync(kFull, (unsigned long long)incl >= need);
      const int l = __ffs(hit) - 1;
      uint32_t run = __shfl_sync(kFull, incl - c, l);
      int d = 0;
      for (int q = 0; q < 8; ++q) {
        const int b = 255 - 8 * l - q;
        const uint32_t h = sm.chist[b];
        if (run + h >= need) {
          d = b;
          break;
        }
        run += h;
      }
      if (lane == 0) {
        sm.thr = prefix | ((uint32_t)d << shift);
        sm.need = need - run;
      }
    }
    __syncthreads();
    prefix = sm.thr;
    pmask |= 255u << shift;
    need = sm.need;
    __syncthreads();
  }
  *need_out = need;
  return prefix;
}

template <class E>
__global__ void __launch_bounds__(kTThreads, 2) topk_kernel(const __grid_constant__ TruncParams P) {
  extern __shared__ __align__(16) unsigned char ksm_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(ksm_raw);
  using Raw = typename E::Raw;
  constexpr int KB = 8 * E::ES;
  constexpr int PV = E::PV;
  const int V = P.V;
  const bool al = P.aligned != 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = P.top_k;  // 0 < k < V, k <= kKMax
  const bool do_p = P.top_p < 1.0f;
  const float s = P.s;
  constexpr uint32_t kNegInfWord = PV == 8 ? 0xFF80FF80u : 0xFF800000u;  // a 32-bit word of -inf values
  uint32_t* wkey = sm.key[warp];
  int* widx = sm.idx[warp];
  for (int row = blockIdx.x; row < P.rows; row += gridDim.x) {
    const Raw* zin = reinterpret_cast<const Raw*>(P.in) + (long long)row * V;
    Raw* zout = reinterpret_cast<Raw*>(P.out) + (long long)row * V;
    __syncthreads();  // the previous row is done with the shared state

    // ---- pass 1: per-warp candidate lists ----
    // A warp's own threshold tau filters strictly (its later elements of that
    // key have larger indices than the ones it keeps); the largest threshold
    // of any warp, gkey, is a lower bound of the row's k-th key, so elements
    // below it are dropped too (but not its ties, which may have smaller
    // indices than the other warp's).
    if (threadIdx.x == 0) sm.gkey = 0u;
    __syncthreads();
    int n = 0;
    float tau = -INFINITY;   // elements above it enter the list
    float taug = -INFINITY;  // elements at or above it may enter the list
    uint32_t gseen = 0u;
    float mx = -INFINITY;
    int nan = 0;
    auto refresh = [&]() {
      const uint32_t g = *reinterpret_cast<const volatile uint32_t*>(&sm.gkey);
      if (g != gseen) {
        gseen = g;
        taug = key_value<KB>(g);
      }
    };
    // appends the elements of mask m (values x, element indices e0 + j * es)
    auto append = [&](uint32_t m, const float (&x)[PV], int e0, int es) {
      const unsigned who = __ballot_sync(kFull, m != 0u);
      int p;
      if (__popc(who) == 1) {  // the usual case once the bounds are tight: one lane
        const int l = __ffs(who) - 1;
        p = n;
        n += __shfl_sync(kFull, __popc(m), l);
      } else {
        const int c = __popc(m);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        p = n + incl - c;
        n += __shfl_sync(kFull, incl, 31);
      }
      while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1u;
        wkey[p] = order_key<KB>(x[j]);
        widx[p] = e0 + j * es;
        mx = fmaxf(mx, x[j]);
        ++p;
      }
      if (n > kKTrig) {
        __syncwarp();
        int need = 0;
        const uint32_t t = warp_list_select<KB>(wkey, n, k, sm.hist[warp], lane, &need);
        n = warp_list_keep(wkey, widx, n, t, need, lane);
        tau = key_value<KB>(t);
        if (lane == 0) atomicMax(&sm.gkey, t);
      }
      refresh();
    };
    if (al) {
      // 16-byte vectors, the warp's contiguous chunk; a vector whose maximum
      // passes neither threshold costs a packed maximum and two compares
      const uint4* r4 = reinterpret_cast<const uint4*>(zin);
      const int nvec = V / PV;
      const int cw = (nvec + kTWarps - 1) / kTWarps;
      const int lo = min(warp * cw, nvec), hi = min(lo + cw, nvec);
      for (int base = lo, step = 0; step == 0 || base < hi; base += 32 * kTUnroll, ++step) {
        uint4 raw[kTUnroll];
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
          const int i = base + u * 32 + lane;
          raw[u] = i < hi ? __ldcg(r4 + i) : make_uint4(kNegInfWord, kNegInfWord, kNegInfWord, kNegInfWord);
        }
        if (step == 0) {
          // a common lower bound before any list: the k-th largest of the
          // 512 lanes' maxima of their first vectors (distinct elements of
          // the row, so at least k of the row's elements reach it)
          float lm = -INFINITY;
#pragma unroll
          for (int u = 0; u < kTUnroll; ++u) lm = fmaxf(lm, E::vmax(raw[u]));
          wkey[lane] = order_key<KB>(lm);
          unsigned long long nd = 0;
          const uint32_t t = cta_list_select<KB>(sm, wkey, 32, k, &nd);
          if (threadIdx.x == 0) sm.gkey = t;
          __syncthreads();
          refresh();
        }
#pragma unroll
        for (int u = 0; u < kTUnroll; ++u) {
          if (base + u * 32 >= hi) break;  // warp-uniform
          const int i = base + u * 32 + lane;
          bool nn;
          const float vm = E::vmax_nan(raw[u], nn);
          nan |= nn;
          const bool maybe = vm > tau && vm >= taug;
          if (__any_sync(kFull, maybe)) {
            float x[PV];
            E::unpack(raw[u], x);
            uint32_t m = 0;
            if (maybe) {
#pragma unroll
              for (int j = 0; j < PV; ++j)
                if (x[j] > tau && x[j] >= taug) m |= 1u << j;
            }
            append(m, x, i * PV, 1);
          }
        }
      }
    } else {
      chunk_walk<E>(zin, V, al, [&](int i, bool valid, const float (&x)[PV]) {
        nan |= (x[0] != x[0]);
        const uint32_t m = (valid && x[0] > tau && x[0] >= taug) ? 1u : 0u;
        if (__any_sync(kFull, m != 0u)) append(m, x, i, 1);
      });
    }
    __syncwarp();
    if (n > k) {
      int need = 0;
      const uint32_t t = warp_list_select<KB>(wkey, n, k, sm.hist[warp], lane, &need);
      n = warp_list_keep(wkey, widx, n, t, need, lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    nan = __any_sync(kFull, nan);
    if (lane == 0) {
      sm.cnt[warp] = n;
      sm.wmax[warp] = mx;
      sm.wnan[warp] = nan;
    }
    __syncthreads();
    float M = -INFINITY;
    int bad = 0, total = 0;
    for (int w = 0; w < kTWarps; ++w) {
      M = fmaxf(M, sm.wmax[w]);
      bad |= sm.wnan[w];
      total += sm.cnt[w];
    }
    bad |= !(M > -INFINITY && M < INFINITY);

    // ---- the CTA's k-th key over all lists, and its tie by index ----
    // With k candidates or more the k-th is selected (exactly k may pass the
    // bounds while finite elements below them are dropped).  With fewer,
    // no bound ever rose above -inf, so every element above -inf is a
    // candidate and among the top k (the rest, -inf, stay -inf whatever the
    // cut): all candidates are kept.
    uint32_t thr = 0;
    int tie = V;
    const int nset = total < k ? total : k;  // the top-k set's elements above -inf
    if (!bad && total >= k) {
      unsigned long long need = 0;
      const uint32_t prefix = cta_list_select<KB>(sm, wkey, n, k, &need);
      thr = prefix;
      // the need-th element of key thr in index order: lists are in index
      // order and the warps' chunks ascend
      int tc = 0;
      for (int e = lane; e < n; e += 32) tc += (wkey[e] == thr) ? 1 : 0;
      tc = __reduce_add_sync(kFull, (unsigned)tc);
      if (lane == 0) sm.tiec[warp] = tc;
      if (threadIdx.x == 0) sm.tie = V;
      __syncthreads();
      unsigned long long before = 0;
      for (int w = 0; w < warp; ++w) before += (unsigned long long)sm.tiec[w];
      if (before < need && need <= before + (unsigned long long)sm.tiec[warp]) {
        unsigned long long r = need - before;  // 1-based rank inside this warp's list
        int seen = 0;
        for (int base = 0; base < n; base += 32) {
          const int e = base + lane;
          const bool eq = e < n && wkey[e] == thr;
          const unsigned te = __ballot_sync(kFull, eq);
          if ((unsigned long long)(seen + __popc(te)) >= r) {
            const unsigned lt = (1u << lane) - 1u;
            if (eq && (unsigned long long)(seen + __popc(te & lt) + 1) == r) sm.tie = widx[e];
            break;
          }
          seen += __popc(te);
        }
      }
      __syncthreads();
      tie = sm.tie;
      __syncthreads();
    }
    if (!bad) {
      // ---- top-p over the kept tokens: sort them, cut by fixed-point mass ----
      if (do_p) {
        // the kept entries, compacted into skey/sidx in warp order
        int kept = 0;
        for (int e = lane; e < n; e += 32) {
          const uint32_t kk = wkey[e];
          kept += (kk > thr || (kk == thr && widx[e] <= tie)) ? 1 : 0;
        }
        kept = (int)__reduce_add_sync(kFull, (unsigned)kept);
        if (lane == 0) sm.tiec[warp] = kept;
        __syncthreads();
        int off = 0;
        for (int w = 0; w < warp; ++w) off += sm.tiec[w];
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < n; base += 32) {
          const int e = base + lane;
          const uint32_t kk = e < n ? wkey[e] : 0u;
          const int ii = e < n ? widx[e] : 0;
          const bool keep = e < n && (kk > thr || (kk == thr && ii <= tie));
          const unsigned ke = __ballot_sync(kFull, keep);
          if (keep) {
            sm.skey[off + __popc(ke & lt)] = kk;
            sm.sidx[off + __popc(ke & lt)] = ii;
          }
          off += __popc(ke);
        }
        __syncthreads();
        // bitonic sort of the nset entries (padded to a power of two) by (key desc, index asc)
        int w2 = 1;
        while (w2 < nset) w2 <<= 1;
        for (int i = nset + (int)threadIdx.x; i < w2; i += kTThreads) {
          sm.skey[i] = 0u;
          sm.sidx[i] = 0x7FFFFFFF;
        }
        __syncthreads();
        for (int kb = 2; kb <= w2; kb <<= 1) {
          for (int j = kb >> 1; j > 0; j >>= 1) {
            const int t = threadIdx.x;
            if (t < (w2 >> 1)) {
              const int i = 2 * t - (t & (j - 1));
              const int q = i + j;
              const bool up = (i & kb) == 0;
              const uint32_t ka = sm.skey[i], kb2 = sm.skey[q];
              const int ia = sm.sidx[i], ib = sm.sidx[q];
              const bool b_first = kb2 > ka || (kb2 == ka && ib < ia);
              const bool a_first = ka > kb2 || (ka == kb2 && ia < ib);
              if (up ? b_first : a_first) {
                sm.skey[i] = kb2;
                sm.skey[q] = ka;
                sm.sidx[i] = ib;
                sm.sidx[q] = ia;
              }
            }
            __syncthreads();
          }
        }
        // masses in ranking order; the first place whose running mass reaches tau
        const int t = threadIdx.x;
        const unsigned long long wm = t < nset ? fixed_mass(key_value<KB>(sm.skey[t]), M, s) : 0ull;
        unsigned long long z = 0;
        unsigned long long incl = warp_incl_scan_u64(wm, lane);
        if (lane == 31) sm.wtot[warp] = incl;
        __syncthreads();
        unsigned long long woff = 0;
        for (int w = 0; w < kTWarps; ++w) {
          if (w < warp) woff += sm.wtot[w];
          z += sm.wtot[w];
        }
        incl += woff;
        unsigned long long tp = (unsigned long long)ceil((double)P.top_p * (double)z);
        if (tp == 0ull) tp = 1ull;
        if (t == 0) sm.cut = nset - 1;
        __syncthreads();
        if (t < nset && incl >= tp && incl - wm < tp) sm.cut = t;
        __syncthreads();
        thr = sm.skey[sm.cut];
        tie = sm.sidx[sm.cut];
        __syncthreads();
      }
    }
    // a row with NaN or infinite logits (or none finite) is copied unchanged
    if (bad && threadIdx.x == 0 && P.status) atomicOr(P.status, kBadLogits);
    const bool cut = !bad && (total >= k || do_p);
    const float thr_f = key_value<KB>(thr);

    // ---- pass 2: write ----
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
          if (cut && E::vmax(w) < thr_f) {  // the whole vector is dropped
            __stcs(o4 + i, make_uint4(kNegInfWord, kNegInfWord, kNegInfWord, kNegInfWord));
            continue;
          }
          float x[PV];
          E::unpack(w, x);
          uint32_t wd[4] = {w.x, w.y, w.z, w.w};
          if (cut) {
#pragma unroll
            for (int j = 0; j < PV; ++j) {
              if (x[j] > thr_f || (x[j] == thr_f && i * PV + j <= tie)) continue;
              if constexpr (PV == 8) {  // bf16: element 2q in the low half of word q
                wd[j >> 1] = (j & 1) ? ((wd[j >> 1] & 0x0000FFFFu) | 0xFF800000u)
                                     : ((wd[j >> 1] & 0xFFFF0000u) | 0xFF80u);
              } else {
                wd[j] = 0xFF800000u;
              }
            }
          }
          __stcs(o4 + i, make_uint4(wd[0], wd[1], wd[2], wd[3]));
        }
      }
    } else {
      for (int v = threadIdx.x; v < V; v += kTThreads) {
        const Raw r = __ldcg(zin + v);
        const float x = E::to_f32(r);
        zout[v] = (!cut || x > thr_f || (x == thr_f && v <= tie)) ? r : E::kNegInf;
      }
    }
  }
}

}  // namespace ssv
