// Vocabulary sweep kernels for sm_103a.
//
// One thread-block cluster of S CTAs owns one (batch row b, position k) unit.
// CTA r of the cluster holds the slice [r*L, min((r+1)*L, V)) of the target
// row (and of the draft row) in shared memory, loaded ONCE from HBM by 1-D
// bulk copies (one per warp segment, completing on a per-warp mbarrier).
// Every later pass reads shared memory only:
//
//   pass A  max of each row                  -> DSMEM exchange 1
//   pass B  sum of 2^((z - M) s), s = log2e/T -> DSMEM exchange 2
//   pass C  overlap sum_v min(p, q) (one exp per element through
//           min(log p, log q)), or, at a rejected / bonus position, the
//           residual max(0, p - q) (or p) with per-round warp scans
//                                            -> DSMEM exchange 3
//   search  the CTA / warp / lane / element holding u' * total mass
//                                            -> DSMEM exchange 4
//
// Rank 0 then publishes a per-unit record in the workspace and bumps a
// per-row arrival counter; the CTA that arrives last for a row runs the
// prefix-order decision over the row's K+1 records (first rejection, tokens,
// overlap) with one warp and re-zeroes the counter.
//
// Data in shared memory is laid out by element index, so thread (warp w,
// lane l) always sees the same vocabulary entries of the target and draft
// rows; a warp only ever reads its own segment of vectors, so no block-wide
// barrier separates the staging from the compute.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace ssv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait

constexpr uint32_t kBadToken = 1u, kBadLogits = 2u, kBadUniform = 4u, kTimeout = 8u,
                   kEmptyResidual = 16u;

enum Mode : int { kVerify = 0, kVerifyGreedy = 1, kOverlap = 2, kOverlapGreedy = 3, kE2E = 4 };

struct VerifyRecord {  // one per (b, k), k = 0..K
  int32_t acc;         // 1 accepted, 0 rejected (draft positions)
  int32_t token;       // correction / bonus / greedy choice; -1 if none
  float alpha;         // overlap of the position
  uint32_t pad;
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
  VerifyRecord* rec;
  E2EStats* stats;
  float* row_loss;
  uint32_t* row_cnt;
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
  __device__ static __forceinline__ float to_f32(Raw r) { return __uint_as_float(uint32_t(r) << 16); }
  // Running maximum kept packed (bf16x2); max needs no rounding.
  struct MaxAcc {
    __nv_bfloat162 m;
    __device__ MaxAcc() { m = __bfloat162bfloat162(__ushort_as_bfloat16(kNegInf)); }
    __device__ __forceinline__ void add(const uint4& w) {
      const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
      const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
      const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
      m = __hmax2(m, __hmax2(__hmax2(a, b), __hmax2(c, d)));
    }
    __device__ __forceinline__ float get() const { return fmaxf(__low2float(m), __high2float(m)); }
  };
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
  __device__ static __forceinline__ float to_f32(Raw r) { return __uint_as_float(r); }
  struct MaxAcc {
    float m = -INFINITY;
    __device__ __forceinline__ void add(const uint4& w) {
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                         fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
    }
    __device__ __forceinline__ float get() const { return m; }
  };
};

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
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v = __fadd_rn(v, t);
  }
  return v;
}

// (value, index) argmax reduction: larger value wins, ties to the smaller index.
__device__ __forceinline__ void arg_better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    arg_better(v, i, v2, i2);
  }
}

// Per-element weights of the residual / bonus draws.  The same function runs
// in the first pass and in the replay of the owning warp, with every rounding
// pinned (__fmul_rn / __fadd_rn / fmaf), so both see bit-identical values.
template <class E, bool kResidual>
__device__ __forceinline__ float draw_weights(const uint4& wt, const uint4& wd, float s, float c1t, float c1d,
                                              float ratio, float (&w)[E::PV], float& min_mass) {
  float t[E::PV];
  E::unpack(wt, t);
  if constexpr (kResidual) {
    float d[E::PV];
    E::unpack(wd, d);
    float m[E::PV];
#pragma unroll
    for (int i = 0; i < E::PV; ++i) {
      const float et = ex2(fmaf(t[i], s, -c1t));
      const float ed = ex2(fmaf(d[i], s, -c1d));
      // rho' = Z_t * max(0, p - q) = max(0, e_t - e_d * Z_t / Z_d)
      const float r = fmaxf(fmaf(-ed, ratio, et), 0.0f);
      w[i] = r;
      m[i] = __fadd_rn(et, -r);  // Z_t * min(p, q)
    }
    min_mass = __fadd_rn(min_mass, tree_sum(m));
  } else {
#pragma unroll
    for (int i = 0; i < E::PV; ++i) w[i] = ex2(fmaf(t[i], s, -c1t));
  }
  return tree_sum(w);
}

// ---- the sweep kernel ----------------------------------------------------------

template <class E, int MODE>
__global__ void __launch_bounds__(kThreads) sweep_kernel(const SweepParams P) {
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t mbar[kWarps];
  __shared__ float red_a[kWarps], red_b[kWarps], red_c[kWarps];
  __shared__ int red_i[kWarps], red_j[kWarps];
  __shared__ float warp_total[kWarps];
  // Cluster mailboxes: written by this CTA, read by peers after a barrier.
  __shared__ float mail_f[8];
  __shared__ int mail_i[4];
  __shared__ uint32_t mail_tok;
  // Block-wide broadcast of values thread 0 computed.
  __shared__ float bc_f[8];
  __shared__ int bc_i[8];

  constexpr int PV = E::PV;
  constexpr bool kGreedy = (MODE == kVerifyGreedy || MODE == kOverlapGreedy);
  constexpr bool kVerifyMode = (MODE == kVerify || MODE == kVerifyGreedy);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = P.S;
  const uint32_t rank = cluster_rank();
  const int unit = blockIdx.x / S;
  const int K = P.K, V = P.V;

  int b, k;
  bool bonus = false;
  if constexpr (kVerifyMode) {
    b = unit / (K + 1);
    k = unit - b * (K + 1);
    bonus = (k == K);
  } else {
    b = unit / K;
    k = unit - b * K;
  }
  const long long trow = (long long)b * P.KT + k;
  const long long drow = (long long)b * K + k;
  bool has_draft = !bonus;
  if constexpr (MODE == kVerifyGreedy) has_draft = !bonus && P.alpha != nullptr;

  const typename E::Raw* tg = reinterpret_cast<const typename E::Raw*>(P.target) + trow * V;
  const typename E::Raw* dg =
      has_draft ? reinterpret_cast<const typename E::Raw*>(P.draft) + drow * V : nullptr;

  // ---- slice and warp segment ----
  const int e0 = (int)rank * P.L;
  const int e1 = min(e0 + P.L, V);
  const int n = max(e1 - e0, 0);
  const int nvec = (n + PV - 1) / PV;
  const int nvec_alloc = P.L / PV;
  const int seg = (nvec + kWarps - 1) / kWarps;
  const int v_lo = min(warp * seg, nvec);
  const int v_hi = min(v_lo + seg, nvec);
  uint4* st = reinterpret_cast<uint4*>(dyn_smem);
  uint4* sd = st + nvec_alloc;

  // Scalars of the decision, fetched early so their latency hides under the
  // staging: drafted token, its two logits, the uniforms.
  int y = -1;
  float u = 0.0f, uf = 0.0f, zt_y = 0.0f, zd_y = 0.0f;
  bool tok_ok = true;
  if constexpr (MODE == kVerify || MODE == kVerifyGreedy) {
    if (!bonus) {
      y = P.draft_tokens[b * K + k];
      tok_ok = (y >= 0 && y < V);
      if constexpr (MODE == kVerify) {
        u = P.u_accept[b * K + k];
        if (tok_ok) {
          zt_y = E::to_f32(tg[y]);
          zd_y = E::to_f32(dg[y]);
        }
      }
    }
    if constexpr (MODE == kVerify) uf = P.u_final[b];
  }

  // ---- staging: one bulk copy per row per warp segment ----
  bool staged = true;
  if (v_hi > v_lo) {
    if (P.aligned) {
      const uint32_t bar = smem_addr(&mbar[warp]);
      const uint32_t bytes = (uint32_t)(v_hi - v_lo) * 16u;
      if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, has_draft ? 2u * bytes : bytes);
        const uint64_t pol = l2_evict_first_policy();
        bulk_load(smem_addr(st + v_lo), tg + e0 + (long long)v_lo * PV, bytes, bar, pol);
        if (has_draft) bulk_load(smem_addr(sd + v_lo), dg + e0 + (long long)v_lo * PV, bytes, bar, pol);
      }
      __syncwarp();
      staged = mbar_wait_bounded(bar, 0, kWaitLimitNs);
    } else {
      // Element-wise staging for rows that do not start on 16-byte
      // boundaries; the tail of the last vector is padded with -inf.
      typename E::Raw* rt = reinterpret_cast<typename E::Raw*>(st);
      typename E::Raw* rd = reinterpret_cast<typename E::Raw*>(sd);
      const int lo = v_lo * PV, hi = v_hi * PV;
      for (int i = lo + lane; i < hi; i += 32) {
        const bool in = (e0 + i) < e1;
        rt[i] = in ? tg[e0 + i] : E::kNegInf;
        if (has_draft) rd[i] = in ? dg[e0 + i] : E::kNegInf;
      }
      __syncwarp();
    }
  }
  if (!staged && lane == 0) atomicOr(P.status, kTimeout);
  const bool work = staged;

  // Reads a value of field `slot` from every CTA of the cluster, in rank order.
  auto gather_f = [&](float* slot, float* out) {
    for (int r = 0; r < S; ++r) out[r] = ld_cluster_f32(map_rank(smem_addr(slot), r));
  };

  uint32_t flags = 0;
  if (tid == 0) mail_tok = 0xFFFFFFFFu;  // peers write it only after exchange 3

  if constexpr (kGreedy) {
    // ================= greedy: argmax of target (and draft) =================
    float bt = -INFINITY, bd = -INFINITY;
    int jt = -1, jd = -1;
    bool nan_seen = false;
    if (work) {
      for (int j = v_lo + lane; j < v_hi; j += 32) {
        float x[PV];
        E::unpack(st[j], x);
        float vm = x[0];
#pragma unroll
        for (int i = 1; i < PV; ++i) vm = fmaxf(vm, x[i]);
#pragma unroll
        for (int i = 0; i < PV; ++i) nan_seen |= (x[i] != x[i]);
        if (vm > bt) {
          bt = vm;
          jt = j;
        }
        if (has_draft) {
          E::unpack(sd[j], x);
          vm = x[0];
#pragma unroll
          for (int i = 1; i < PV; ++i) vm = fmaxf(vm, x[i]);
#pragma unroll
          for (int i = 0; i < PV; ++i) nan_seen |= (x[i] != x[i]);
          if (vm > bd) {
            bd = vm;
            jd = j;
          }
        }
      }
    }
    int it = 0x7FFFFFFF, id = 0x7FFFFFFF;
    if (jt >= 0) {
      float x[PV];
      E::unpack(st[jt], x);
      for (int i = PV - 1; i >= 0; --i)
        if (x[i] == bt) it = e0 + jt * PV + i;
    }
    if (jd >= 0) {
      float x[PV];
      E::unpack(sd[jd], x);
      for (int i = PV - 1; i >= 0; --i)
        if (x[i] == bd) id = e0 + jd * PV + i;
    }
    warp_argmax(bt, it);
    warp_argmax(bd, id);
    nan_seen = __any_sync(0xFFFFFFFFu, nan_seen);
    if (lane == 0) {
      red_a[warp] = bt;
      red_i[warp] = it;
      red_b[warp] = bd;
      red_j[warp] = id;
      red_c[warp] = nan_seen ? 1.0f : 0.0f;
    }
    __syncthreads();
    if (tid == 0) {
      float v1 = red_a[0], v2 = red_b[0], nn = red_c[0];
      int i1 = red_i[0], i2 = red_j[0];
      for (int w = 1; w < kWarps; ++w) {
        arg_better(v1, i1, red_a[w], red_i[w]);
        arg_better(v2, i2, red_b[w], red_j[w]);
        nn = fmaxf(nn, red_c[w]);
      }
      mail_f[0] = v1;
      mail_i[0] = i1;
      mail_f[1] = v2;
      mail_i[1] = i2;
      mail_f[2] = nn;
    }
    cluster_sync();  // ---- exchange 1
    if (rank == 0 && tid == 0) {
      float v1 = -INFINITY, v2 = -INFINITY, nn = 0.0f;
      int i1 = 0x7FFFFFFF, i2 = 0x7FFFFFFF;
      for (int r = 0; r < S; ++r) {
        arg_better(v1, i1, ld_cluster_f32(map_rank(smem_addr(&mail_f[0]), r)),
                   (int)ld_cluster_u32(map_rank(smem_addr(&mail_i[0]), r)));
        arg_better(v2, i2, ld_cluster_f32(map_rank(smem_addr(&mail_f[1]), r)),
                   (int)ld_cluster_u32(map_rank(smem_addr(&mail_i[1]), r)));
        nn = fmaxf(nn, ld_cluster_f32(map_rank(smem_addr(&mail_f[2]), r)));
      }
      const bool bad = nn != 0.0f || !(v1 < INFINITY) || i1 == 0x7FFFFFFF ||
                       (has_draft && (!(v2 < INFINITY) || i2 == 0x7FFFFFFF));
      if (bad) flags |= kBadLogits;
      const int am_t = bad ? -1 : i1;
      const float al = has_draft ? ((am_t >= 0 && am_t == i2) ? 1.0f : 0.0f) : 0.0f;
      bc_i[0] = am_t;
      bc_f[0] = al;
    }
    cluster_sync();  // ---- peers may exit once rank 0 has read their mailboxes
    if (rank != 0) return;
    if constexpr (MODE == kVerifyGreedy) {
      if (tid == 0) {
        if (!bonus && !tok_ok) flags |= kBadToken;
        VerifyRecord r;
        r.acc = (!bonus && tok_ok && y == bc_i[0]) ? 1 : 0;
        r.token = bc_i[0];
        r.alpha = bc_f[0];
        r.pad = 0;
        P.rec[unit] = r;
      }
    } else {
      if (tid == 0) {
        P.alpha[b * K + k] = bc_f[0];
        if (P.tv) P.tv[b * K + k] = 1.0f - bc_f[0];
      }
    }
  } else {
    // ================= sampling path: T > 0 =================
    const float s = P.s;
    // ---- pass A: maxima ----
    typename E::MaxAcc mt, md;
    if (work) {
      for (int j = v_lo + lane; j < v_hi; j += 32) {
        mt.add(st[j]);
        if (has_draft) md.add(sd[j]);
      }
    }
    {
      const float a = warp_max(mt.get());
      const float d = warp_max(md.get());
      if (lane == 0) {
        red_a[warp] = a;
        red_b[warp] = d;
      }
    }
    __syncthreads();
    if (tid == 0) {
      float a = red_a[0], d = red_b[0];
      for (int w = 1; w < kWarps; ++w) {
        a = fmaxf(a, red_a[w]);
        d = fmaxf(d, red_b[w]);
      }
      mail_f[0] = a;
      mail_f[1] = d;
    }
    cluster_sync();  // ---- exchange 1
    if (tid == 0) {
      float a = -INFINITY, d = -INFINITY;
      for (int r = 0; r < S; ++r) {
        a = fmaxf(a, ld_cluster_f32(map_rank(smem_addr(&mail_f[0]), r)));
        d = fmaxf(d, ld_cluster_f32(map_rank(smem_addr(&mail_f[1]), r)));
      }
      bc_f[0] = __fmul_rn(a, s);  // c1t
      bc_f[1] = __fmul_rn(d, s);  // c1d
    }
    __syncthreads();
    const float c1t = bc_f[0], c1d = bc_f[1];

    // ---- pass B: normalisers ----
    float zt = 0.0f, zd = 0.0f;
    if (work) {
      for (int j = v_lo + lane; j < v_hi; j += 32) {
        float x[PV], e[PV];
        E::unpack(st[j], x);
#pragma unroll
        for (int i = 0; i < PV; ++i) e[i] = ex2(fmaf(x[i], s, -c1t));
        zt = __fadd_rn(zt, tree_sum(e));
        if (has_draft) {
          E::unpack(sd[j], x);
#pragma unroll
          for (int i = 0; i < PV; ++i) e[i] = ex2(fmaf(x[i], s, -c1d));
          zd = __fadd_rn(zd, tree_sum(e));
        }
      }
    }
    zt = warp_sum(zt);
    zd = warp_sum(zd);
    __syncthreads();  // red_* reuse
    if (lane == 0) {
      red_a[warp] = zt;
      red_b[warp] = zd;
    }
    __syncthreads();
    if (tid == 0) {
      float a = 0.0f, d = 0.0f;
      for (int w = 0; w < kWarps; ++w) {
        a = __fadd_rn(a, red_a[w]);
        d = __fadd_rn(d, red_b[w]);
      }
      mail_f[2] = a;
      mail_f[3] = d;
    }
    cluster_sync();  // ---- exchange 2
    if (tid == 0) {
      float a = 0.0f, d = 0.0f;
      for (int r = 0; r < S; ++r) {
        a = __fadd_rn(a, ld_cluster_f32(map_rank(smem_addr(&mail_f[2]), r)));
        d = __fadd_rn(d, ld_cluster_f32(map_rank(smem_addr(&mail_f[3]), r)));
      }
      const bool valid = (a > 0.0f && a < INFINITY) && (!has_draft || (d > 0.0f && d < INFINITY));
      int mode_c = 0;  // 0: overlap only, 1: residual draw, 2: draw from p
      int acc = 1;
      if constexpr (MODE == kVerify) {
        if (bonus) {
          mode_c = 2;
        } else {
          // Acceptance: u * q(y) <= p(y), with p(y), q(y) formed exactly like
          // the per-element values of the residual pass.
          const float py = __fmul_rn(ex2(fmaf(zt_y, s, -c1t)), 1.0f / a);
          const float qy = __fmul_rn(ex2(fmaf(zd_y, s, -c1d)), 1.0f / d);
          acc = (tok_ok && __fmul_rn(u, qy) <= py) ? 1 : 0;
          mode_c = acc ? 0 : 1;
        }
        if (!(u >= 0.0f && u < 1.0f) && !bonus) flags |= kBadUniform;
        if (!(uf >= 0.0f && uf < 1.0f)) flags |= kBadUniform;
        if (!tok_ok) flags |= kBadToken;
      }
      if (!valid) {
        flags |= kBadLogits;
        mode_c = 3;  // skip: invalid row
      }
      bc_f[2] = a;
      bc_f[3] = d;
      bc_f[5] = has_draft && valid ? c1d + log2f(d / a) : 0.0f;  // c1d + log2(Z_d / Z_t)
      bc_i[0] = mode_c;
      bc_i[1] = acc;
    }
    __syncthreads();
    const float Zt = bc_f[2], Zd = bc_f[3], cd2 = bc_f[5];
    int mode_c = bc_i[0];
    const int acc = bc_i[1];

    // ---- pass C ----
    float alpha_part = 0.0f, smass_part = 0.0f;
    float a_sum = 0.0f, s_sum = 0.0f;  // cluster totals (thread 0 of rank 0)
    int token = -1;
    for (int attempt = 0; attempt < 2; ++attempt) {
      if (mode_c == 0 && attempt == 0) {
        // overlap through min(log2 p, log2 q): one exp per element
        if (work && has_draft) {
          for (int j = v_lo + lane; j < v_hi; j += 32) {
            float t[PV], d[PV], e[PV], g[PV];
            E::unpack(st[j], t);
            E::unpack(sd[j], d);
#pragma unroll
            for (int i = 0; i < PV; ++i) {
              const float xt = fmaf(t[i], s, -c1t);
              const float xd = fmaf(d[i], s, -cd2);
              e[i] = ex2(fminf(xt, xd));
              if constexpr (MODE == kE2E) g[i] = (xd < xt) ? e[i] : 0.0f;
            }
            alpha_part = __fadd_rn(alpha_part, tree_sum(e));
            if constexpr (MODE == kE2E) smass_part = __fadd_rn(smass_part, tree_sum(g));
          }
        }
        alpha_part = warp_sum(alpha_part);
        smass_part = warp_sum(smass_part);
        __syncthreads();
        if (lane == 0) {
          red_a[warp] = alpha_part;
          red_b[warp] = smass_part;
        }
        __syncthreads();
        if (tid == 0) {
          float a = 0.0f, m = 0.0f;
          for (int w = 0; w < kWarps; ++w) {
            a = __fadd_rn(a, red_a[w]);
            m = __fadd_rn(m, red_b[w]);
          }
          mail_f[4] = a;
          mail_f[5] = m;
        }
        cluster_sync();  // ---- exchange 3
        if (rank == 0 && tid == 0) {
          for (int r = 0; r < S; ++r) {
            a_sum = __fadd_rn(a_sum, ld_cluster_f32(map_rank(smem_addr(&mail_f[4]), r)));
            s_sum = __fadd_rn(s_sum, ld_cluster_f32(map_rank(smem_addr(&mail_f[5]), r)));
          }
        }
        break;
      }
      if (mode_c == 3) {
        cluster_sync();  // keep the barrier count of the other branches
        break;
      }
      // ---- residual (mode 1) or target (mode 2) draw ----
      const bool resid = (mode_c == 1);
      const float ratio = __fdiv_rn(Zt, Zd);
      float run = 0.0f, mmass = 0.0f;
      const int nrounds = (v_hi - v_lo + 31) >> 5;
      if (work) {
        for (int rr = 0; rr < nrounds; ++rr) {
          const int j = v_lo + rr * 32 + lane;
          float rs = 0.0f;
          if (j < v_hi) {
            float w[PV];
            rs = resid ? draw_weights<E, true>(st[j], sd[j], s, c1t, c1d, ratio, w, mmass)
                       : draw_weights<E, false>(st[j], st[j], s, c1t, c1d, ratio, w, mmass);
          }
          const float incl = warp_incl_scan(rs, lane);
          run = __fadd_rn(run, __shfl_sync(0xFFFFFFFFu, incl, 31));
        }
      }
      mmass = warp_sum(mmass);
      __syncthreads();
      if (lane == 0) {
        warp_total[warp] = run;
        red_a[warp] = mmass;
      }
      __syncthreads();
      if (tid == 0) {
        float tot = 0.0f, a = 0.0f;
        for (int w = 0; w < kWarps; ++w) {
          tot = __fadd_rn(tot, warp_total[w]);
          a = __fadd_rn(a, red_a[w]);
        }
        mail_f[6 + attempt] = tot;  // own slot per attempt: no reuse race
        if (attempt == 0) mail_f[4] = a;
      }
      cluster_sync();  // ---- exchange 3
      if (tid == 0) {
        // Locate the CTA whose slice holds u' * total (vocabulary order).
        float off = 0.0f, tot_all = 0.0f, my_off = 0.0f, my_tot = 0.0f;
        int owner = -1, last_pos = -1;
        float parts[16];
        for (int r = 0; r < S; ++r) parts[r] = ld_cluster_f32(map_rank(smem_addr(&mail_f[6 + attempt]), r));
        for (int r = 0; r < S; ++r) tot_all = __fadd_rn(tot_all, parts[r]);
        const float thr = __fmul_rn(uf, tot_all);
        for (int r = 0; r < S; ++r) {
          const float nxt = __fadd_rn(off, parts[r]);
          if (owner < 0 && nxt > thr) owner = r;
          if (parts[r] > 0.0f) last_pos = r;
          if (r == (int)rank) {
            my_off = off;
            my_tot = parts[r];
          }
          off = nxt;
        }
        bool fallback = false;
        if (owner < 0) {
          owner = last_pos;
          fallback = true;
        }
        if (attempt == 0 && rank == 0)
          for (int r = 0; r < S; ++r) a_sum = __fadd_rn(a_sum, ld_cluster_f32(map_rank(smem_addr(&mail_f[4]), r)));
        bc_i[2] = (tot_all > 0.0f) ? 1 : 0;
        bc_i[3] = (owner == (int)rank) ? 1 : 0;
        bc_f[4] = fallback ? INFINITY : __fadd_rn(thr, -my_off);
        (void)my_tot;
      }
      __syncthreads();
      if (!bc_i[2]) {
        // Rejection with no residual mass (rounding only): draw from p.
        if (attempt == 0 && resid) {
          flags |= kEmptyResidual;
          mode_c = 2;
          continue;
        }
        break;  // no mass at all: no token
      }
      if (bc_i[3]) {
        // This CTA owns the threshold: warp offsets, then the owning warp
        // replays its rounds bit-identically to find the element.
        __shared__ int s_warp;
        __shared__ float s_thr;
        if (tid == 0) {
          const float th = bc_f[4];
          float off = 0.0f;
          int wsel = -1, wlast = -1;
          float wthr = INFINITY;
          for (int w = 0; w < kWarps; ++w) {
            const float nxt = __fadd_rn(off, warp_total[w]);
            if (wsel < 0 && nxt > th) {
              wsel = w;
              wthr = __fadd_rn(th, -off);
            }
            if (warp_total[w] > 0.0f) wlast = w;
            off = nxt;
          }
          if (wsel < 0) {
            wsel = wlast;
            wthr = INFINITY;
          }
          s_warp = wsel;
          s_thr = wthr;
        }
        __syncthreads();
        if (warp == s_warp) {
          const float th = s_thr;
          float rrun = 0.0f;
          int found = -1;
          int last_el = -1;
          for (int rr = 0; rr < nrounds && found < 0; ++rr) {
            const int j = v_lo + rr * 32 + lane;
            float rs = 0.0f, w[PV], dummy = 0.0f;
#pragma unroll
            for (int i = 0; i < PV; ++i) w[i] = 0.0f;
            if (j < v_hi)
              rs = resid ? draw_weights<E, true>(st[j], sd[j], s, c1t, c1d, ratio, w, dummy)
                         : draw_weights<E, false>(st[j], st[j], s, c1t, c1d, ratio, w, dummy);
            const float incl = warp_incl_scan(rs, lane);
            const float rtot = __shfl_sync(0xFFFFFFFFu, incl, 31);
            // remember the last positive element seen, for the fallback
            int my_last = -1;
#pragma unroll
            for (int i = 0; i < PV; ++i)
              if (w[i] > 0.0f) my_last = e0 + j * PV + i;
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, my_last >= 0);
            if (pos) last_el = __shfl_sync(0xFFFFFFFFu, my_last, 31 - __clz(pos));
            if (__fadd_rn(rrun, rtot) > th) {
              const unsigned hit = __ballot_sync(0xFFFFFFFFu, __fadd_rn(rrun, incl) > th);
              const int l = __ffs(hit) - 1;
              const float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
              if (lane == l) {
                float accu = __fadd_rn(rrun, lane > 0 ? excl : 0.0f);
                int pick = -1, lastp = -1;
#pragma unroll
                for (int i = 0; i < PV; ++i) {
                  accu = __fadd_rn(accu, w[i]);
                  if (w[i] > 0.0f) {
                    lastp = i;
                    if (pick < 0 && accu > th) pick = i;
                  }
                }
                if (pick < 0) pick = lastp;
                found = e0 + j * PV + pick;
              }
              found = __shfl_sync(0xFFFFFFFFu, found, l);
            }
            rrun = __fadd_rn(rrun, rtot);
          }
          if (found < 0) found = last_el;
          if (lane == 0) st_cluster_u32(map_rank(smem_addr(&mail_tok), 0), (uint32_t)found);
        }
      }
      break;
    }
    cluster_sync();  // ---- exchange 4: token in rank 0; peers done reading
    if (rank != 0) return;
    if (tid == 0) {
      const float izt = 1.0f / Zt;
      if (mode_c == 1 || mode_c == 2) token = (int)mail_tok;  // -1 if no draw completed
      if constexpr (MODE == kVerify) {
        VerifyRecord r;
        r.acc = acc;
        r.token = (mode_c == 3) ? -1 : token;
        r.alpha = (mode_c == 3) ? __int_as_float(0x7FC00000) : __fmul_rn(a_sum, izt);
        r.pad = 0;
        P.rec[unit] = r;
      } else if constexpr (MODE == kOverlap) {
        const float al = (mode_c == 3) ? __int_as_float(0x7FC00000) : __fmul_rn(a_sum, izt);
        P.alpha[b * K + k] = al;
        if (P.tv) P.tv[b * K + k] = 1.0f - al;
      } else {  // kE2E
        E2EStats st2;
        st2.c1t = c1t;
        st2.cd = cd2;
        st2.izt = izt;
        st2.smass = __fmul_rn(s_sum, izt);
        st2.alpha = (mode_c == 3) ? __int_as_float(0x7FC00000) : __fmul_rn(a_sum, izt);
        st2.b1 = 0.0f;
        st2.b0 = 0.0f;
        st2.pad = 0.0f;
        P.stats[unit] = st2;
      }
    }
  }

  // ================= per-row completion (rank 0 only) =================
  __shared__ int s_last;
  if (tid == 0) {
    if (flags) atomicOr(P.status, flags);
    bool need = true;
    if constexpr (MODE == kOverlap || MODE == kOverlapGreedy) need = (P.surv != nullptr || P.exp_acc != nullptr);
    int last = 0;
    if (need) {
      __threadfence();
      const uint32_t per_row = kVerifyMode ? (uint32_t)(K + 1) : (uint32_t)K;
      const uint32_t old = atomicAdd(&P.row_cnt[b], 1u);
      last = (old == per_row - 1) ? 1 : 0;
      if (last) __threadfence();
    }
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;

  if constexpr (kVerifyMode) {
    // One warp decides the row: first rejection in prefix order.
    if (warp != 0) return;
    const VerifyRecord* rr = P.rec + (long long)b * (K + 1);
    int nacc = K;
    for (int base = 0; base < K; base += 32) {
      const int kk = base + lane;
      bool rej = false;
      if (kk < K) rej = (__ldcg(&rr[kk].acc) == 0);
      const unsigned m = __ballot_sync(0xFFFFFFFFu, rej);
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
    __syncwarp();
    // Leave the workspace zero-filled: the records of this row are consumed.
    VerifyRecord* rw = P.rec + (long long)b * (K + 1);
    for (int kk = lane; kk <= K; kk += 32) rw[kk] = VerifyRecord{0, 0, 0.0f, 0u};
    if (lane == 0) {
      P.n_accepted[b] = nacc;
      P.row_cnt[b] = 0;
    }
  } else if constexpr (MODE == kOverlap || MODE == kOverlapGreedy) {
    if (tid != 0) return;
    float pr = 1.0f, sum = 0.0f;
    for (int kk = 0; kk < K; ++kk) {
      pr = __fmul_rn(pr, __ldcg(&P.alpha[b * K + kk]));
      sum = __fadd_rn(sum, pr);
      if (P.surv) P.surv[b * K + kk] = pr;
    }
    if (P.exp_acc) P.exp_acc[b] = sum;
    P.row_cnt[b] = 0;
  } else {  // kE2E
    __shared__ int s_glast;
    if (tid == 0) {
      E2EStats* sr = P.stats + (long long)b * K;
      // prefix products P_{k-1} and suffix sums G_k = 1 + alpha_{k+1} G_{k+1}
      float g = 1.0f;
      float suffix[64];
      for (int kk = K - 1; kk >= 0; --kk) {
        suffix[kk] = g;
        g = fmaf(__ldcg(&sr[kk].alpha), g, 1.0f);
      }
      float pre = 1.0f, rowl = 0.0f;
      const float scale = P.grad_scale / (float)P.B;
      for (int kk = 0; kk < K; ++kk) {
        const float al = __ldcg(&sr[kk].alpha);
        const float coef = __fmul_rn(__fmul_rn(scale, pre), suffix[kk]);
        const float A = __fmul_rn(__fmul_rn(coef, __ldcg(&sr[kk].izt)), P.inv_t);
        const float S_ = __ldcg(&sr[kk].smass);
        sr[kk].b1 = __fmul_rn(A, 1.0f - S_);
        sr[kk].b0 = __fmul_rn(A, -S_);
        pre = __fmul_rn(pre, al);
        rowl = __fadd_rn(rowl, pre);
        if (P.alpha) P.alpha[b * K + kk] = al;
      }
      P.row_loss[b] = rowl;
      P.row_cnt[b] = 0;
      __threadfence();
      const uint32_t old = atomicAdd(P.glob_cnt, 1u);
      s_glast = (old == (uint32_t)P.B - 1) ? 1 : 0;
      if (s_glast) __threadfence();
    }
    __syncthreads();
    if (!s_glast || warp != 0) return;
    float acc_l = 0.0f;
    for (int i = lane; i < P.B; i += 32) {
      acc_l = __fadd_rn(acc_l, __ldcg(&P.row_loss[i]));
      P.row_loss[i] = 0.0f;  // consumed: leave the workspace zero-filled
    }
    acc_l = warp_sum(acc_l);
    if (lane == 0) {
      *P.loss = acc_l / (float)P.B;
      *P.glob_cnt = 0;
    }
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
