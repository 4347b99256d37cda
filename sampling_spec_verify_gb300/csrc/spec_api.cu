// C ABI of the verify library: argument checks, workspace layout, launch
// plan and kernel launches.  No entry point allocates device memory or
// synchronises the stream.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>

#include "pipe.cuh"
#include "spec_verify.h"

namespace {

using ssv::Bf16;
using ssv::E2EStats;
using ssv::F32;
using ssv::PipeParams;
using ssv::Rec;

constexpr int kMaxK = 64;
constexpr int kMaxDevices = 64;
constexpr int kStageCap = 32768;  // bytes of logits per shared-memory stage
constexpr int kMinChunk = 256;    // smallest chunk a launch override may force
constexpr int kSmemSlack = 1024;

std::atomic<int> g_chunk_override{0};
std::atomic<int> g_stage_override{0};

struct DevInfo {
  int sms = 0;
  int smem_optin = 0;
};

DevInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

bool device_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::call_once(g_dev_once[dev], [dev]() {
    DevInfo d;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    g_dev[dev] = d;
  });
  *out = g_dev[dev];
  return out->sms > 0 && out->smem_optin > 0;
}

int elem_size(spec_dtype_t dt) { return dt == SPEC_BF16 ? 2 : 4; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

spec_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// ---- chunking ----------------------------------------------------------------------

// Largest chunk (elements) for rows of `es`-byte logits, `rows` rows per stage.
int chunk_cap(int es, int rows, bool draws) {
  const int pv = 16 / es;
  int cap = kStageCap / (rows * es);
  const int ov = g_chunk_override.load();
  if (ov > 0) cap = ov < cap ? ov : cap;
  if (draws) {
    const int segcap = ssv::kMaxSegs * ssv::kSegVecs * pv;
    cap = cap < segcap ? cap : segcap;
  }
  cap = cap / pv * pv;
  return cap < pv ? pv : cap;
}

struct Chunking {
  int C = 0, Lc = 0;
};

// Chunk length for C chunks of V logits: a multiple of 128 bytes (so that
// chunks of 128-byte-aligned rows start on cache-line boundaries) unless the
// cap is smaller than that, and never above the cap.
int chunk_len(int es, int V, int C, int cap) {
  const int pv = 16 / es;
  const int line = 128 / es;
  int Lc = (int)(ceil_div(ceil_div(V, C), line) * line);
  if (Lc > cap) Lc = (int)(ceil_div(ceil_div(V, C), pv) * pv);
  return Lc;
}

Chunking chunking(int es, int V, int rows, bool draws) {
  const int cap = chunk_cap(es, rows, draws);
  Chunking ch;
  ch.Lc = chunk_len(es, V, (int)ceil_div(V, cap), cap);
  ch.C = (int)ceil_div(V, ch.Lc);  // every chunk starts below V
  return ch;
}

// Chunks per unit that a workspace must hold for any dtype / temperature.
int ws_chunks(int V) {
  int cap = kStageCap / (2 * 4);  // fp32, two rows per stage
  const int ov = g_chunk_override.load();
  if (ov > 0) {
    const int o = ov < kMinChunk ? kMinChunk : ov;
    cap = o < cap ? o : cap;
  }
  cap = cap / 8 * 8;  // the widest vector (8 bf16) rounds every chunk cap down to this
  return (int)ceil_div(V, cap);
}

// ---- workspace layout (all offsets 256-byte aligned) ----------------------------

struct WsLayout {
  size_t part1 = 0, part2 = 0, seg = 0, cnt = 0, rec = 0, stats = 0, row_cnt = 0, row_loss = 0, ctl = 0, total = 0;
  bool has_seg = false;
};

WsLayout ws_layout(bool e2e, bool with_seg, long long units, int B, int C) {
  WsLayout w;
  size_t off = 0;
  const size_t tasks = (size_t)units * (size_t)C;
  w.part1 = off;
  off += align256(tasks * 4 * sizeof(uint64_t));
  w.part2 = off;
  off += align256(tasks * sizeof(uint64_t));
  w.has_seg = with_seg;
  if (with_seg) {
    w.seg = off;
    off += align256(tasks * ssv::kMaxSegs * sizeof(float));
  }
  w.cnt = off;
  off += align256((size_t)units * sizeof(uint32_t));
  if (e2e) {
    w.stats = off;
    off += align256((size_t)units * sizeof(E2EStats));
  } else {
    w.rec = off;
    off += align256((size_t)units * sizeof(Rec));
  }
  w.row_cnt = off;
  off += align256((size_t)B * sizeof(uint32_t));
  if (e2e) {
    w.row_loss = off;
    off += align256((size_t)B * sizeof(float));
  }
  w.ctl = off;
  off += 256;
  w.total = off;
  return w;
}

void bind_workspace(PipeParams& P, const WsLayout& w, void* ws, size_t bytes) {
  char* base = static_cast<char*>(ws);
  P.part1 = reinterpret_cast<uint64_t*>(base + w.part1);
  P.part2 = reinterpret_cast<uint64_t*>(base + w.part2);
  P.seg = w.has_seg ? reinterpret_cast<uint32_t*>(base + w.seg) : nullptr;
  P.cnt = reinterpret_cast<uint32_t*>(base + w.cnt);
  P.rec = w.stats ? nullptr : reinterpret_cast<Rec*>(base + w.rec);
  P.stats = w.stats ? reinterpret_cast<E2EStats*>(base + w.stats) : nullptr;
  P.row_cnt = reinterpret_cast<uint32_t*>(base + w.row_cnt);
  P.row_loss = w.row_loss ? reinterpret_cast<float*>(base + w.row_loss) : nullptr;
  P.ctl = reinterpret_cast<uint32_t*>(base + w.ctl);
  P.ws = reinterpret_cast<uint8_t*>(base);
  P.ws_bytes = bytes;
}

// ---- launch plan -------------------------------------------------------------------

struct Plan {
  int C = 0, Lc = 0, D = 0, stage = 0, doff = 0, smem = 0, G = 0;
};

template <class E, int MODE>
std::atomic<uint64_t>& prepared_mask() {
  static std::atomic<uint64_t> m{0};
  return m;
}

template <class E, int MODE>
int static_smem() {
  static std::atomic<int> v{-1};
  int x = v.load();
  if (x < 0) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, ssv::pipe_kernel<E, MODE>) != cudaSuccess) return -1;
    x = (int)a.sharedSizeBytes;
    v.store(x);
  }
  return x;
}

std::mutex g_occ_mu;
std::map<std::tuple<const void*, int, int>, int> g_occ;  // (kernel, smem, device) -> CTAs per SM

// Resident CTAs per SM of `fn` with `smem` dynamic bytes (queried once per
// kernel, size and device: the query costs tens of microseconds).
template <class Fn>
int occupancy(Fn fn, int smem, int dev) {
  const auto key = std::make_tuple((const void*)fn, smem, dev);
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    const auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, ssv::kThreads, (size_t)smem) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lk(g_occ_mu);
  g_occ[key] = nb;
  return nb;
}

// Sets the kernel's shared-memory limit (once per device) and computes the
// plan: chunking, stages that fit, and the persistent grid.  In the sampling
// modes the chunk is shrunk until kLag + 4 stages fit (the kLag + 1 stages a
// CTA holds for its two passes, and three in flight).
template <class E, int MODE>
spec_status_t make_plan(int V, int rows, Plan* pl) {
  constexpr bool kSample = !(MODE == ssv::kVerifyGreedy || MODE == ssv::kOverlapGreedy);
  DevInfo di;
  if (!device_info(&di)) return SPEC_ERR_CUDA;
  auto fn = ssv::pipe_kernel<E, MODE>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  const int sstat = static_smem<E, MODE>();
  if (sstat < 0) return SPEC_ERR_CUDA;
  const int avail = di.smem_optin - sstat - kSmemSlack;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(prepared_mask<E, MODE>().load() & bit)) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, avail) != cudaSuccess)
      return SPEC_ERR_CUDA;
    prepared_mask<E, MODE>().fetch_or(bit);
  }
  Chunking ch = chunking(E::ES, V, rows, MODE == ssv::kVerify);
  const int cap = chunk_cap(E::ES, rows, MODE == ssv::kVerify);
  const int want = kSample ? ssv::kLag + 4 : 4;
  int c_try = ch.C;
  Plan p;
  for (;;) {
    p.C = ch.C;
    p.Lc = ch.Lc;
    p.doff = (int)((ch.Lc * E::ES + 127) / 128 * 128);
    p.stage = rows == 2 ? (int)((p.doff + ch.Lc * E::ES + 127) / 128 * 128) : p.doff;
    if (avail / p.stage >= want || g_chunk_override.load() > 0) break;
    // smaller chunks, more stages, as long as the workspace holds the chunks
    const int nLc = chunk_len(E::ES, V, c_try + 1, cap);
    const int nC = (int)ceil_div(V, nLc);
    if (nC > ws_chunks(V)) break;
    ++c_try;
    ch.Lc = nLc;
    ch.C = nC;
  }
  int D = avail / p.stage;
  if (D > ssv::kMaxStages) D = ssv::kMaxStages;
  const int dmin = kSample ? ssv::kLag + 2 : 2;
  if (D < dmin) return SPEC_ERR_UNSUPPORTED;
  const int ovs = g_stage_override.load();
  if (ovs > 0 && ovs < D) D = ovs < dmin ? dmin : ovs;
  p.D = D;
  p.smem = D * p.stage;
  const int nb = occupancy(fn, p.smem, dev);
  if (nb < 0) return SPEC_ERR_CUDA;
  if (nb < 1) return SPEC_ERR_UNSUPPORTED;
  p.G = nb * di.sms;
  // a unit's chunks must sit in different CTAs for the phase-2 exchange
  if (kSample && p.C > p.G) return SPEC_ERR_UNSUPPORTED;
  *pl = p;
  return SPEC_OK;
}

template <int MODE>
spec_status_t make_plan_dt(spec_dtype_t dt, int V, int rows, Plan* pl) {
  return dt == SPEC_BF16 ? make_plan<Bf16, MODE>(V, rows, pl) : make_plan<F32, MODE>(V, rows, pl);
}

template <class E, int MODE>
cudaError_t launch(const PipeParams& P, const Plan& pl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.G, 1, 1);
  cfg.blockDim = dim3(ssv::kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the exchange between CTAs needs it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ssv::pipe_kernel<E, MODE>, P);
}

template <int MODE>
cudaError_t launch_dt(spec_dtype_t dt, const PipeParams& P, const Plan& pl, cudaStream_t stream) {
  return dt == SPEC_BF16 ? launch<Bf16, MODE>(P, pl, stream) : launch<F32, MODE>(P, pl, stream);
}

void fill_plan(PipeParams& P, const Plan& pl, int es, int V, const void* t, const void* d) {
  P.C = pl.C;
  P.Lc = pl.Lc;
  P.D = pl.D;
  P.stage = pl.stage;
  P.doff = pl.doff;
  P.aligned = aligned16(t) && (!d || aligned16(d)) && ((long long)V * es) % 16 == 0;
}

template <class E>
cudaError_t launch_grad(const ssv::GradParams& G, cudaStream_t stream) {
  const int nvec = G.aligned ? G.V / E::PV : G.V;
  int gx = (nvec + 256 * 2 - 1) / (256 * 2);
  gx = gx < 1 ? 1 : gx;
  const int gy = G.units < 65535 ? G.units : 65535;
  ssv::e2e_grad_kernel<E><<<dim3(gx, gy, 1), 256, 0, stream>>>(G);
  return cudaGetLastError();
}

bool dims_ok(int B, int K, int V) { return B >= 0 && K >= 0 && K <= kMaxK && V >= 1; }

bool dtype_ok(spec_dtype_t dt) { return dt == SPEC_F32 || dt == SPEC_BF16; }

}  // namespace

extern "C" {

int spec_abi_version(void) { return 3; }

const char* spec_status_string(spec_status_t s) {
  switch (s) {
    case SPEC_OK:
      return "ok";
    case SPEC_ERR_INVALID_ARG:
      return "invalid argument";
    case SPEC_ERR_UNSUPPORTED:
      return "unsupported size or configuration";
    case SPEC_ERR_CUDA:
      return "CUDA runtime error";
  }
  return "unknown status";
}

void spec_set_launch_override(int chunk_elems, int stages) {
  g_chunk_override.store(chunk_elems >= kMinChunk ? chunk_elems : 0);
  g_stage_override.store(stages >= 2 && stages <= ssv::kMaxStages ? stages : 0);
}

spec_status_t spec_launch_shape(spec_dtype_t dtype, int V, int* chunk_elems, int* chunks, int* threads,
                                int* smem_bytes, int* ctas, int* stages) {
  if (!dtype_ok(dtype) || V < 1) return SPEC_ERR_INVALID_ARG;
  Plan pl;
  const spec_status_t r = make_plan_dt<ssv::kVerify>(dtype, V, 2, &pl);
  if (r != SPEC_OK) return r;
  if (chunk_elems) *chunk_elems = pl.Lc;
  if (chunks) *chunks = pl.C;
  if (threads) *threads = ssv::kThreads;
  if (smem_bytes) *smem_bytes = pl.smem;
  if (ctas) *ctas = pl.G;
  if (stages) *stages = pl.D;
  return SPEC_OK;
}

size_t spec_verify_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return ws_layout(false, true, (long long)B * (K + 1), B, ws_chunks(V)).total;
}

spec_status_t spec_verify(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B, int K,
                          int V, float temperature, const int32_t* draft_tokens, const float* u_accept,
                          const float* u_final, int32_t* out_tokens, int32_t* n_accepted, float* alpha_out,
                          uint32_t* dev_status, void* workspace, size_t workspace_bytes, void* stream) {
  if (!dims_ok(B, K, V) || !dtype_ok(dtype)) return SPEC_ERR_INVALID_ARG;
  if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  const bool greedy = temperature == 0.0f;
  if (!target_logits || !out_tokens || !n_accepted || !workspace) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && !draft_logits && (!greedy || alpha_out)) return SPEC_ERR_INVALID_ARG;
  if (!greedy && (!u_final || (K > 0 && !u_accept))) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * (K + 1);
  if (units * (long long)ws_chunks(V) > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_layout(false, true, units, B, ws_chunks(V)).total) return SPEC_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const int rows = (greedy && !alpha_out) ? 1 : 2;  // greedy without overlap reads no draft row
  Plan pl;
  {
    const spec_status_t r = greedy ? make_plan_dt<ssv::kVerifyGreedy>(dtype, V, rows, &pl)
                                   : make_plan_dt<ssv::kVerify>(dtype, V, rows, &pl);
    if (r != SPEC_OK) return r;
  }
  const WsLayout wl = ws_layout(false, !greedy, units, B, pl.C);
  if (workspace_bytes < wl.total) return SPEC_ERR_INVALID_ARG;

  PipeParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = K + 1;
  P.V = V;
  P.units = (int)units;
  fill_plan(P, pl, es, V, target_logits, draft_logits);
  P.s = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = greedy ? 0.0f : (float)(1.0 / (double)temperature);
  P.draft_tokens = draft_tokens;
  P.u_accept = u_accept;
  P.u_final = u_final;
  P.out_tokens = out_tokens;
  P.n_accepted = n_accepted;
  P.alpha = alpha_out;
  P.status = dev_status;
  bind_workspace(P, wl, workspace, wl.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = greedy ? launch_dt<ssv::kVerifyGreedy>(dtype, P, pl, st) : launch_dt<ssv::kVerify>(dtype, P, pl, st);
  return from_cuda(e);
}

size_t spec_overlap_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return ws_layout(false, false, (long long)B * K, B, ws_chunks(V)).total;
}

spec_status_t spec_overlap(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B, int K,
                           int KT, int V, float temperature, float* alpha, float* tv, float* prefix_survival,
                           float* expected_accepted, uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!dims_ok(B, K, V) || !dtype_ok(dtype) || KT < K) return SPEC_ERR_INVALID_ARG;
  if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0) return SPEC_OK;
  if (K == 0) {
    if (expected_accepted) return from_cuda(cudaMemsetAsync(expected_accepted, 0, (size_t)B * sizeof(float), st));
    return SPEC_OK;
  }
  if (!target_logits || !draft_logits || !alpha) return SPEC_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * K;
  if (units * (long long)ws_chunks(V) > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_layout(false, false, units, B, ws_chunks(V)).total) return SPEC_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const bool greedy = temperature == 0.0f;
  Plan pl;
  {
    const spec_status_t r = greedy ? make_plan_dt<ssv::kOverlapGreedy>(dtype, V, 2, &pl)
                                   : make_plan_dt<ssv::kOverlap>(dtype, V, 2, &pl);
    if (r != SPEC_OK) return r;
  }
  const WsLayout wl = ws_layout(false, false, units, B, pl.C);
  if (workspace_bytes < wl.total) return SPEC_ERR_INVALID_ARG;
  PipeParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = KT;
  P.V = V;
  P.units = (int)units;
  fill_plan(P, pl, es, V, target_logits, draft_logits);
  P.s = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = greedy ? 0.0f : (float)(1.0 / (double)temperature);
  P.alpha = alpha;
  P.tv = tv;
  P.surv = prefix_survival;
  P.exp_acc = expected_accepted;
  P.status = dev_status;
  bind_workspace(P, wl, workspace, wl.total);
  cudaError_t e = greedy ? launch_dt<ssv::kOverlapGreedy>(dtype, P, pl, st) : launch_dt<ssv::kOverlap>(dtype, P, pl, st);
  return from_cuda(e);
}

size_t spec_e2e_tv_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return ws_layout(true, false, (long long)B * K, B, ws_chunks(V)).total;
}

spec_status_t spec_e2e_tv_fwd_bwd(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B,
                                  int K, int KT, int V, float temperature, float grad_scale, float* loss_out,
                                  float* alpha_out, float* grad_draft_logits, uint32_t* dev_status, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!dims_ok(B, K, V) || !dtype_ok(dtype) || KT < K) return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature) || !std::isfinite(grad_scale)) return SPEC_ERR_INVALID_ARG;
  if (!loss_out) return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0 || K == 0) return from_cuda(cudaMemsetAsync(loss_out, 0, sizeof(float), st));
  if (!target_logits || !draft_logits || !grad_draft_logits || !workspace) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * K;
  if (units * (long long)ws_chunks(V) > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  if (workspace_bytes < ws_layout(true, false, units, B, ws_chunks(V)).total) return SPEC_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  Plan pl;
  {
    const spec_status_t r = make_plan_dt<ssv::kE2E>(dtype, V, 2, &pl);
    if (r != SPEC_OK) return r;
  }
  const WsLayout wl = ws_layout(true, false, units, B, pl.C);
  if (workspace_bytes < wl.total) return SPEC_ERR_INVALID_ARG;
  PipeParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = KT;
  P.V = V;
  P.units = (int)units;
  fill_plan(P, pl, es, V, target_logits, draft_logits);
  P.s = (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = (float)(1.0 / (double)temperature);
  P.grad_scale = grad_scale;
  P.alpha = alpha_out;
  P.loss = loss_out;
  P.status = dev_status;
  bind_workspace(P, wl, workspace, wl.total);
  cudaError_t e = launch_dt<ssv::kE2E>(dtype, P, pl, st);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  ssv::GradParams G = {};
  G.target = target_logits;
  G.draft = draft_logits;
  G.B = B;
  G.K = K;
  G.KT = KT;
  G.V = V;
  G.units = (int)units;
  G.aligned = P.aligned && aligned16(grad_draft_logits);
  G.s = P.s;
  G.stats = P.stats;
  G.grad = grad_draft_logits;
  e = dtype == SPEC_BF16 ? launch_grad<Bf16>(G, st) : launch_grad<F32>(G, st);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  // The per-position statistics are consumed by the gradient kernel; clear
  // them so the workspace is zero-filled again when the call completes.
  return from_cuda(cudaMemsetAsync(static_cast<char*>(workspace) + wl.stats, 0, (size_t)units * sizeof(E2EStats), st));
}

}  // extern "C"
