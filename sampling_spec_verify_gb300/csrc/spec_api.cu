// C ABI of the verify library: argument checks, workspace layout, launch
// shape and kernel launches.  No entry point allocates device memory or
// synchronises the stream.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>

#include "spec_verify.h"
#include "sweep.cuh"
#include "pipe.cuh"
#include "truncate.cuh"
#include "topk.cuh"
#include "schedule.cuh"
#include "tree.cuh"

namespace {

using ssv::Bf16;
using ssv::E2EStats;
using ssv::F32;
using ssv::SweepParams;
using ssv::VerifyRecord;

constexpr int kMaxK = 64;
constexpr int kMaxCluster = 16;
constexpr int kMaxDevices = 64;
constexpr int kStaticSmemReserve = 4096;

std::atomic<int> g_cluster_override{0};
std::atomic<int> g_stage_override{0};
std::atomic<int> g_kernel_override{0};  // 0 automatic, 1 single-read sweep, 2 two-pass sweep

// Kernels launched by this library (counted on the host when a launch is
// enqueued without error).
std::atomic<unsigned long long> g_launches{0};

cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

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

// Per-device "attributes already set" flags for each kernel instantiation.
template <class Fn>
cudaError_t prepare_kernel(Fn fn, std::atomic<uint64_t>& done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  DevInfo di;
  if (!device_info(&di)) return cudaErrorInvalidDevice;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin - kStaticSmemReserve);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  done_mask.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

struct Shape {
  int S = 0;     // CTAs per cluster
  int L = 0;     // slice length (elements)
  int nst = 0;   // shared-memory stages per CTA (2: the next unit is prefetched)
  int smem = 0;  // dynamic shared memory per CTA: nst stages of both rows
  int G = 0;     // clusters launched (persistent)
};

int elem_size(spec_dtype_t dt) { return dt == SPEC_BF16 ? 2 : 4; }

std::mutex g_occ_mu;
std::map<std::tuple<const void*, int, int, int>, int> g_occ;  // (kernel, S, smem, device) -> clusters

// Clusters of S CTAs with `smem` dynamic bytes each that fit on the device at once.
template <class Fn>
int max_active_clusters(Fn fn, int S, int smem, int threads = ssv::kThreads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple((const void*)fn, S, smem, dev);
  {
    std::lock_guard<std::mutex> g(g_occ_mu);
    auto itc = g_occ.find(key);
    if (itc != g_occ.end()) return itc->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> g(g_occ_mu);
  g_occ[key] = n;
  return n;
}

// Picks the cluster size S and the stage count for a sweep over V: the
// stages must fit in shared memory, and among the shapes that fit the one
// with the lowest estimated time wins -- (units per cluster, rounded up) x
// (vectors per thread + a fixed per-unit allowance for the
// exchanges, larger when the load of a unit is not prefetched).
template <class Fn>
bool pick_shape(Fn fn, int es, long long units, int V, int rows, Shape* out) {
  DevInfo di;
  if (!device_info(&di)) return false;
  const long long smem_max = di.smem_optin - kStaticSmemReserve;
  const int pv = 16 / es;
  const int ov = g_cluster_override.load();
  const int ovs = g_stage_override.load();
  double best_cost = -1.0;
  for (int nst = 2; nst >= 1; --nst) {
    if (ovs > 0 && nst != ovs) continue;
    for (int S = (ov > 0 ? ov : 1); S <= (ov > 0 ? ov : kMaxCluster); ++S) {
      long long L = ((long long)V + S - 1) / S;
      L = (L + 7) / 8 * 8;
      const long long smem = (long long)rows * nst * L * es;
      if (smem > smem_max) continue;
      const long long nvec = L / pv;
      long long cpt = (nvec + ssv::kThreads - 1) / ssv::kThreads;
      if ((cpt & 1) == 0) ++cpt;
      const int G = max_active_clusters(fn, S, (int)smem);
      if (G <= 0) continue;
      const long long Ge = units < G ? units : G;
      const double cost = (double)((units + Ge - 1) / Ge) * ((double)cpt + (nst == 2 ? 2.0 : 4.0));
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        out->S = S;
        out->L = (int)L;
        out->nst = nst;
        out->smem = (int)smem;
        out->G = (int)Ge;
      }
    }
  }
  return best_cost >= 0;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

spec_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

template <class E, int MODE>
std::atomic<uint64_t>& prepared_mask() {
  static std::atomic<uint64_t> m{0};
  return m;
}

// Sets the kernel's attributes (once per device) and picks its launch shape.
template <class E, int MODE>
spec_status_t shape_for(long long units, int V, int rows, Shape* sh) {
  auto fn = ssv::sweep_kernel<E, MODE>;
  if (prepare_kernel(fn, prepared_mask<E, MODE>()) != cudaSuccess) return SPEC_ERR_CUDA;
  if (!pick_shape(fn, E::ES, units, V, rows, sh)) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

// rows: logit rows staged per unit (2, or 1 when no draft row is read).
template <int MODE>
spec_status_t shape_for_dt(spec_dtype_t dt, long long units, int V, int rows, Shape* sh) {
  return dt == SPEC_BF16 ? shape_for<Bf16, MODE>(units, V, rows, sh) : shape_for<F32, MODE>(units, V, rows, sh);
}

// Sets the attributes of the dtype's instantiation of a mode whose launch
// shape was picked with another mode's (same code size and shared memory).
template <int MODE>
cudaError_t prepare_dt(spec_dtype_t dt) {
  return dt == SPEC_BF16 ? prepare_kernel(ssv::sweep_kernel<Bf16, MODE>, prepared_mask<Bf16, MODE>())
                         : prepare_kernel(ssv::sweep_kernel<F32, MODE>, prepared_mask<F32, MODE>());
}

template <class E, int MODE>
cudaError_t launch_sweep(const SweepParams& P0, const Shape& sh, cudaStream_t stream) {
  auto fn = ssv::sweep_kernel<E, MODE>;
  SweepParams P = P0;
  // vectors per thread: enough for the slice, rounded up to an odd count
  const int nvec = P.L / E::PV;
  P.cpt = (nvec + ssv::kThreads - 1) / ssv::kThreads;
  if ((P.cpt & 1) == 0) ++P.cpt;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sh.G * sh.S), 1, 1);
  cfg.blockDim = dim3(ssv::kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)sh.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, fn, P));
}

template <int MODE>
cudaError_t launch_sweep_dt(spec_dtype_t dt, const SweepParams& P, const Shape& sh, cudaStream_t stream) {
  return dt == SPEC_BF16 ? launch_sweep<Bf16, MODE>(P, sh, stream) : launch_sweep<F32, MODE>(P, sh, stream);
}

template <class E>
cudaError_t launch_grad(const ssv::GradParams& G, cudaStream_t stream) {
  const int nvec = G.aligned ? G.V / E::PV : G.V;
  int gx = (nvec + 256 * 2 - 1) / (256 * 2);
  gx = gx < 1 ? 1 : gx;
  const int gy = G.units < 65535 ? G.units : 65535;
  ssv::e2e_grad_kernel<E><<<dim3(gx, gy, 1), 256, 0, stream>>>(G);
  return counted(cudaGetLastError());
}

// ---- the two-pass sweep (pass A from HBM, pass C from L2) -------------------------

struct PShape {
  int S = 0, G = 0, NV = 0, CV = 0, NCH = 0, WV = 0, NS = 0, rows = 0, smem = 0;
};

constexpr int kPSmemReserve = 1024;

template <class Fn>
cudaError_t prepare_pipe(Fn fn, std::atomic<uint64_t>& done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  DevInfo di;
  if (!device_info(&di)) return cudaErrorInvalidDevice;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           di.smem_optin - (int)sizeof(ssv::PipeSmem) - kPSmemReserve);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  done_mask.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

// Vectors per lane per row of a chunk.  Stages holding target and draft rows
// take 4 (64 KB, three stages): fewer, larger items beat a deeper ring there,
// as each item costs a barrier wait, a warp sync and an arrival per consumer
// warp.  Target-only stages (greedy) take 3 (24 KB, eight stages), which
// measured faster for them (56.5 against 60.4 µs at B=128, K=7, V=129280).
constexpr int kPipeVpl = 4;
constexpr int kPipeVplTarget = 3;
constexpr int pipe_vpl(int rows) { return rows == 1 ? kPipeVplTarget : kPipeVpl; }
static_assert(32 * kPipeVpl <= ssv::kPSegV, "a draw's warp sub-segment fits the completion warp's copy of it");

// Picks the cluster size S for a two-pass sweep: every S whose slices fit the
// ring (at most kPMaxCh chunks per slice, S x chunks <= kPMaxParts, at least
// three stages) is costed as (waves of units over the resident clusters) x
// (the fresh bytes of one CTA's slice over its share of HBM bandwidth, plus a
// fixed allowance per unit); slices above 320 KB pay a penalty: every
// resident CTA holds one unit slice in L2 between its two passes, and beyond
// about 48 MB in all (152 x 320 KB) the pass-C copies start to miss L2 and
// read HBM again (measured: one-CTA slices of 517 KB read 25% more DRAM
// bytes than the logits hold, two-CTA slices of 258 KB read them once).
template <class Fn>
bool pick_pipe_shape(Fn fn, int es, long long units, int V, int rows, PShape* out) {
  DevInfo di;
  if (!device_info(&di)) return false;
  const long long smem_avail = di.smem_optin - (long long)sizeof(ssv::PipeSmem) - kPSmemReserve;
  const int pv = 16 / es;
  const long long nvec_row = V / pv;
  const int vpl = pipe_vpl(rows);
  const long long CV = (long long)ssv::kPNC * 32 * vpl;
  const int ov = g_cluster_override.load();
  const int ovs = g_stage_override.load();
  double best = -1.0;
  for (int S = (ov > 0 ? ov : 1); S <= (ov > 0 ? ov : ssv::kPMaxS); ++S) {
    const long long NV = (nvec_row + S - 1) / S;
    long long NCH = (NV + CV - 1) / CV;
    if (NCH < 1) NCH = 1;
    if (NCH > ssv::kPMaxCh || S * NCH > ssv::kPMaxParts) continue;
    const long long stage = (long long)rows * CV * 16;
    const long long fixed = (long long)(ssv::pipe_mbox_bytes(S) + ssv::pipe_wt_bytes((int)NCH));
    long long NS = (smem_avail - fixed) / stage;
    if (NS > ssv::kPMaxNS) NS = ssv::kPMaxNS;
    if (ovs > 0 && NS > ovs) NS = ovs;
    if (NS < 1 || (ovs == 0 && NS < 3)) continue;
    const int G = max_active_clusters(fn, S, (int)ssv::pipe_dyn_bytes((int)NS, rows, (int)CV, S, (int)NCH),
                                      ssv::kPThreads);
    if (G <= 0) continue;
    const long long Ge = units < G ? units : G;
    const double waves = (double)((units + Ge - 1) / Ge);
    const double bytes_cta = (double)NV * rows * 16.0;
    double bw = 6.8e12 / (double)(Ge * S);
    if (bw > 1.2e11) bw = 1.2e11;
    double t = waves * (bytes_cta / bw + 1.0e-6);
    if (bytes_cta > 320.0 * 1024.0) t *= 1.5;
    if (best < 0 || t < best) {
      best = t;
      out->S = S;
      out->G = (int)Ge;
      out->NV = (int)NV;
      out->CV = (int)CV;
      out->NCH = (int)NCH;
      out->WV = 32 * vpl;
      out->NS = (int)NS;
      out->rows = rows;
      out->smem = (int)ssv::pipe_dyn_bytes((int)NS, rows, (int)CV, S, (int)NCH);
    }
  }
  return best >= 0;
}

template <class E, int MODE, int VPL>
std::atomic<uint64_t>& pipe_prepared_mask() {
  static std::atomic<uint64_t> m{0};
  return m;
}

template <class E, int MODE, int VPL>
spec_status_t pipe_shape_for(long long units, int V, int rows, PShape* sh) {
  auto fn = ssv::pipe_kernel<E, MODE, VPL>;
  if (prepare_pipe(fn, pipe_prepared_mask<E, MODE, VPL>()) != cudaSuccess) return SPEC_ERR_CUDA;
  if (!pick_pipe_shape(fn, E::ES, units, V, rows, sh)) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

// Only greedy verify stages the target alone (rows == 1).
template <int MODE>
spec_status_t pipe_shape_dt(spec_dtype_t dt, long long units, int V, int rows, PShape* sh) {
  if constexpr (MODE == ssv::kPGreedy) {
    if (rows == 1)
      return dt == SPEC_BF16 ? pipe_shape_for<Bf16, MODE, kPipeVplTarget>(units, V, rows, sh)
                             : pipe_shape_for<F32, MODE, kPipeVplTarget>(units, V, rows, sh);
  }
  if (rows != 2) return SPEC_ERR_UNSUPPORTED;
  return dt == SPEC_BF16 ? pipe_shape_for<Bf16, MODE, kPipeVpl>(units, V, rows, sh)
                         : pipe_shape_for<F32, MODE, kPipeVpl>(units, V, rows, sh);
}

template <class E, int MODE, int VPL>
cudaError_t launch_pipe(const ssv::PipeParams& P, const PShape& sh, cudaStream_t stream) {
  auto fn = ssv::pipe_kernel<E, MODE, VPL>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sh.G * sh.S), 1, 1);
  cfg.blockDim = dim3(ssv::kPThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)sh.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sh.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, fn, P));
}

template <int MODE>
cudaError_t launch_pipe_dt(spec_dtype_t dt, const ssv::PipeParams& P, const PShape& sh, cudaStream_t stream) {
  if constexpr (MODE == ssv::kPGreedy) {
    if (sh.rows == 1)
      return dt == SPEC_BF16 ? launch_pipe<Bf16, MODE, kPipeVplTarget>(P, sh, stream)
                             : launch_pipe<F32, MODE, kPipeVplTarget>(P, sh, stream);
  }
  if (sh.rows != 2) return cudaErrorInvalidValue;
  return dt == SPEC_BF16 ? launch_pipe<Bf16, MODE, kPipeVpl>(P, sh, stream)
                         : launch_pipe<F32, MODE, kPipeVpl>(P, sh, stream);
}

// Fills the shape fields of a two-pass launch.
void pipe_geometry(ssv::PipeParams* P, const PShape& sh) {
  P->S = sh.S;
  P->G = sh.G;
  P->NV = sh.NV;
  P->CV = sh.CV;
  P->NCH = sh.NCH;
  P->WV = sh.WV;
  P->NS = sh.NS;
  P->rows = sh.rows;
}

// The two-pass sweep serves rows that start on 16-byte boundaries.
// The automatic choice takes the two-pass sweep for calls that stream at
// least this many bytes of logits.  Below it the single-read sweep, whose
// clusters hold a unit's rows in shared memory for one read, finishes first
// (measured on GB300: at 175 MB, B=64, K=4, V=151936, single-read 67.5 µs
// against 78.0; at 248 MB, B=64, K=7, V=129280, two-pass 79.8 against 92.1).
constexpr double kPipeMinBytes = 200.0e6;

bool pipe_allowed(const void* a, const void* b, int V, int es, long long rows_read) {
  const int ov = g_kernel_override.load();
  if (ov == 1) return false;
  if (ov != 2 && (double)rows_read * (double)V * (double)es < kPipeMinBytes) return false;
  return ((long long)V * es) % 16 == 0 && (reinterpret_cast<uintptr_t>(a) & 15u) == 0 &&
         (b == nullptr || (reinterpret_cast<uintptr_t>(b) & 15u) == 0);
}

// Workspace layouts (all offsets 256-byte aligned).
size_t part_bytes(long long units) { return align256((size_t)units * ssv::kPartStride * sizeof(float)); }

struct VerifyWs {
  size_t rec = 0, part = 0, cnt = 0, rej = 0, dtot = 0, dcnt = 0, total = 0;
};
VerifyWs verify_ws(int B, int K) {
  const long long units = (long long)B * (K + 1);
  VerifyWs w;
  w.rec = 0;
  w.part = align256((size_t)units * sizeof(VerifyRecord));
  w.cnt = w.part + part_bytes(units);
  w.rej = w.cnt + align256((size_t)B * sizeof(uint32_t));
  w.dtot = w.rej + align256((size_t)B * sizeof(uint32_t));
  w.dcnt = w.dtot + align256((size_t)units * ssv::kPSegs * sizeof(float));
  w.total = w.dcnt + align256((size_t)units * sizeof(uint32_t));
  return w;
}
struct OverlapWs {
  size_t part = 0, cnt = 0, total = 0;
};
OverlapWs overlap_ws(int B, int K) {
  OverlapWs w;
  w.part = 0;
  w.cnt = part_bytes((long long)B * K);
  w.total = w.cnt + align256((size_t)B * sizeof(uint32_t));
  return w;
}
struct E2EWs {
  size_t stats = 0, part = 0, part2 = 0, row_loss = 0, cnt = 0, glob = 0, total = 0;
};
E2EWs e2e_ws(int B, int K) {
  const long long units = (long long)B * K;
  E2EWs w;
  w.stats = 0;
  w.part = align256((size_t)units * sizeof(E2EStats));
  w.part2 = w.part + part_bytes(units);
  w.row_loss = w.part2 + part_bytes(units);
  w.cnt = w.row_loss + align256((size_t)B * sizeof(float));
  w.glob = w.cnt + align256((size_t)B * sizeof(uint32_t));
  w.total = w.glob + 256;
  return w;
}

struct DiagWs {
  size_t part = 0, part2 = 0, part3 = 0, cnt = 0, total = 0;
};
DiagWs diag_ws(int B, int K) {
  const long long units = (long long)B * K;
  DiagWs w;
  w.part = 0;
  w.part2 = part_bytes(units);
  w.part3 = w.part2 + part_bytes(units);
  w.cnt = w.part3 + part_bytes(units);
  w.total = w.cnt + align256((size_t)B * sizeof(uint32_t));
  return w;
}

// Ragged verify workspace: records and partials per unit, row counters and
// row words, then the unit entries {flattened row, packed word} and the
// offsets-rejected flag.
struct RaggedWs {
  size_t rec = 0, part = 0, cnt = 0, rej = 0, uinfo = 0, bad = 0, total = 0;
};
RaggedWs ragged_ws(int B, long long units) {
  RaggedWs w;
  w.rec = 0;
  w.part = align256((size_t)units * sizeof(VerifyRecord));
  w.cnt = w.part + part_bytes(units);
  w.rej = w.cnt + align256((size_t)B * sizeof(uint32_t));
  w.uinfo = w.rej + align256((size_t)B * sizeof(uint32_t));
  w.bad = w.uinfo + align256((size_t)units * sizeof(uint2));
  w.total = w.bad + 256;
  return w;
}

// One thread per row: checks the row's offsets and writes its units' entries
// {flattened target row, packed word}; any bad row sets the flag that makes
// the sweep return at once.
__global__ void ragged_units_kernel(const int32_t* roff, int B, int units, uint2* uinfo, uint32_t* bad,
                                    uint32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int s0 = roff[b], s1 = roff[b + 1];
  const int l = s1 - s0 - 1;
  const int d0 = s0 - b;  // drafted positions of the rows before b (valid offsets)
  const bool ok = s0 >= 0 && s1 > s0 && l <= kMaxK && s1 <= units && (b > 0 || s0 == 0) &&
                  (b < B - 1 || s1 == units) && d0 >= 0 && d0 + l <= units - B;
  if (!ok) {
    atomicOr(bad, 1u);
    if (status) atomicOr(status, SPEC_DEV_BAD_OFFSETS);
    return;
  }
  // drafted positions first, in flattened order, then every row's bonus: the
  // last units read the target only and usually skip their draw
  for (int k = 0; k < l; ++k)
    uinfo[d0 + k] = make_uint2((uint32_t)(s0 + k), ssv::pack_unit((uint32_t)b, (uint32_t)k, false));
  uinfo[units - B + b] = make_uint2((uint32_t)(s0 + l), ssv::pack_unit((uint32_t)b, (uint32_t)l, true));
}

bool dims_ok(int B, int K, int V) { return B >= 0 && K >= 0 && K <= kMaxK && V >= 1; }

bool dtype_ok(spec_dtype_t dt) { return dt == SPEC_F32 || dt == SPEC_BF16; }

// One warp waits on a fresh mbarrier that nothing arrives at: phase 0 never
// completes, so the bounded wait runs out and reports it.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = ssv::smem_addr(&bar);
  if (threadIdx.x == 0) ssv::mbar_init(a, 1u);
  __syncthreads();
  const bool done = ssv::mbar_wait_bounded(a, 0u, limit_ns);
  if (!done && threadIdx.x == 0) atomicOr(status, ssv::kTimeout);
}

}  // namespace

extern "C" {

int spec_abi_version(void) { return 2; }

unsigned long long spec_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

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

void spec_set_launch_override(int cluster_ctas, int stages) {
  g_cluster_override.store(cluster_ctas > 0 && cluster_ctas <= kMaxCluster ? cluster_ctas : 0);
  g_stage_override.store(stages == 1 || stages == 2 ? stages : 0);
}

void spec_set_kernel_override(int kernel) { g_kernel_override.store(kernel == 1 || kernel == 2 ? kernel : 0); }

spec_status_t spec_launch_shape(spec_dtype_t dtype, int units, int V, int* cluster_ctas, int* threads,
                                int* smem_bytes, int* clusters, int* stages) {
  if (!dtype_ok(dtype) || units < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  const int ov = g_kernel_override.load();
  const bool big = (double)units * 2.0 * (double)V * (double)elem_size(dtype) >= kPipeMinBytes;  // ~2 rows per unit
  if (ov != 1 && (ov == 2 || big) && ((long long)V * elem_size(dtype)) % 16 == 0) {
    PShape ps;
    const spec_status_t r = pipe_shape_dt<ssv::kPSample>(dtype, units, V, 2, &ps);
    if (r == SPEC_ERR_CUDA) return r;
    if (r == SPEC_OK) {
      if (cluster_ctas) *cluster_ctas = ps.S;
      if (threads) *threads = ssv::kPThreads;
      if (smem_bytes) *smem_bytes = ps.smem;
      if (clusters) *clusters = ps.G;
      if (stages) *stages = ps.NS;
      return SPEC_OK;
    }
  }
  Shape sh;
  const spec_status_t r = shape_for_dt<ssv::kVerify>(dtype, units, V, 2, &sh);
  if (r != SPEC_OK) return r;
  if (cluster_ctas) *cluster_ctas = sh.S;
  if (threads) *threads = ssv::kThreads;
  if (smem_bytes) *smem_bytes = sh.smem;
  if (clusters) *clusters = sh.G;
  if (stages) *stages = sh.nst;
  return SPEC_OK;
}

size_t spec_verify_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return verify_ws(B, K).total;
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
  const VerifyWs ws = verify_ws(B, K);
  if (workspace_bytes < ws.total || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * (K + 1);
  if (units > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  const int rows = (greedy && !alpha_out) ? 1 : 2;  // greedy without overlap reads no draft row
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pipe_allowed(target_logits, rows == 2 ? draft_logits : nullptr, V, es,
                   (long long)B * (K + 1) + (rows == 2 ? (long long)B * K : 0))) {
    PShape ps;
    const spec_status_t r = greedy ? pipe_shape_dt<ssv::kPGreedy>(dtype, units, V, rows, &ps)
                                   : pipe_shape_dt<ssv::kPSample>(dtype, units, V, rows, &ps);
    if (r == SPEC_ERR_CUDA) return r;
    if (r == SPEC_OK) {
      ssv::PipeParams P = {};
      P.target = target_logits;
      P.draft = draft_logits;
      P.B = B;
      P.K = K;
      P.KT = K + 1;
      P.V = V;
      P.units = (int)units;
      pipe_geometry(&P, ps);
      P.grouped = (!greedy && B >= ps.G) ? 1 : 0;
      P.s = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
      P.inv_t = greedy ? 0.0f : (float)(1.0 / (double)temperature);
      P.draft_tokens = draft_tokens;
      P.u_accept = u_accept;
      P.u_final = u_final;
      P.out_tokens = out_tokens;
      P.n_accepted = n_accepted;
      P.alpha = alpha_out;
      char* w = static_cast<char*>(workspace);
      P.rec = reinterpret_cast<VerifyRecord*>(w + ws.rec);
      P.part = reinterpret_cast<float*>(w + ws.part);
      P.row_cnt = reinterpret_cast<uint32_t*>(w + ws.cnt);
      P.rej = reinterpret_cast<uint32_t*>(w + ws.rej);
      P.dtot = reinterpret_cast<float*>(w + ws.dtot);
      P.dcnt = reinterpret_cast<uint32_t*>(w + ws.dcnt);
      P.status = dev_status;
      return from_cuda(greedy ? launch_pipe_dt<ssv::kPGreedy>(dtype, P, ps, st)
                              : launch_pipe_dt<ssv::kPSample>(dtype, P, ps, st));
    }
  }
  Shape sh;
  {
    // both sampling orders share one launch shape
    const spec_status_t r = greedy ? shape_for_dt<ssv::kVerifyGreedy>(dtype, units, V, rows, &sh)
                                   : shape_for_dt<ssv::kVerify>(dtype, units, V, rows, &sh);
    if (r != SPEC_OK) return r;
  }

  SweepParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = K + 1;
  P.V = V;
  P.units = (int)units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 2;
  P.aligned = aligned16(target_logits) && (!draft_logits || aligned16(draft_logits)) && ((long long)V * es) % 16 == 0;
  P.s = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = greedy ? 0.0f : (float)(1.0 / (double)temperature);
  P.rows = rows;
  P.draft_tokens = draft_tokens;
  P.u_accept = u_accept;
  P.u_final = u_final;
  P.out_tokens = out_tokens;
  P.n_accepted = n_accepted;
  P.alpha = alpha_out;
  P.rec = reinterpret_cast<VerifyRecord*>(static_cast<char*>(workspace) + ws.rec);
  P.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.part);
  P.row_cnt = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws.cnt);
  P.rej = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws.rej);
  P.status = dev_status;
  // At least one row per cluster: rows in groups, position-major (later
  // positions can skip draws that an earlier rejection makes unused).
  // Fewer rows: row-major order, which measured faster there.
  cudaError_t e;
  if (greedy) {
    e = launch_sweep_dt<ssv::kVerifyGreedy>(dtype, P, sh, st);
  } else if (B >= sh.G) {
    e = prepare_dt<ssv::kVerifyGrouped>(dtype);
    if (e == cudaSuccess) e = launch_sweep_dt<ssv::kVerifyGrouped>(dtype, P, sh, st);
  } else {
    e = launch_sweep_dt<ssv::kVerify>(dtype, P, sh, st);
  }
  return from_cuda(e);
}

size_t spec_overlap_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return overlap_ws(B, K).total;
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
  const OverlapWs ws = overlap_ws(B, K);
  if (!workspace || workspace_bytes < ws.total || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * K;
  if (units > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  const bool greedy = temperature == 0.0f;
  if (!greedy && pipe_allowed(target_logits, draft_logits, V, es, 2 * units)) {
    PShape ps;
    const spec_status_t r = pipe_shape_dt<ssv::kPOverlap>(dtype, units, V, 2, &ps);
    if (r == SPEC_ERR_CUDA) return r;
    if (r == SPEC_OK) {
      ssv::PipeParams P = {};
      P.target = target_logits;
      P.draft = draft_logits;
      P.B = B;
      P.K = K;
      P.KT = KT;
      P.V = V;
      P.units = (int)units;
      pipe_geometry(&P, ps);
      P.s = (float)(1.4426950408889634 / (double)temperature);
      P.inv_t = (float)(1.0 / (double)temperature);
      P.alpha = alpha;
      P.tv = tv;
      P.surv = prefix_survival;
      P.exp_acc = expected_accepted;
      P.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.part);
      P.row_cnt = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws.cnt);
      P.status = dev_status;
      return from_cuda(launch_pipe_dt<ssv::kPOverlap>(dtype, P, ps, st));
    }
  }
  Shape sh;
  {
    const spec_status_t r = greedy ? shape_for_dt<ssv::kOverlapGreedy>(dtype, units, V, 2, &sh)
                                   : shape_for_dt<ssv::kOverlap>(dtype, units, V, 2, &sh);
    if (r != SPEC_OK) return r;
  }
  SweepParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = KT;
  P.V = V;
  P.units = (int)units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 2;
  P.aligned = aligned16(target_logits) && aligned16(draft_logits) && ((long long)V * es) % 16 == 0;
  P.s = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = greedy ? 0.0f : (float)(1.0 / (double)temperature);
  P.alpha = alpha;
  P.tv = tv;
  P.surv = prefix_survival;
  P.exp_acc = expected_accepted;
  P.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.part);
  P.row_cnt = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws.cnt);
  P.status = dev_status;
  cudaError_t e = greedy ? launch_sweep_dt<ssv::kOverlapGreedy>(dtype, P, sh, st)
                         : launch_sweep_dt<ssv::kOverlap>(dtype, P, sh, st);
  return from_cuda(e);
}

size_t spec_e2e_tv_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return e2e_ws(B, K).total;
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
  const E2EWs ws = e2e_ws(B, K);
  if (workspace_bytes < ws.total || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * K;
  if (units > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  char* w = static_cast<char*>(workspace);
  const bool aligned = aligned16(target_logits) && aligned16(draft_logits) && ((long long)V * es) % 16 == 0;
  cudaError_t e = cudaSuccess;
  bool launched = false;
  if (pipe_allowed(target_logits, draft_logits, V, es, 2 * units)) {
    PShape ps;
    const spec_status_t r = pipe_shape_dt<ssv::kPE2E>(dtype, units, V, 2, &ps);
    if (r == SPEC_ERR_CUDA) return r;
    if (r == SPEC_OK) {
      ssv::PipeParams Q = {};
      Q.target = target_logits;
      Q.draft = draft_logits;
      Q.B = B;
      Q.K = K;
      Q.KT = KT;
      Q.V = V;
      Q.units = (int)units;
      pipe_geometry(&Q, ps);
      Q.s = (float)(1.4426950408889634 / (double)temperature);
      Q.inv_t = (float)(1.0 / (double)temperature);
      Q.grad_scale = grad_scale;
      Q.alpha = alpha_out;
      Q.loss = loss_out;
      Q.stats = reinterpret_cast<E2EStats*>(w + ws.stats);
      Q.part = reinterpret_cast<float*>(w + ws.part);
      Q.part2 = reinterpret_cast<float*>(w + ws.part2);
      Q.row_loss = reinterpret_cast<float*>(w + ws.row_loss);
      Q.row_cnt = reinterpret_cast<uint32_t*>(w + ws.cnt);
      Q.glob_cnt = reinterpret_cast<uint32_t*>(w + ws.glob);
      Q.status = dev_status;
      e = launch_pipe_dt<ssv::kPE2E>(dtype, Q, ps, st);
      if (e != cudaSuccess) return SPEC_ERR_CUDA;
      launched = true;
    }
  }
  Shape sh;
  if (!launched) {
    const spec_status_t r = shape_for_dt<ssv::kE2E>(dtype, units, V, 2, &sh);
    if (r != SPEC_OK) return r;
  }
  SweepParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = KT;
  P.V = V;
  P.units = (int)units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 2;
  P.aligned = aligned;
  P.s = (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = (float)(1.0 / (double)temperature);
  P.grad_scale = grad_scale;
  P.alpha = alpha_out;
  P.loss = loss_out;
  P.stats = reinterpret_cast<E2EStats*>(w + ws.stats);
  P.part = reinterpret_cast<float*>(w + ws.part);
  P.part2 = reinterpret_cast<float*>(w + ws.part2);
  P.row_loss = reinterpret_cast<float*>(w + ws.row_loss);
  P.row_cnt = reinterpret_cast<uint32_t*>(w + ws.cnt);
  P.glob_cnt = reinterpret_cast<uint32_t*>(w + ws.glob);
  P.status = dev_status;
  if (!launched) {
    e = launch_sweep_dt<ssv::kE2E>(dtype, P, sh, st);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
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
  return from_cuda(cudaMemsetAsync(w + ws.stats, 0, (size_t)B * K * sizeof(E2EStats), st));
}

size_t spec_diagnostics_workspace_bytes(int B, int K, int V) {
  if (!dims_ok(B, K, V)) return 0;
  return diag_ws(B, K).total;
}

spec_status_t spec_diagnostics(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B, int K,
                               int KT, int V, float temperature, float* alpha, float* entropy, float* cross_entropy,
                               float* kl, float* alpha_target_only, uint32_t* dev_status, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!dims_ok(B, K, V) || !dtype_ok(dtype) || KT < K) return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  if (B == 0 || K == 0) return SPEC_OK;
  if (!target_logits || !draft_logits) return SPEC_ERR_INVALID_ARG;
  const DiagWs ws = diag_ws(B, K);
  if (!workspace || workspace_bytes < ws.total || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * K;
  if (units > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  Shape sh;
  {
    const spec_status_t r = shape_for_dt<ssv::kDiag>(dtype, units, V, 2, &sh);
    if (r != SPEC_OK) return r;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SweepParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = KT;
  P.V = V;
  P.units = (int)units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 2;
  P.aligned = aligned16(target_logits) && aligned16(draft_logits) && ((long long)V * es) % 16 == 0;
  P.s = (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = (float)(1.0 / (double)temperature);
  P.alpha = alpha;
  P.ent = entropy;
  P.ce = cross_entropy;
  P.kl = kl;
  P.ato = alpha_target_only;
  char* w = static_cast<char*>(workspace);
  P.part = reinterpret_cast<float*>(w + ws.part);
  P.part2 = reinterpret_cast<float*>(w + ws.part2);
  P.part3 = reinterpret_cast<float*>(w + ws.part3);
  P.row_cnt = reinterpret_cast<uint32_t*>(w + ws.cnt);
  P.status = dev_status;
  return from_cuda(launch_sweep_dt<ssv::kDiag>(dtype, P, sh, st));
}

spec_status_t spec_truncate_logits(const void* logits, void* out, spec_dtype_t dtype, int rows, int V,
                                   float temperature, int top_k, float top_p, uint32_t* dev_status, void* stream) {
  if (rows < 0 || V < 1 || !dtype_ok(dtype) || top_k < 0) return SPEC_ERR_INVALID_ARG;
  if (!(top_p > 0.0f && top_p <= 1.0f)) return SPEC_ERR_INVALID_ARG;
  if (top_p < 1.0f && (!(temperature > 0.0f) || !std::isfinite(temperature))) return SPEC_ERR_INVALID_ARG;
  if (rows == 0) return SPEC_OK;
  if (!logits || !out) return SPEC_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const size_t bytes = (size_t)rows * (size_t)V * (size_t)es;
  const uintptr_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(out);
  if (a != b && a < b + bytes && b < a + bytes) return SPEC_ERR_INVALID_ARG;  // partial overlap
  DevInfo di;
  if (!device_info(&di)) return SPEC_ERR_CUDA;
  ssv::TruncParams P = {};
  P.in = logits;
  P.out = out;
  P.rows = rows;
  P.V = V;
  P.aligned = aligned16(logits) && aligned16(out) && ((long long)V * es) % 16 == 0;
  P.s = top_p < 1.0f ? (float)(1.4426950408889634 / (double)temperature) : 0.0f;
  P.top_k = top_k;
  P.top_p = top_p;
  P.status = dev_status;
  const int grid = rows < 2 * di.sms ? rows : 2 * di.sms;  // two resident CTAs per SM
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  const int which = dtype == SPEC_BF16 ? 1 : 0;
  if (top_k > 0 && top_k < V && top_k <= ssv::kKMax) {
    // a small top-k (with or without top-p over it): candidate filtering
    const int smem = (int)sizeof(ssv::TopkSmem);
    static std::atomic<uint64_t> prepared_k[2];
    if (!(prepared_k[which].load(std::memory_order_acquire) & bit)) {
      const cudaError_t e =
          dtype == SPEC_BF16
              ? cudaFuncSetAttribute(ssv::topk_kernel<Bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
              : cudaFuncSetAttribute(ssv::topk_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return SPEC_ERR_CUDA;
      prepared_k[which].fetch_or(bit, std::memory_order_release);
    }
    if (dtype == SPEC_BF16)
      ssv::topk_kernel<Bf16><<<grid, ssv::kTThreads, smem, st>>>(P);
    else
      ssv::topk_kernel<F32><<<grid, ssv::kTThreads, smem, st>>>(P);
    return from_cuda(counted(cudaGetLastError()));
  }
  const int smem = (int)sizeof(ssv::TruncSmem);
  static std::atomic<uint64_t> prepared[2];
  if (!(prepared[which].load(std::memory_order_acquire) & bit)) {
    const cudaError_t e = dtype == SPEC_BF16
                              ? cudaFuncSetAttribute(ssv::truncate_kernel<Bf16>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                              : cudaFuncSetAttribute(ssv::truncate_kernel<F32>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    prepared[which].fetch_or(bit, std::memory_order_release);
  }
  if (dtype == SPEC_BF16)
    ssv::truncate_kernel<Bf16><<<grid, ssv::kTThreads, smem, st>>>(P);
  else
    ssv::truncate_kernel<F32><<<grid, ssv::kTThreads, smem, st>>>(P);
  return from_cuda(counted(cudaGetLastError()));
}

spec_status_t spec_selftest_bounded_wait(uint64_t limit_ns, uint32_t* dev_status, void* stream) {
  if (!dev_status || limit_ns == 0 || limit_ns > 10000000000ull) return SPEC_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, dev_status);
  return from_cuda(counted(cudaGetLastError()));
}

spec_status_t spec_schedule_lengths(const float* survival, int R, int L, const float* sps, int sps_len,
                                    int32_t* lengths, float* objective, uint32_t* dev_status, void* stream) {
  if (R < 0 || L < 1 || L > kMaxK || sps_len < 0) return SPEC_ERR_INVALID_ARG;
  if (R == 0) return SPEC_OK;
  if ((long long)sps_len < (long long)R * (1 + L) + 1) return SPEC_ERR_INVALID_ARG;
  if (!survival || !sps || !lengths) return SPEC_ERR_INVALID_ARG;
  if ((long long)R * L > ssv::kSchedMaxItems || L > ssv::kSchedMaxL) return SPEC_ERR_UNSUPPORTED;
  const size_t smem = sizeof(ssv::SchedSmem);
  static std::atomic<uint64_t> prepared{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(prepared.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(ssv::schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ssv::schedule_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    prepared.fetch_or(bit, std::memory_order_release);
  }
  ssv::SchedParams P = {};
  P.surv = survival;
  P.R = R;
  P.L = L;
  P.sps = sps;
  P.nsps = sps_len;
  P.lengths = lengths;
  P.objective = objective;
  P.status = dev_status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ssv::kSCtas, 1, 1);
  cfg.blockDim = dim3(ssv::kSThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ssv::kSCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return from_cuda(counted(cudaLaunchKernelEx(&cfg, ssv::schedule_kernel, P)));
}

size_t spec_verify_ragged_workspace_bytes(int B, int units, int V) {
  if (B < 0 || units < B || V < 1) return 0;
  return ragged_ws(B, units).total;
}

spec_status_t spec_verify_ragged(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B,
                                 const int32_t* row_offsets, int units, int V, float temperature,
                                 const int32_t* draft_tokens, const float* u_accept, const float* u_final,
                                 int32_t* out_tokens, int32_t* n_accepted, float* alpha_out, uint32_t* dev_status,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || units < B || V < 1 || !dtype_ok(dtype)) return SPEC_ERR_INVALID_ARG;
  if ((long long)units > (long long)B * (kMaxK + 1)) return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !row_offsets || !u_final || !out_tokens || !n_accepted || !workspace)
    return SPEC_ERR_INVALID_ARG;
  const bool drafted = units > B;
  if (drafted && (!draft_logits || !draft_tokens || !u_accept)) return SPEC_ERR_INVALID_ARG;
  const RaggedWs ws = ragged_ws(B, units);
  if (workspace_bytes < ws.total || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  Shape sh;
  {
    const spec_status_t r = shape_for_dt<ssv::kVerify>(dtype, units, V, 2, &sh);
    if (r != SPEC_OK) return r;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(workspace);
  uint2* uinfo = reinterpret_cast<uint2*>(w + ws.uinfo);
  uint32_t* bad = reinterpret_cast<uint32_t*>(w + ws.bad);
  ragged_units_kernel<<<(B + 255) / 256, 256, 0, st>>>(row_offsets, B, units, uinfo, bad, dev_status);
  cudaError_t e = counted(cudaGetLastError());
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  SweepParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = kMaxK;
  P.KT = kMaxK + 1;
  P.V = V;
  P.units = units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 2;
  P.aligned = aligned16(target_logits) && (!draft_logits || aligned16(draft_logits)) && ((long long)V * es) % 16 == 0;
  P.s = (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = (float)(1.0 / (double)temperature);
  P.draft_tokens = draft_tokens;
  P.u_accept = u_accept;
  P.u_final = u_final;
  P.out_tokens = out_tokens;
  P.n_accepted = n_accepted;
  P.alpha = alpha_out;
  P.rec = reinterpret_cast<VerifyRecord*>(w + ws.rec);
  P.part = reinterpret_cast<float*>(w + ws.part);
  P.row_cnt = reinterpret_cast<uint32_t*>(w + ws.cnt);
  P.rej = reinterpret_cast<uint32_t*>(w + ws.rej);
  P.uinfo = uinfo;
  P.roff = row_offsets;
  P.ragbad = bad;
  P.status = dev_status;
  e = prepare_dt<ssv::kVerifyRagged>(dtype);
  if (e == cudaSuccess) e = launch_sweep_dt<ssv::kVerifyRagged>(dtype, P, sh, st);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  // the unit words and the flag are the only parts not left zero by the sweep
  e = cudaMemsetAsync(w + ws.uinfo, 0, ws.total - ws.uinfo, st);
  return from_cuda(e);
}

spec_status_t spec_verify_relaxed(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B,
                                  int K, int V, float temperature, int top_k, float delta,
                                  const int32_t* draft_tokens, const float* u_final, int32_t* out_tokens,
                                  int32_t* n_accepted, float* alpha_out, uint32_t* dev_status, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!dims_ok(B, K, V) || !dtype_ok(dtype)) return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature) || !(delta >= 0.0f)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !u_final || !out_tokens || !n_accepted || !workspace) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && (!draft_logits || !draft_tokens)) return SPEC_ERR_INVALID_ARG;
  const VerifyWs ws = verify_ws(B, K);
  if (workspace_bytes < ws.total || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * (K + 1);
  if (units > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  Shape sh;
  {
    const spec_status_t r = shape_for_dt<ssv::kVerify>(dtype, units, V, 2, &sh);
    if (r != SPEC_OK) return r;
  }
  SweepParams P = {};
  P.target = target_logits;
  P.draft = draft_logits;
  P.B = B;
  P.K = K;
  P.KT = K + 1;
  P.V = V;
  P.units = (int)units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 2;
  P.aligned = aligned16(target_logits) && (!draft_logits || aligned16(draft_logits)) && ((long long)V * es) % 16 == 0;
  P.s = (float)(1.4426950408889634 / (double)temperature);
  P.inv_t = (float)(1.0 / (double)temperature);
  P.relax_k = top_k;
  P.relax_delta = delta;
  P.draft_tokens = draft_tokens;
  P.u_final = u_final;
  P.out_tokens = out_tokens;
  P.n_accepted = n_accepted;
  P.alpha = alpha_out;
  char* w = static_cast<char*>(workspace);
  P.rec = reinterpret_cast<VerifyRecord*>(w + ws.rec);
  P.part = reinterpret_cast<float*>(w + ws.part);
  P.row_cnt = reinterpret_cast<uint32_t*>(w + ws.cnt);
  P.rej = reinterpret_cast<uint32_t*>(w + ws.rej);
  P.status = dev_status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = prepare_dt<ssv::kVerifyRelaxed>(dtype);
  if (e == cudaSuccess) e = launch_sweep_dt<ssv::kVerifyRelaxed>(dtype, P, sh, st);
  return from_cuda(e);
}

spec_status_t spec_tree_mask(const int32_t* parent, int B, int N, uint8_t* mask, int32_t* depth,
                             uint32_t* dev_status, void* stream) {
  if (B < 0 || N < 0) return SPEC_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return SPEC_OK;
  if (!parent || !mask) return SPEC_ERR_INVALID_ARG;
  const long long n = (long long)B * N;
  if (n * N > (1ll << 40)) return SPEC_ERR_UNSUPPORTED;
  const unsigned grid = (unsigned)((n + 255) / 256);
  ssv::tree_mask_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(parent, B, N, mask, depth,
                                                                             dev_status);
  return from_cuda(counted(cudaGetLastError()));
}

size_t spec_tree_verify_workspace_bytes(int B, int N, int V) {
  if (B < 0 || N < 0 || V < 1) return 0;
  return align256((size_t)B * (N + 1) * sizeof(int32_t));
}

spec_status_t spec_tree_verify_greedy(const void* target_logits, spec_dtype_t dtype, int B, int N, int V,
                                      const int32_t* parent, const int32_t* node_tokens, int32_t* path,
                                      int32_t* out_tokens, int32_t* n_accepted, uint32_t* dev_status,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || N < 0 || V < 1 || !dtype_ok(dtype)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !out_tokens || !n_accepted || !workspace) return SPEC_ERR_INVALID_ARG;
  if (N > 0 && (!parent || !node_tokens || !path)) return SPEC_ERR_INVALID_ARG;
  if (workspace_bytes < spec_tree_verify_workspace_bytes(B, N, V) || !aligned16(workspace))
    return SPEC_ERR_INVALID_ARG;
  const long long units = (long long)B * (N + 1);
  if (units > 0x7FFFFFFFLL) return SPEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  Shape sh;
  {
    const spec_status_t r = shape_for_dt<ssv::kVerifyGreedy>(dtype, units, V, 1, &sh);
    if (r != SPEC_OK) return r;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* am = static_cast<int32_t*>(workspace);  // target argmax of every slot
  SweepParams P = {};
  P.target = target_logits;
  P.B = B;
  P.K = N + 1;
  P.KT = N + 1;
  P.V = V;
  P.units = (int)units;
  P.S = sh.S;
  P.L = sh.L;
  P.nst = sh.nst;
  P.rows = 1;
  P.aligned = aligned16(target_logits) && ((long long)V * es) % 16 == 0;
  P.out_tokens = am;
  P.status = dev_status;
  cudaError_t e = prepare_dt<ssv::kArgmax>(dtype);
  if (e == cudaSuccess) e = launch_sweep_dt<ssv::kArgmax>(dtype, P, sh, st);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  ssv::tree_walk_kernel<<<(B + 127) / 128, 128, 0, st>>>(am, parent, node_tokens, B, N, path, out_tokens,
                                                          n_accepted, dev_status);
  e = counted(cudaGetLastError());
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  // the argmax array is the only workspace written: leave it zero
  return from_cuda(cudaMemsetAsync(am, 0, (size_t)units * sizeof(int32_t), st));
}

}  // extern "C"
