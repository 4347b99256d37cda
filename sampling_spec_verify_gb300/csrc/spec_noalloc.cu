// Allocation-free variant of spec_verify.
//
// Some callers cannot allocate device memory at the point where they need a
// verify step: runtimes that hand every byte of device memory to their own
// pool at start-up and forbid raw allocations afterwards, plugin hosts that
// give a plugin its input and output buffers but no allocator, and
// latency-critical decode loops that cannot take the implicit device-wide
// synchronisation of cudaMalloc / cudaFree.  spec_verify_noalloc serves them:
// it takes the same inputs and outputs as spec_verify but no workspace; its
// scratch space is the fixed-size device array below, which every GPU that
// loads this library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "spec_verify.h"

namespace {

// Scratch of the allocation-free entry point (arrival counters and per-position
// records of spec_verify).  Shared by every call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];  // null until a lookup on that device succeeds
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in: a kernel must be given this address instead.
// Looked up with that device current; only a successful lookup is kept, so a
// failed one (which also clears the error it left pending) is retried on the
// next call.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> g(g_scratch_mu);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
      }
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" spec_status_t spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                             spec_dtype_t dtype, int B, int K, int V, float temperature,
                                             const int32_t* draft_tokens, const float* u_accept,
                                             const float* u_final, int32_t* out_tokens, int32_t* n_accepted,
                                             float* alpha_out, uint32_t* dev_status, void* stream) {
  const size_t need = spec_verify_workspace_bytes(B, K, V);
  // An empty batch, or dimensions spec_verify rejects: nothing needs scratch,
  // and spec_verify gives the same answer it gives any caller (its argument
  // checks, then SPEC_OK for B == 0).
  if (B <= 0 || need == 0)
    return spec_verify(target_logits, draft_logits, dtype, B, K, V, temperature, draft_tokens, u_accept, u_final,
                       out_tokens, n_accepted, alpha_out, dev_status, nullptr, 0, stream);
  if (need > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SPEC_ERR_CUDA;
  // The array keeps whatever the previous call left; the counters must start
  // at zero, so clear the part this call uses (on the caller's stream).
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, need, st) != cudaSuccess) return SPEC_ERR_CUDA;
  return spec_verify(target_logits, draft_logits, dtype, B, K, V, temperature, draft_tokens, u_accept, u_final,
                     out_tokens, n_accepted, alpha_out, dev_status, scratch, need, stream);
}
