// m2rnn_noalloc.cu — m2rnn_backward_bf16_noalloc: the bf16 backward pass with its
// workspace taken from a fixed scratch array that lives in the module, so the caller
// passes no workspace at all.
//
// The M²RNN notes have no counterpart to this entry point: it is a library
// convenience for callers that cannot hand over device memory (it computes exactly
// what m2rnn_backward_bf16 computes, with the same kernels).
//
// Limits and hazards:
//  * The scratch holds kNoAllocScratchFloats floats (16 MiB).  Shapes whose
//    workspace is larger are rejected with M2RNN_ERR_UNSUPPORTED before anything is
//    enqueued; nothing is ever allocated.
//  * One scratch array exists per device and every call on that device uses it.
//    Two calls whose work overlaps in time (different streams, or several host
//    threads, with no ordering between them) race on it and give wrong results;
//    calls must be ordered (one stream, or events).
//  * The first call on a device resolves the scratch address with
//    cudaGetSymbolAddress (under a mutex) and caches it for the current CUDA context.
//    That call may load the module, which is not allowed while a stream is being
//    captured: make one call on each device before capturing it into a CUDA graph.
//    A later call under another context (after cudaDeviceReset, say, which ends the
//    context and unloads the module) resolves the address again instead of handing the
//    kernels a stale one; that call, too, must come before any capture.
#include <mutex>

#include "../../include/m2rnn.h"
#include "m2rnn_internal.h"

namespace m2rnn {
namespace {

constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;  // 16 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;

// Device address of this device's scratch array, cached per CUDA context: a new context
// on the device (the module reloaded, possibly at another address) is resolved again.
float* scratch_address(int dev) {
  struct Entry {
    unsigned long long ctx;
    float* addr;
  };
  static Entry cache[kMaxDevices] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (have_id && cache[dev].addr && cache[dev].ctx == id) return cache[dev].addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
  if (have_id || current_context_id(&id)) cache[dev] = Entry{id, static_cast<float*>(p)};
  return static_cast<float*>(p);
}

}  // namespace
}  // namespace m2rnn

using namespace m2rnn;

extern "C" m2rnn_status m2rnn_backward_bf16_noalloc(
    const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* a, const float* alpha,
    const float* beta, const uint16_t* W, const float* w_r, const float* H0, const uint16_t* Hs,
    const float* dy, const float* dH_T, float* dq, float* dk, float* dv, float* da, float* dalpha,
    float* dbeta, float* dW, float* dw_r, float* dH0, int B, int T, int N, int Nqk, int K, int V,
    void* stream) {
  // Size checks first: an oversized request is refused before the device is touched.
  if (B < 1 || N < 1 || K < 1 || V < 1 || T < 0 || (Nqk != 1 && Nqk != N))
    return M2RNN_ERR_INVALID_ARG;
  if (K > 128 || V > 128 || (long long)B * N > 0x7fffffffLL) return M2RNN_ERR_UNSUPPORTED;
  const size_t need = backward_workspace_floats(B, T, N, Nqk, K, V);
  if (need > kNoAllocScratchFloats) return M2RNN_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  float* ws = scratch_address(dev);
  if (!ws) return M2RNN_ERR_CUDA;
  return m2rnn_backward_bf16(q, k, v, a, alpha, beta, W, w_r, H0, Hs, dy, dH_T, dq, dk, dv, da,
                             dalpha, dbeta, dW, dw_r, dH0, B, T, N, Nqk, K, V, 0, ws,
                             need * sizeof(float), stream);
}
