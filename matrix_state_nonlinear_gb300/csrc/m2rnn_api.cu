// m2rnn_api.cu — host layer behind include/m2rnn.h: argument validation, variant
// choice, the per-device status word, and the launches.  All arithmetic of the
// recurrence runs in the kernels of the other translation units.
#include <mutex>

#include "../../include/m2rnn.h"
#include "m2rnn_internal.h"

namespace m2rnn {

// One status word per device (every device that loads the module holds its copy).
__device__ int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;

// Device address of this device's status word, cached per CUDA context (see
// current_context_id).
int* status_address(int dev) {
  struct Entry {
    unsigned long long ctx;
    int* addr;
  };
  static Entry cache[kMaxDevices] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (have_id && cache[dev].addr && cache[dev].ctx == id) return cache[dev].addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  if (have_id || current_context_id(&id)) cache[dev] = Entry{id, static_cast<int*>(p)};
  return static_cast<int*>(p);
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

enum Variant : int {
  kAuto = 0,
  kMmaRowWarp = 1,
  kMmaPipe = 2,
  kTc5 = 3,
  kMmaCluster = 4,
  kMmaR8 = 5,
  kMmaR8Cluster = 6,
  kTc5Balanced = 7,
  kMmaC8 = 8,
  kMmaC4x2 = 9,
  kNumVariants = 10
};

m2rnn_status common_checks(const void* q, const void* k, const void* v, const void* a,
                           const float* alpha, const float* beta, const void* W, const float* w_r,
                           const float* y, int B, int T, int N, int K, int V) {
  if (!alpha || !beta || !W || !w_r) return M2RNN_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !a || !y)) return M2RNN_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || K < 1 || V < 1 || T < 0) return M2RNN_ERR_INVALID_ARG;
  if ((long long)B * N > 0x7fffffffLL) return M2RNN_ERR_UNSUPPORTED;
  return M2RNN_OK;
}

// T == 0: the final state is the initial state.
m2rnn_status empty_sequence(const float* H0, float* H_T, int B, int N, int K, int V,
                            cudaStream_t s) {
  if (!H_T) return M2RNN_OK;
  const size_t bytes = sizeof(float) * (size_t)B * N * K * V;
  cudaError_t err = cudaSuccess;
  if (!H0)
    err = cudaMemsetAsync(H_T, 0, bytes, s);
  else if (H0 != H_T)
    err = cudaMemcpyAsync(H_T, H0, bytes, cudaMemcpyDeviceToDevice, s);
  return err == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

m2rnn_status backward_checks(const BackwardProblem& p, size_t workspace_bytes) {
  if (p.B < 1 || p.N < 1 || p.K < 1 || p.V < 1 || p.T < 0) return M2RNN_ERR_INVALID_ARG;
  if (p.Nqk != 1 && p.Nqk != p.N) return M2RNN_ERR_INVALID_ARG;
  if ((long long)p.B * p.N > 0x7fffffffLL) return M2RNN_ERR_UNSUPPORTED;
  if (p.K > 128 || p.V > 128) return M2RNN_ERR_UNSUPPORTED;
  if (!p.alpha || !p.beta || !p.W || !p.w_r || !p.dalpha || !p.dbeta || !p.dW || !p.dw_r ||
      !p.ws)
    return M2RNN_ERR_INVALID_ARG;
  if (p.T > 0 && (!p.q || !p.k || !p.v || !p.a || !p.Hs || !p.dy || !p.dq || !p.dk || !p.dv ||
                  !p.da))
    return M2RNN_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(float) * backward_workspace_floats(p.B, p.T, p.N, p.Nqk, p.K, p.V))
    return M2RNN_ERR_INVALID_ARG;
  if (!aligned(p.ws, 16)) return M2RNN_ERR_INVALID_ARG;
  return M2RNN_OK;
}

// SMs of the current device (152 on GB300, also the answer when no device can be queried).
int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 152;
  return sms;
}

// Clusters of R CTAs (R = 8 or 4) of the eight-SMs-per-pair K = 64, V = 128 kernel that the
// device runs at once: the occupancy calculator's answer, or, without a device to ask, the
// count it gives on a 152-SM GB300 (15 of eight: its graphics processing clusters are of
// unequal size; 36 of four) scaled to the SM count.
int c8_capacity(int R, int sms) {
  const int n = mma_c8_max_clusters(R);
  return n > 0 ? n : sms * (R == 8 ? 15 : 36) / 152;
}
// Eight SMs per pair for K = 64, V = 128, while every cluster of the launch is resident at
// once: one 8-CTA cluster per pair (kMmaC8), else two 4-CTA clusters (kMmaC4x2); 0 when
// neither fits (the 4-CTA kernel then runs, four SMs per pair).
int c8_form(long long pairs, int sms) {
  if (pairs <= c8_capacity(8, sms)) return kMmaC8;
  if (2 * pairs <= c8_capacity(4, sms)) return kMmaC4x2;
  return 0;
}

// The automatic variant: a function of the shape and of how many (batch, head) pairs there
// are for the GPU's SMs.  Eight-row warps split over a two-block cluster when the pairs fill
// at most half the SMs (each block then holds one compute warp per sub-partition), else one
// block per pair.  K = 64, V = 128: eight SMs per pair while every pair's cluster is resident
// at once, else four.
int pick(long long pairs, int K, int V, int sms) {
  if (tc5_supports(K, V)) return pairs > 2LL * sms ? kTc5Balanced : kTc5;
  if (mma_c8_supports(K, V)) {
    const int form = c8_form(pairs, sms);
    if (form) return form;
  }
  if (mma_cluster_supports(K, V)) return kMmaCluster;
  if (mma_r8_cluster_supports(K, V) && 2 * pairs <= sms) return kMmaR8Cluster;
  if (mma_r8_supports(K, V)) return kMmaR8;
  if (mma_pipe_supports(K, V)) return kMmaPipe;
  if (mma_rowwarp_supports(K, V)) return kMmaRowWarp;
  return 0;
}

bool supports(int variant, int K, int V) {
  switch (variant) {
    case kMmaRowWarp: return mma_rowwarp_supports(K, V);
    case kMmaPipe: return mma_pipe_supports(K, V);
    case kTc5:
    case kTc5Balanced: return tc5_supports(K, V);
    case kMmaCluster: return mma_cluster_supports(K, V);
    case kMmaR8: return mma_r8_supports(K, V);
    case kMmaR8Cluster: return mma_r8_cluster_supports(K, V);
    case kMmaC8:
    case kMmaC4x2: return mma_c8_supports(K, V);
  }
  return false;
}

}  // namespace

bool current_context_id(unsigned long long* id) {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace m2rnn

using namespace m2rnn;

extern "C" {

const char* m2rnn_status_string(m2rnn_status s) {
  switch (s) {
    case M2RNN_OK: return "ok";
    case M2RNN_ERR_INVALID_ARG: return "invalid argument";
    case M2RNN_ERR_UNSUPPORTED: return "unsupported shape or variant";
    case M2RNN_ERR_CUDA: return "CUDA error";
    case M2RNN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int m2rnn_version(void) { return 100; }

const char* m2rnn_variant_name(int variant) {
  switch (variant) {
    case kAuto: return "auto";
    case kMmaRowWarp: return "mma_sync_rowwarp";
    case kMmaPipe: return "mma_sync_pipelined";
    case kTc5: return "tcgen05_k128_v128";
    case kTc5Balanced: return "tcgen05_k128_v128_balanced";
    case kMmaCluster: return "mma_sync_cluster4_k64_v128";
    case kMmaR8: return "mma_sync_rows8";
    case kMmaR8Cluster: return "mma_sync_rows8_cluster2";
    case kMmaC8: return "mma_sync_rows8_cluster8_k64_v128";
    case kMmaC4x2: return "mma_sync_rows8_cluster4x2_k64_v128";
  }
  return nullptr;
}

int m2rnn_pick_variant(int B, int T, int N, int K, int V) {
  (void)T;
  if (B < 1 || N < 1) return 0;
  return pick((long long)B * N, K, V, sm_count());
}

int m2rnn_balanced_stretch(long long pairs, int T, long long workers, long long worker,
                           long long* begin, long long* end) {
  if (pairs < 1 || T < 1 || workers < 1 || worker < 0 || worker >= workers || !begin || !end)
    return -1;
  const long long total = pairs * (long long)T;
  const long long line = tc5_line_per_block(pairs, T, workers);
  *begin = tc5_cut(worker * line, total, T);
  *end = tc5_cut((worker + 1) * line, total, T);
  return 0;
}

int m2rnn_variant_supports(int variant, int B, int T, int N, int K, int V) {
  (void)B;
  (void)T;
  (void)N;
  return supports(variant, K, V) ? 1 : 0;
}

m2rnn_status m2rnn_forward_f32_qk(const float* q, const float* k, const float* v, const float* a,
                                  const float* alpha, const float* beta, const float* W,
                                  const float* w_r, const float* H0, float* y, float* H_T, int B,
                                  int T, int N, int Nqk, int K, int V, void* stream) {
  m2rnn_status st = common_checks(q, k, v, a, alpha, beta, W, w_r, y, B, T, N, K, V);
  if (st != M2RNN_OK) return st;
  if (Nqk != 1 && Nqk != N) return M2RNN_ERR_INVALID_ARG;
  if (K > 128 || V > 128) return M2RNN_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return empty_sequence(H0, H_T, B, N, K, V, s);
  Problem p{q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, K, V, Nqk, 0, nullptr};
  return launch_fwd_f32(p, s) == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_forward_f32(const float* q, const float* k, const float* v, const float* a,
                               const float* alpha, const float* beta, const float* W,
                               const float* w_r, const float* H0, float* y, float* H_T, int B,
                               int T, int N, int K, int V, void* stream) {
  return m2rnn_forward_f32_qk(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, N, K, V,
                              stream);
}

m2rnn_status m2rnn_forward_bf16_qk(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const uint16_t* a, const float* alpha, const float* beta,
                                   const uint16_t* W, const float* w_r, const float* H0, float* y,
                                   float* H_T, int B, int T, int N, int Nqk, int K, int V,
                                   int variant, void* stream) {
  m2rnn_status st = common_checks(q, k, v, a, alpha, beta, W, w_r, y, B, T, N, K, V);
  if (st != M2RNN_OK) return st;
  if (Nqk != 1 && Nqk != N) return M2RNN_ERR_INVALID_ARG;
  const int debug = variant >> 8;
  int base = variant & 0xff;
  if (base < 0 || base >= kNumVariants) return M2RNN_ERR_INVALID_ARG;
  if (base == kAuto) base = pick((long long)B * N, K, V, sm_count());
  if (base == 0) return M2RNN_ERR_UNSUPPORTED;
  if (!supports(base, K, V)) return M2RNN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(W, 16) ||
      !aligned(y, 16) || !aligned(H0, 16) || !aligned(H_T, 16) || !aligned(a, 2))
    return M2RNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return empty_sequence(H0, H_T, B, N, K, V, s);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  int* status = status_address(dev);
  EncodeTiledFn enc = encode_fn();
  if (!status || !enc) return M2RNN_ERR_CUDA;
  Problem p{q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, K, V, Nqk, debug, status};
  cudaError_t err = cudaErrorInvalidValue;
  switch (base) {
    case kMmaRowWarp: err = launch_fwd_bf16_mma_rowwarp(p, enc, s); break;
    case kMmaPipe: err = launch_fwd_bf16_mma_pipe(p, enc, s); break;
    case kTc5: err = launch_fwd_bf16_tc5(p, enc, s, false); break;
    case kTc5Balanced: err = launch_fwd_bf16_tc5(p, enc, s, true); break;
    case kMmaCluster: err = launch_fwd_bf16_mma_cluster(p, enc, s); break;
    case kMmaC8: err = launch_fwd_bf16_mma_c8(p, enc, s, 8); break;
    case kMmaC4x2: err = launch_fwd_bf16_mma_c8(p, enc, s, 4); break;
    case kMmaR8: err = launch_fwd_bf16_mma_r8(p, enc, s); break;
    case kMmaR8Cluster: err = launch_fwd_bf16_mma_r8_cluster(p, enc, s); break;
  }
  return err == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_forward_conv_bf16(const uint16_t* xq, const uint16_t* xk, const uint16_t* xv,
                                     const float* wq, const float* bq, const float* wk,
                                     const float* bk, const float* wv, const float* bv,
                                     const uint16_t* a, const float* alpha, const float* beta,
                                     const uint16_t* W, const float* w_r, const float* H0,
                                     float* y, float* H_T, int B, int T, int N, int Nqk, int K,
                                     int V, void* stream) {
  m2rnn_status st = common_checks(xq, xk, xv, a, alpha, beta, W, w_r, y, B, T, N, K, V);
  if (st != M2RNN_OK) return st;
  if (Nqk != 1 && Nqk != N) return M2RNN_ERR_INVALID_ARG;
  if (T > 0 && (!wq || !wk || !wv)) return M2RNN_ERR_INVALID_ARG;
  if (!mma_r8_supports(K, V)) return M2RNN_ERR_UNSUPPORTED;
  if (!aligned(xq, 16) || !aligned(xk, 16) || !aligned(xv, 16) || !aligned(W, 16) ||
      !aligned(y, 16) || !aligned(H0, 16) || !aligned(H_T, 16) || !aligned(a, 2) ||
      !aligned(wq, 16) || !aligned(wk, 16) || !aligned(wv, 16))
    return M2RNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return empty_sequence(H0, H_T, B, N, K, V, s);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  int* status = status_address(dev);
  EncodeTiledFn enc = encode_fn();
  if (!status || !enc) return M2RNN_ERR_CUDA;
  Problem p{xq, xk, xv, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, K, V, Nqk, 0, status};
  p.conv.wq = wq, p.conv.bq = bq, p.conv.wk = wk, p.conv.bk = bk, p.conv.wv = wv, p.conv.bv = bv;
  const int base = pick((long long)B * N, K, V, sm_count());
  const cudaError_t err = base == kMmaR8Cluster ? launch_fwd_bf16_mma_r8_cluster(p, enc, s)
                                                : launch_fwd_bf16_mma_r8(p, enc, s);
  return err == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_forward_bf16_variant(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                        const uint16_t* a, const float* alpha, const float* beta,
                                        const uint16_t* W, const float* w_r, const float* H0,
                                        float* y, float* H_T, int B, int T, int N, int K, int V,
                                        int variant, void* stream) {
  return m2rnn_forward_bf16_qk(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, N, K, V,
                               variant, stream);
}

m2rnn_status m2rnn_forward_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const uint16_t* a, const float* alpha, const float* beta,
                                const uint16_t* W, const float* w_r, const float* H0, float* y,
                                float* H_T, int B, int T, int N, int K, int V, void* stream) {
  return m2rnn_forward_bf16_qk(q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, N, K, V,
                               kAuto, stream);
}

m2rnn_status m2rnn_forward_train_f32(const float* q, const float* k, const float* v,
                                     const float* a, const float* alpha, const float* beta,
                                     const float* W, const float* w_r, const float* H0, float* y,
                                     float* H_T, float* Hs, int B, int T, int N, int Nqk, int K,
                                     int V, void* stream) {
  m2rnn_status st = common_checks(q, k, v, a, alpha, beta, W, w_r, y, B, T, N, K, V);
  if (st != M2RNN_OK) return st;
  if (Nqk != 1 && Nqk != N) return M2RNN_ERR_INVALID_ARG;
  if (T > 0 && !Hs) return M2RNN_ERR_INVALID_ARG;
  if (K > 128 || V > 128) return M2RNN_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return empty_sequence(H0, H_T, B, N, K, V, s);
  Problem p{q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, K, V, Nqk, 0, nullptr, Hs};
  return launch_fwd_f32(p, s) == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_forward_train_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      const uint16_t* a, const float* alpha, const float* beta,
                                      const uint16_t* W, const float* w_r, const float* H0,
                                      float* y, float* H_T, uint16_t* Hs, int B, int T, int N,
                                      int Nqk, int K, int V, void* stream) {
  m2rnn_status st = common_checks(q, k, v, a, alpha, beta, W, w_r, y, B, T, N, K, V);
  if (st != M2RNN_OK) return st;
  if (Nqk != 1 && Nqk != N) return M2RNN_ERR_INVALID_ARG;
  if (T > 0 && !Hs) return M2RNN_ERR_INVALID_ARG;
  const bool pipe = mma_pipe_supports(K, V);
  const bool tc5 = tc5_supports(K, V);
  const bool cluster = mma_cluster_supports(K, V);
  if (!pipe && !tc5 && !cluster && !mma_rowwarp_supports(K, V)) return M2RNN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(W, 16) ||
      !aligned(y, 16) || !aligned(H0, 16) || !aligned(H_T, 16) || !aligned(Hs, 16) ||
      !aligned(a, 2))
    return M2RNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return empty_sequence(H0, H_T, B, N, K, V, s);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  int* status = status_address(dev);
  EncodeTiledFn enc = encode_fn();
  if (!status || !enc) return M2RNN_ERR_CUDA;
  Problem p{q, k, v, a, alpha, beta, W, w_r, H0, y, H_T, B, T, N, K, V, Nqk, 0, status, Hs};
  // K, V <= 64: the pipelined kernel; K = V = 128: the tcgen05 kernel (balanced above two
  // pairs per SM); K = 64, V = 128: eight SMs per pair while every cluster is resident at once
  // (one 8-CTA or two 4-CTA clusters per pair), else the 4-CTA kernel; other shapes (V = 128,
  // K up to 128): the row-warp kernel.
  const int form = cluster ? c8_form((long long)B * N, sm_count()) : 0;
  const bool c8 = form != 0;
  const cudaError_t err =
      pipe      ? launch_fwd_bf16_mma_pipe(p, enc, s)
      : tc5     ? launch_fwd_bf16_tc5(p, enc, s, (long long)B * N > 2LL * sm_count())
      : c8      ? launch_fwd_bf16_mma_c8(p, enc, s, form == kMmaC8 ? 8 : 4)
      : cluster ? launch_fwd_bf16_mma_cluster(p, enc, s)
                : launch_fwd_bf16_mma_rowwarp(p, enc, s);
  return err == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

size_t m2rnn_backward_workspace_bytes(int B, int T, int N, int Nqk, int K, int V) {
  if (B < 1 || N < 1 || K < 1 || V < 1 || T < 0 || K > 128 || V > 128) return 0;
  if (Nqk != 1 && Nqk != N) return 0;
  return sizeof(float) * backward_workspace_floats(B, T, N, Nqk, K, V);
}

m2rnn_status m2rnn_backward_f32(const float* q, const float* k, const float* v, const float* a,
                                const float* alpha, const float* beta, const float* W,
                                const float* w_r, const float* H0, const float* Hs,
                                const float* dy, const float* dH_T, float* dq, float* dk,
                                float* dv, float* da, float* dalpha, float* dbeta, float* dW,
                                float* dw_r, float* dH0, int B, int T, int N, int Nqk, int K,
                                int V, void* workspace, size_t workspace_bytes, void* stream) {
  BackwardProblem p{q,  k,  v,  a,      alpha, beta, W,  w_r,  H0, Hs, dy, dH_T, dq, dk,
                    dv, da, dalpha, dbeta, dW,   dw_r, dH0, static_cast<float*>(workspace),
                    B,  T,  N,  K,      V,     Nqk};
  m2rnn_status st = backward_checks(p, workspace_bytes);
  if (st != M2RNN_OK) return st;
  return launch_bwd_f32(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? M2RNN_OK
                                                                               : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_backward_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const uint16_t* a, const float* alpha, const float* beta,
                                 const uint16_t* W, const float* w_r, const float* H0,
                                 const uint16_t* Hs, const float* dy, const float* dH_T, float* dq,
                                 float* dk, float* dv, float* da, float* dalpha, float* dbeta,
                                 float* dW, float* dw_r, float* dH0, int B, int T, int N, int Nqk,
                                 int K, int V, int variant, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  BackwardProblem p{q,  k,  v,  a,      alpha, beta, W,  w_r,  H0, Hs, dy, dH_T, dq, dk,
                    dv, da, dalpha, dbeta, dW,   dw_r, dH0, static_cast<float*>(workspace),
                    B,  T,  N,  K,      V,     Nqk};
  m2rnn_status st = backward_checks(p, workspace_bytes);
  if (st != M2RNN_OK) return st;
  const int debug = variant >> 8;
  int base = variant & 0xff;
  if (base < 0 || base > 7) return M2RNN_ERR_INVALID_ARG;
  const bool mma_ok = bwd_mma_supports(K, V) && T > 0;
  const bool tc128_ok = bwd_tc128_supports(K, V) && T > 0;
  const bool tc128t_ok = bwd_tc128t_supports(K, V) && T > 0;
  if (base == 0) base = mma_ok ? 5 : tc128t_ok ? 7 : tc128_ok ? 6 : 1;
  if (base >= 2 && base <= 5 && !mma_ok) return M2RNN_ERR_UNSUPPORTED;
  if (base == 6 && !tc128_ok) return M2RNN_ERR_UNSUPPORTED;
  if (base == 7 && !tc128t_ok) return M2RNN_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (base == 1) return launch_bwd_simt_bf16(p, s) == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(W, 16) ||
      !aligned(Hs, 16) || !aligned(dy, 16) || !aligned(dv, 16) || !aligned(dH0, 16) ||
      !aligned(dH_T, 16) || !aligned(H0, 16) || !aligned(w_r, 8))
    return M2RNN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  int* status = status_address(dev);
  EncodeTiledFn enc = encode_fn();
  if (!status || !enc) return M2RNN_ERR_CUDA;
  const cudaError_t err =
      base == 7   ? launch_bwd_bf16_tc128t(p, enc, debug, status, s)
      : base == 6 ? launch_bwd_bf16_tc128(p, enc, debug, status, s)
      : base == 5 ? launch_bwd_bf16_tcc(p, enc, debug, status, s)
      : base >= 3 ? launch_bwd_bf16_tc(p, enc, debug, status, base == 4 ? 8 : 4, s)
                  : launch_bwd_bf16_mma(p, enc, debug, status, s);
  return err == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_decode_step_bf16_variant(const uint16_t* q, const uint16_t* k,
                                            const uint16_t* v, const uint16_t* a,
                                            const float* alpha, const float* beta,
                                            const uint16_t* W, const float* w_r,
                                            const float* H_in, float* H_out, float* y, int B,
                                            int N, int Nqk, int K, int V, int variant,
                                            void* stream) {
  m2rnn_status st = common_checks(q, k, v, a, alpha, beta, W, w_r, y, B, 1, N, K, V);
  if (st != M2RNN_OK) return st;
  if (!H_out) return M2RNN_ERR_INVALID_ARG;
  if (Nqk != 1 && Nqk != N) return M2RNN_ERR_INVALID_ARG;
  const int debug = variant >> 8, which = variant & 0xff;
  if (which < 0 || which > 2) return M2RNN_ERR_INVALID_ARG;
  if (!decode_supports(K, V)) return M2RNN_ERR_UNSUPPORTED;
  if (!aligned(v, 4) || !aligned(W, 16) || !aligned(H_in, 8) || !aligned(H_out, 8) ||
      !aligned(q, 2) || !aligned(k, 2) || !aligned(a, 2))
    return M2RNN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  int* status = status_address(dev);
  EncodeTiledFn enc = encode_fn();
  Problem p{q, k, v, a, alpha, beta, W, w_r, H_in, y, H_out, B, 1, N, K, V, Nqk, debug, status};
  if (which == 2 && (!decode_persist_supports(p) || !enc || !status))
    return M2RNN_ERR_UNSUPPORTED;
  return launch_decode_bf16(p, enc, static_cast<cudaStream_t>(stream), which) == cudaSuccess
             ? M2RNN_OK
             : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_decode_step_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const uint16_t* a, const float* alpha, const float* beta,
                                    const uint16_t* W, const float* w_r, const float* H_in,
                                    float* H_out, float* y, int B, int N, int Nqk, int K, int V,
                                    void* stream) {
  return m2rnn_decode_step_bf16_variant(q, k, v, a, alpha, beta, W, w_r, H_in, H_out, y, B, N,
                                        Nqk, K, V, 0, stream);
}

m2rnn_status m2rnn_conv_silu_bf16(const uint16_t* x, const float* w, const float* bias,
                                  uint16_t* out, int B, int T, int C, void* stream) {
  if (B < 1 || T < 0 || C < 1) return M2RNN_ERR_INVALID_ARG;
  if (T > 0 && (!x || !w || !out)) return M2RNN_ERR_INVALID_ARG;
  if (C % 8 != 0) return M2RNN_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(w, 16) || !aligned(bias, 4))
    return M2RNN_ERR_INVALID_ARG;
  if (T == 0) return M2RNN_OK;
  return launch_conv_silu(x, w, bias, out, B, T, C, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? M2RNN_OK
             : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_gate_rmsnorm_bf16(const float* y, const uint16_t* g_pre, const float* w_norm,
                                     float eps, uint16_t* out, long long rows, int D,
                                     void* stream) {
  if (rows < 0 || D < 1 || !(eps >= 0.f)) return M2RNN_ERR_INVALID_ARG;
  if (rows > 0 && (!y || !g_pre || !w_norm || !out)) return M2RNN_ERR_INVALID_ARG;
  if (D % 8 != 0) return M2RNN_ERR_UNSUPPORTED;
  if (!aligned(y, 16) || !aligned(g_pre, 16) || !aligned(w_norm, 16) || !aligned(out, 16))
    return M2RNN_ERR_INVALID_ARG;
  if (rows == 0) return M2RNN_OK;
  return launch_gate_rmsnorm(y, g_pre, w_norm, eps, out, rows, D,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? M2RNN_OK
             : M2RNN_ERR_CUDA;
}

m2rnn_status m2rnn_stream_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return M2RNN_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  int* addr = status_address(dev);
  if (!addr) return M2RNN_ERR_CUDA;
  int word = 0;
  const int zero = 0;
  if (cudaMemcpy(&word, addr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(addr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return M2RNN_ERR_CUDA;
  return word == kStatusTimeout ? M2RNN_ERR_TIMEOUT : M2RNN_OK;
}

}  // extern "C"
