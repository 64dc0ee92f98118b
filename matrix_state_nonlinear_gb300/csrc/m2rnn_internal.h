// m2rnn_internal.h — shared between the host API layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace m2rnn {

// Device status word values (written by kernels, read by m2rnn_stream_status).
enum : int { kStatusOk = 0, kStatusTimeout = 4 };

// Test hook carried in bits 8.. of the variant id: the kernel's first wait is on
// a barrier that nothing arrives at, with a short limit, so the timeout path runs.
enum : int { kDebugForceTimeout = 1 };

// Bounded waits give up after this many SM cycles (about one second at 2 GHz).
constexpr long long kWaitLimitCycles = 2000000000LL;
// Limit used by the forced-timeout test hook (about 0.5 ms).
constexpr long long kDebugWaitLimitCycles = 1000000LL;

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or false when no
// context is current yet.  Device addresses of module symbols are cached per context id,
// so a device reset (which ends the context and may reload the module elsewhere) makes
// the next call resolve them again.
bool current_context_id(unsigned long long* id);

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const void* a;
  const float* alpha;
  const float* beta;
  const void* W;
  const float* w_r;
  const float* H0;
  float* y;
  float* H_T;
  int B, T, N, K, V;
  int Nqk;          // heads of q and k: N (one per head) or 1 (shared by all heads)
  int debug;        // kDebug* bits (tests only)
  int* status;      // device address of this device's status word
  void* Hs = nullptr;  // optional: every step's state [B, N, T, K, V] (fp32 path: float;
                      // bf16 path: the bf16-rounded state, uint16_t bits)
  // Optional fused block prologue (eight-row kernels): q, k, v are then the raw projections
  // and these the causal conv's taps [C][4] and biases [C] (biases may be null).
  struct Conv {
    const float *wq = nullptr, *bq = nullptr, *wk = nullptr, *bk = nullptr, *wv = nullptr,
                *bv = nullptr;
  } conv;
};

// Backward pass (reverse scan of the notes' Sec. 2.7).  Pointers as in the C ABI;
// `ws` is the caller's workspace (backward_workspace_floats floats).
struct BackwardProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* a;
  const float* alpha;
  const float* beta;
  const void* W;
  const float* w_r;
  const float* H0;   // may be null (zero initial state)
  const void* Hs;    // [B, N, T, K, V] states of the training forward (fp32 or bf16 bits)
  const float* dy;   // [B, T, N, V]
  const float* dH_T; // may be null (zero)
  float* dq;         // [B, T, Nqk, K]
  float* dk;         // [B, T, Nqk, K]
  float* dv;         // [B, T, N, V]
  float* da;         // [B, T, N]
  float* dalpha;     // [N]
  float* dbeta;      // [N]
  float* dW;         // [N, V, V]
  float* dw_r;       // [N, V]
  float* dH0;        // [B, N, K, V], may be null
  float* ws;
  int B, T, N, K, V, Nqk;
};

// Floats of the per-pair partial block: C (K V), dW partial (V V), dw_r partial (V),
// dalpha and dbeta partials (2), padded to a multiple of 4.
__host__ __device__ inline size_t backward_pair_floats(int K, int V) {
  return ((size_t)K * V + (size_t)V * V + V + 2 + 3) & ~(size_t)3;
}
// Workspace floats: the pair blocks, plus per-head dq, dk when q, k are shared.
inline size_t backward_workspace_floats(int B, int T, int N, int Nqk, int K, int V) {
  size_t n = (size_t)B * N * backward_pair_floats(K, V);
  if (Nqk == 1 && N > 1) n += 2 * (size_t)B * T * N * K;
  return n;
}

// fp32 SIMT backward (any 1 <= K, V <= 128), then the reduction over the batch.
cudaError_t launch_bwd_f32(const BackwardProblem& p, cudaStream_t stream);
// The same SIMT backward on bf16 q, k, v, a, W (fp32 arithmetic), then the reduction.
cudaError_t launch_bwd_simt_bf16(const BackwardProblem& p, cudaStream_t stream);
// Sum the per-pair partials over the batch (and per-head dq, dk over heads when q, k
// are shared) into dW, dw_r, dalpha, dbeta (dq, dk).  Deterministic order.
cudaError_t launch_bwd_reduce(const BackwardProblem& p, cudaStream_t stream);

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// fp32 SIMT path (any 1 <= K, V <= 128).
cudaError_t launch_fwd_f32(const Problem& p, cudaStream_t stream);

// bf16 warp-MMA path: K % 16 == 0, K <= 128, V in {16, 32, 64, 128}.
bool mma_rowwarp_supports(int K, int V);
cudaError_t launch_fwd_bf16_mma_rowwarp(const Problem& p, EncodeTiledFn enc, cudaStream_t stream);

// bf16 software-pipelined warp-MMA path with a producer warp: K % 16 == 0,
// K <= 64, V in {16, 32, 64}.
bool mma_pipe_supports(int K, int V);
cudaError_t launch_fwd_bf16_mma_pipe(const Problem& p, EncodeTiledFn enc, cudaStream_t stream);

// bf16 warp-MMA path with eight state rows per warp, the product taken transposed and the
// readout on the tensor core, no producer warp: K % 8 == 0, K <= 64, V in {16, 32, 48, 64}.
bool mma_r8_supports(int K, int V);
cudaError_t launch_fwd_bf16_mma_r8(const Problem& p, EncodeTiledFn enc, cudaStream_t stream);
// The same kernel with a pair's rows split over a two-block cluster (readout partials through
// distributed shared memory): K = 64, V in {16, 32, 48, 64}.  For pair counts that fill at
// most half the GPU.
bool mma_r8_cluster_supports(int K, int V);
cudaError_t launch_fwd_bf16_mma_r8_cluster(const Problem& p, EncodeTiledFn enc,
                                           cudaStream_t stream);

// bf16 path on the 5th-generation tensor cores (tcgen05, tensor-memory accumulators),
// two blocks per SM: K = V = 128.  Unbalanced: one block per pair.  Balanced (more pairs
// than resident blocks): every block resident at once, each taking an equal stretch of the
// line of all pairs' steps laid end to end (pair p owns [p T, (p+1) T)); a pair cut by a
// stretch boundary runs its first steps at the start of the later block's stretch and its
// last steps at the end of the earlier block's stretch, the state handed over in between.
bool tc5_supports(int K, int V);
cudaError_t launch_fwd_bf16_tc5(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                                bool balanced);

// Rows of y a handed-off state occupies (K = 128 state rows and one ready word): the
// block that takes a pair over must run at least this many of its steps.
constexpr int kTc5HandoffRows = 129;
// Blocks of the balanced schedule: one per resident slot, at most one per pair.
__host__ __device__ inline long long tc5_balanced_workers(long long pairs, long long slots) {
  return pairs < slots ? pairs : slots;
}
// Steps of the line per block (rounded up).
__host__ __device__ inline long long tc5_line_per_block(long long pairs, int T, long long workers) {
  return (pairs * (long long)T + workers - 1) / workers;
}
// Stretch boundary near line position c: a cut that would leave the earlier block fewer
// than kTc5HandoffRows last steps of a pair moves down to the pair's start instead.
__host__ __device__ inline long long tc5_cut(long long c, long long total, int T) {
  if (c >= total) return total;
  const long long r = c % T;
  return (r != 0 && r < kTc5HandoffRows) ? c - r : c;
}

// bf16 warp-MMA path with a 4-CTA thread-block cluster per pair (rows split over four
// SMs, readout partials exchanged through distributed shared memory): K = 64, V = 128.
bool mma_cluster_supports(int K, int V);
cudaError_t launch_fwd_bf16_mma_cluster(const Problem& p, EncodeTiledFn enc, cudaStream_t stream);
// The same shape on eight SMs per pair (eight rows per CTA, product transposed, each compute
// warp owning 32 value columns), K = 64, V = 128: one 8-CTA cluster per pair (R = 8), or two
// independent 4-CTA clusters per pair (R = 4) that add their halves of y into a y the
// launcher zeroes.  mma_c8_max_clusters(R): the R-CTA clusters the current device runs at
// once (0 when it cannot say).
bool mma_c8_supports(int K, int V);
int mma_c8_max_clusters(int R);
cudaError_t launch_fwd_bf16_mma_c8(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                                   int R);

// Tensor-core backward (warp-level MMA, TMA-staged bf16 states), K = V = 64, then the
// reduction.  `debug` takes the kDebug* bits; `status` is the device status word.
bool bwd_mma_supports(int K, int V);
cudaError_t launch_bwd_bf16_mma(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                int* status, cudaStream_t stream);
// The same backward with H_{t-1} W and the dW sum on tcgen05 (tensor memory), K = V = 64,
// with 4 compute warps (one per 16-row block) or 8 (two per row block, column halves).
cudaError_t launch_bwd_bf16_tc(const BackwardProblem& p, EncodeTiledFn enc, int debug, int* status,
                               int compute_warps, cudaStream_t stream);
// The same backward with the chain product D_t W^T on tcgen05 as well (eight compute warps).
cudaError_t launch_bwd_bf16_tcc(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                int* status, cudaStream_t stream);

// Backward for V = 128 (K a multiple of 16 up to 128, rows padded to 128) with every product
// on tcgen05 (tensor-memory accumulators, TMA-streamed bf16 states), then the reduction.
bool bwd_tc128_supports(int K, int V);
cudaError_t launch_bwd_bf16_tc128(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                  int* status, cudaStream_t stream);
// The same backward for V = 128 and K <= 64 (a multiple of 16) with the recurrence's products
// transposed (M over the 128 value columns, N = K), so no state row is padding.
bool bwd_tc128t_supports(int K, int V);
cudaError_t launch_bwd_bf16_tc128t(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                   int* status, cudaStream_t stream);

// One decode step (T = 1) on the warp MMA: K % 16 == 0, K <= 128, V in {16, 32, 64, 128}.
// Uses q, k, v, a, alpha, beta, W, w_r, H0 (state in, may be null), H_T (state out, may
// equal H0), y, B, N, K, V, Nqk and status of the problem.  K = V = 64 with at least 2048
// pairs takes a persistent TMA-fed kernel (same arithmetic); `enc` may be null.
// `which`: 0 picks (persistent kernel at K = V = 64 with >= 2048 pairs), 1 forces the
// one-block-per-pair kernel, 2 the persistent kernel (decode_persist_supports must hold).
// The persistent kernel honours p.debug (kDebugForceTimeout).
bool decode_supports(int K, int V);
bool decode_persist_supports(const Problem& p);
cudaError_t launch_decode_bf16(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                               int which);

// Block prologue / epilogue (memory-bound): causal depthwise Conv1D (kernel 4) + SiLU
// over [B, T, C] bf16 (C % 8 == 0), and the output gate + RMSNorm over rows of D
// (D % 8 == 0) values.
cudaError_t launch_conv_silu(const uint16_t* x, const float* w, const float* bias, uint16_t* out,
                             int B, int T, int C, cudaStream_t stream);
cudaError_t launch_gate_rmsnorm(const float* y, const uint16_t* g_pre, const float* w_norm,
                                float eps, uint16_t* out, long long rows, int D,
                                cudaStream_t stream);

}  // namespace m2rnn
