/*
 * m2rnn.h — C ABI of the GB300 (sm_103a) M²RNN forward-recurrence library.
 *
 * What it computes.  The forward pass of the M²RNN matrix-state nonlinear
 * recurrence, as stated in the M²RNN study notes ("M²RNN: 矩阵状态非线性 RNN
 * 的容量、表达力与系统代价", notes on arXiv:2603.14360v2):
 *   Sec. 2.2, Eq. (13)/(17):  f_t = exp(-alpha_n * softplus(a_t + beta_n))
 *   Sec. 2.1, Eq. (10):       Z_t = tanh(H_{t-1} W_n + k_t v_t^T)
 *             Eq. (11):       H_t = f_t H_{t-1} + (1 - f_t) Z_t
 *             Eq. (12):       y_t = H_t^T q_t + w_r ⊙ v_t
 * for every (batch b, head n) independently (Sec. 2.6: each (b, n) pair is an
 * independent work unit), starting from H_0 (zero when not given).
 *
 * Layout.  Every tensor is dense and row-major (innermost index last):
 *   q, k   [B, T, N, K]     keys/queries, one row per (b, t, n)
 *   v      [B, T, N, V]
 *   a      [B, T, N]        gate logits a_{t,n} = (W_f x_t)_n
 *   alpha  [N], beta [N]    gate parameters (float32); alpha_n >= 0 keeps f in [0, 1]
 *   W      [N, V, V]        per-head transition, right-multiplied:
 *                           (H W)_{ij} = sum_l H_{il} W_{lj}
 *   w_r    [N, V]           value residual weight (float32)
 *   H0     [B, N, K, V]     initial state (float32), or NULL for zeros
 *   y      [B, T, N, V]     readout (float32), written
 *   H_T    [B, N, K, V]     final state (float32), written unless NULL
 *
 * Ownership and threading.  The caller owns every buffer: device pointers
 * (cudaMalloc'd or torch-owned) valid until the work on `stream` completes.
 * The library allocates no device memory per call, keeps no per-call state, and
 * only enqueues work on `stream` (a cudaStream_t passed as void*; NULL is the
 * legacy default stream); it returns before the GPU finishes.  Calls from
 * several host threads are safe.  H0 == H_T (in place) is allowed: each pair's
 * initial state is read before anything of that pair's final state is written.
 * No other output may alias an input.
 *
 * Errors.  Arguments are validated on the host before anything is enqueued;
 * a failed check returns an error and launches nothing.  A bounded device-side
 * wait that gives up is recorded in a per-device status word and reported by
 * m2rnn_stream_status().  The kernels never trap.
 */
#ifndef M2RNN_H
#define M2RNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum m2rnn_status {
  M2RNN_OK = 0,
  M2RNN_ERR_INVALID_ARG = 1,   /* null required pointer, B/N/K/V < 1, T < 0, misaligned pointer */
  M2RNN_ERR_UNSUPPORTED = 2,   /* shape outside what the selected path supports */
  M2RNN_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  M2RNN_ERR_TIMEOUT = 4        /* a bounded device wait gave up (from m2rnn_stream_status) */
} m2rnn_status;

/*
 * fp32-operand path.  Every tensor is float32.  Supports 1 <= K, V <= 128 and
 * any B, N >= 1, T >= 0.  tanh, exp and log1p are the accurate CUDA math
 * functions; the contraction H W is an fp32 dot product.
 * T == 0 writes H_T = H0 (or zeros) and no y.
 * Returns INVALID_ARG for a null alpha/beta/W/w_r pointer, a null q/k/v/a/y
 * pointer when T > 0 (the empty tensors of T == 0 may be NULL), B, N, K, V < 1
 * or T < 0; UNSUPPORTED for K or V > 128; CUDA if the launch fails.
 */
m2rnn_status m2rnn_forward_f32(const float* q, const float* k, const float* v, const float* a,
                               const float* alpha, const float* beta, const float* W,
                               const float* w_r, const float* H0, float* y, float* H_T,
                               int B, int T, int N, int K, int V, void* stream);

/*
 * bf16-operand / fp32-state path.  q, k, v, a and W are bfloat16 (passed as
 * their uint16_t bit patterns); alpha, beta, w_r, H0, y and H_T are float32.
 * The state H is carried in fp32 and rounded to bf16 only as the tensor-core
 * operand of each step's H W; the rank-1 term, tanh and gate lerp are fp32, and
 * the readout H_t^T q_t accumulates in fp32 (the eight-row kernels take it on the
 * tensor cores from the same bf16 rounding of H_t that the next step's H W reads).  Supports any 1 <= K <= 128 and V a multiple of 16 with 16 <= V <= 128.
 * K that is not a multiple of 16 runs with its rows padded to the next multiple
 * of 16 inside the kernel (padding rows hold zero state, k and q, stay zero for
 * every t and are never stored), so the results are those of the K-row problem.
 * q, k, v, W, y, H0 and H_T must be 16-byte aligned (INVALID_ARG otherwise).
 * Same argument rules and errors as m2rnn_forward_f32, plus UNSUPPORTED for K or
 * V > 128 and for V not a multiple of 16.
 */
m2rnn_status m2rnn_forward_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const uint16_t* a, const float* alpha, const float* beta,
                                const uint16_t* W, const float* w_r, const float* H0, float* y,
                                float* H_T, int B, int T, int N, int K, int V, void* stream);

/*
 * As m2rnn_forward_bf16, with an explicit kernel variant (for testing each
 * variant's parity and for measurement).  variant 0 = automatic choice (what
 * m2rnn_forward_bf16 uses); other values are listed by m2rnn_variant_name().
 * Returns UNSUPPORTED if the variant cannot run this shape.
 */
m2rnn_status m2rnn_forward_bf16_variant(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                        const uint16_t* a, const float* alpha, const float* beta,
                                        const uint16_t* W, const float* w_r, const float* H0,
                                        float* y, float* H_T, int B, int T, int N, int K, int V,
                                        int variant, void* stream);

/*
 * Multi-value sharing (the notes' Sec. 2.4: one query/key set shared by all value
 * heads, N_q = N_k = 1, while each head keeps its own v, f, W and state).  As
 * m2rnn_forward_f32 / m2rnn_forward_bf16_variant, with q and k of shape
 * [B, T, Nqk, K]: Nqk == N gives one query/key vector per head (the plain entry
 * points), Nqk == 1 uses the same q_t, k_t for every head n.  Any other Nqk
 * returns INVALID_ARG.  Input bytes per token-head drop to about 2 (V + 1) + 4K/N
 * on the bf16 path when Nqk == 1.
 */
m2rnn_status m2rnn_forward_f32_qk(const float* q, const float* k, const float* v, const float* a,
                                  const float* alpha, const float* beta, const float* W,
                                  const float* w_r, const float* H0, float* y, float* H_T, int B,
                                  int T, int N, int Nqk, int K, int V, void* stream);
m2rnn_status m2rnn_forward_bf16_qk(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const uint16_t* a, const float* alpha, const float* beta,
                                   const uint16_t* W, const float* w_r, const float* H0, float* y,
                                   float* H_T, int B, int T, int N, int Nqk, int K, int V,
                                   int variant, void* stream);

/*
 * Training support (the notes' Sec. 2.6-2.7).  The backward pass re-runs the
 * recurrence while keeping every step's state in HBM, then scans time in reverse.
 *
 * m2rnn_forward_train_*: the forward pass of m2rnn_forward_*_qk that also writes
 *   Hs     [B, N, T, K, V]  Hs[b][n][t] = H_t after step t (t = 0..T-1), the states
 *                           the backward reads.  fp32 entry: float32.  bf16 entry:
 *                           bfloat16 (uint16_t bits), the round-to-nearest-even
 *                           rounding of H_t, i.e. exactly the tensor-core operand
 *                           the next step multiplies by W (B·N·T·K·V·2 bytes).
 *   Hs is required when T > 0 (16-byte aligned on the bf16 entry).  The bf16 entry
 *   runs the state-keeping form of a forward kernel, with that kernel's arithmetic:
 *   the pipelined warp-MMA kernel for K a multiple of 16 up to 64 with V in
 *   {16, 32, 64}; the tcgen05 kernel for K = V = 128; eight SMs per pair (or the
 *   4-CTA cluster kernel when their clusters do not all fit) for K = 64, V = 128;
 *   and the row-warp kernel for every other 1 <= K <= 128 with V a multiple of 16
 *   up to 128 (UNSUPPORTED otherwise).  The fp32 entry supports 1 <= K, V <= 128.
 */
m2rnn_status m2rnn_forward_train_f32(const float* q, const float* k, const float* v,
                                     const float* a, const float* alpha, const float* beta,
                                     const float* W, const float* w_r, const float* H0, float* y,
                                     float* H_T, float* Hs, int B, int T, int N, int Nqk, int K,
                                     int V, void* stream);
m2rnn_status m2rnn_forward_train_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      const uint16_t* a, const float* alpha, const float* beta,
                                      const uint16_t* W, const float* w_r, const float* H0,
                                      float* y, float* H_T, uint16_t* Hs, int B, int T, int N,
                                      int Nqk, int K, int V, void* stream);

/*
 * Bytes of device workspace m2rnn_backward_* needs for these sizes (0 for an
 * invalid shape).  Per (b, n) pair it holds the running state gradient and the
 * pair's partial sums of dW, dw_r, dalpha, dbeta; with Nqk == 1 < N also the
 * per-head dq, dk before they are summed over heads.
 */
size_t m2rnn_backward_workspace_bytes(int B, int T, int N, int Nqk, int K, int V);

/*
 * Backward pass: gradients of a loss L that depends on y (dy = dL/dy) and on the
 * final state (dH_T = dL/dH_T, NULL for zero), given the inputs of the forward and
 * its kept states Hs (from m2rnn_forward_train_*, same inputs).  The reverse scan
 * is the notes' Sec. 2.7 with u_t = dy_t, C_T = dH_T:
 *   R_t = C_t + q_t u_t^T,  D_t = ((1 - f_t) R_t) ⊙ (1 - Z_t ⊙ Z_t),
 *   C_{t-1} = f_t R_t + D_t W^T,  dL/df_t = <R_t, H_{t-1} - Z_t>,
 *   dW = sum over b, t of H_{t-1}^T D_t,  dk_t = D_t v_t,
 *   dv_t = D_t^T k_t + w_r ⊙ u_t,  dq_t = H_t u_t,  dH0 = C_{-1},
 * with Z_t = tanh(H_{t-1} W + k_t v_t^T) recomputed from Hs, and the gate of
 * Eq. (13)/(17) differentiated (x = a + beta):
 *   da_t = dL/df_t · (-alpha f sigmoid(x)),  dalpha = sum dL/df_t · (-f softplus(x)),
 *   dbeta = sum da_t,  dw_r = sum over b, t of u_t ⊙ v_t.
 * Outputs (float32, written, caller-owned):
 *   dq, dk [B, T, Nqk, K]  (summed over heads when Nqk == 1)
 *   dv [B, T, N, V], da [B, T, N], dalpha [N], dbeta [N], dW [N, V, V], dw_r [N, V],
 *   dH0 [B, N, K, V] (not written when NULL).
 * dy [B, T, N, V] is float32; Hs has the dtype its forward entry wrote (float32 on
 * the fp32 entry, bf16 bits on the bf16 entry).  On the bf16 entry, t = 0 uses the
 * bf16 rounding of H0, as the forward's first step did.  `workspace` is caller-owned device memory of at least
 * m2rnn_backward_workspace_bytes(...) bytes (INVALID_ARG otherwise); it is
 * overwritten, so two calls in flight at once need two workspaces.  Sums over the
 * batch run in a fixed order: results are deterministic.
 * Errors: INVALID_ARG for a null required pointer (q, k, v, a, Hs, dy, dq, dk, dv,
 * da are required only when T > 0) or a bad size; UNSUPPORTED for K or V > 128.
 * The bf16 entry takes bf16 q, k, v, a, W; its `variant` is 0 (automatic: 5 when
 * K = V = 64 and T > 0, 7 when V = 128, K is a multiple of 16 up to 64 and T > 0,
 * 6 when V = 128, K is a multiple of 16 above 64 and T > 0, else 1),
 * 1 (SIMT kernel, fp32 arithmetic, any K, V <= 128),
 * 2 (H_{t-1} W, D_t W^T and H_{t-1}^T D_t as bf16 warp MMAs with fp32 accumulation) or
 * 3 (H_{t-1} W and H_{t-1}^T D_t on the 5th-generation tensor cores with tensor-memory
 * accumulators, D_t W^T as warp MMAs), 4 (variant 3 with eight compute warps) or 5 (all
 * three products on the 5th-generation tensor cores, the chain product D_t W^T included)
 * or 6 (V = 128: every product on the 5th-generation tensor cores, rows padded to 128;
 * D_t enters the products, dk and dv included, rounded to bf16) or 7 (variant 6 with the
 * recurrence's products transposed, so that the tensor-memory lanes run over the 128
 * columns and no row is padding; K <= 64).
 * Variants 2 to 5 need K = V = 64, variant 6 V = 128 and K a multiple of 16, variant 7
 * V = 128 and K a multiple of 16 up to 64 (UNSUPPORTED otherwise); all of them need q, k, v, W, Hs, dy, dv, H0, dH_T, dH0
 * 16-byte aligned.  Bits 8 and up
 * of `variant` are test hooks (0).
 */
m2rnn_status m2rnn_backward_f32(const float* q, const float* k, const float* v, const float* a,
                                const float* alpha, const float* beta, const float* W,
                                const float* w_r, const float* H0, const float* Hs,
                                const float* dy, const float* dH_T, float* dq, float* dk,
                                float* dv, float* da, float* dalpha, float* dbeta, float* dW,
                                float* dw_r, float* dH0, int B, int T, int N, int Nqk, int K,
                                int V, void* workspace, size_t workspace_bytes, void* stream);
m2rnn_status m2rnn_backward_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const uint16_t* a, const float* alpha, const float* beta,
                                 const uint16_t* W, const float* w_r, const float* H0,
                                 const uint16_t* Hs, const float* dy, const float* dH_T, float* dq,
                                 float* dk, float* dv, float* da, float* dalpha, float* dbeta,
                                 float* dW, float* dw_r, float* dH0, int B, int T, int N, int Nqk,
                                 int K, int V, int variant, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * m2rnn_backward_bf16 without a caller workspace: the workspace comes from a fixed
 * 16 MiB scratch array inside the library (one per device).  The M²RNN notes have
 * no counterpart to this entry point; it computes exactly what m2rnn_backward_bf16
 * (variant 0) computes.
 *   * Shapes whose workspace (m2rnn_backward_workspace_bytes) exceeds 16 MiB return
 *     UNSUPPORTED before anything is enqueued; no memory is ever allocated.
 *   * Every call on a device shares its scratch: calls whose work could overlap in
 *     time (other streams or host threads, unordered) race and give wrong results.
 *     Order them on one stream or with events.
 *   * The first call on a device resolves the scratch address (it may load the
 *     module); make that first call before capturing a stream into a CUDA graph.
 *     The address is cached per CUDA context: after a cudaDeviceReset the next call
 *     resolves it again (and must, again, come before any capture).
 */
m2rnn_status m2rnn_backward_bf16_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                         const uint16_t* a, const float* alpha, const float* beta,
                                         const uint16_t* W, const float* w_r, const float* H0,
                                         const uint16_t* Hs, const float* dy, const float* dH_T,
                                         float* dq, float* dk, float* dv, float* da, float* dalpha,
                                         float* dbeta, float* dW, float* dw_r, float* dH0, int B,
                                         int T, int N, int Nqk, int K, int V, void* stream);

/*
 * One decode step (T = 1) for serving with a fixed-size state: the forward pass of a
 * single token per (b, n), state in, state out.
 *   q, k   [B, Nqk, K] bf16 (Nqk == N, or 1 shared by all heads)
 *   v      [B, N, V] bf16,  a [B, N] bf16
 *   H_in   [B, N, K, V] float32 state before the token (NULL: zero state)
 *   H_out  [B, N, K, V] float32 state after the token (required; H_out == H_in updates
 *          the state in place)
 *   y      [B, N, V] float32
 * The arithmetic is exactly one step of m2rnn_forward_bf16's warp-MMA kernels
 * (the pipelined kernel and the row-warp kernel), so T successive calls reproduce a
 * T-step forward on those kernels bit for bit.  K = V = 128 and K = 64, V = 128 run
 * the forward on other kernels (other summation orders): there the results agree
 * within the bf16 path's tolerance, not bit for bit.  Small batches run one block per (b, n) pair;
 * K = V = 64 with at least 2048 pairs (and every tensor 16-byte aligned) runs a
 * persistent kernel that streams each pair's state and W through shared memory with TMA
 * (same arithmetic, same bits; its bounded waits report timeouts through
 * m2rnn_stream_status).  Either launch is a single kernel, suitable for CUDA-graph capture.
 * Supports any 1 <= K <= 128 and V a multiple of 16 with 16 <= V <= 128 (UNSUPPORTED
 * otherwise; K that is not a multiple of 16 is padded with zero rows as in
 * m2rnn_forward_bf16).  Same pointer and size errors as m2rnn_forward_bf16 (INVALID_ARG
 * for a null H_out, or W not 16-byte aligned).
 */
m2rnn_status m2rnn_decode_step_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const uint16_t* a, const float* alpha, const float* beta,
                                    const uint16_t* W, const float* w_r, const float* H_in,
                                    float* H_out, float* y, int B, int N, int Nqk, int K, int V,
                                    void* stream);

/*
 * As m2rnn_decode_step_bf16 with an explicit kernel: variant 0 = automatic (what
 * m2rnn_decode_step_bf16 uses), 1 = one block per (b, n) pair, 2 = the persistent
 * TMA-fed kernel at any pair count (K = V = 64 and every tensor 16-byte aligned, else
 * UNSUPPORTED).  Both give the same bits.  Bits 8 and up of `variant` are test hooks
 * (0); they act on the persistent kernel only (the per-pair kernel has no device waits).
 * Any other low byte returns INVALID_ARG.
 */
m2rnn_status m2rnn_decode_step_bf16_variant(const uint16_t* q, const uint16_t* k,
                                            const uint16_t* v, const uint16_t* a,
                                            const float* alpha, const float* beta,
                                            const uint16_t* W, const float* w_r,
                                            const float* H_in, float* H_out, float* y, int B,
                                            int N, int Nqk, int K, int V, int variant,
                                            void* stream);

/*
 * The block's elementwise stages around the recurrence (the notes' Sec. 2.3,
 * Eq. (14)-(23); the projections W_q, W_k, W_v, W_g, W_f, W_o are plain GEMMs outside).
 *
 * m2rnn_conv_silu_bf16: prologue of q, k and v (call once per tensor).
 *   out[b,t,c] = SiLU(bias[c] + sum_{j=0..3} w[c][j] * x[b, t-3+j, c]),  x[b, t<0, c] = 0
 *   x, out [B, T, C] bf16 (16-byte aligned, C % 8 == 0, else UNSUPPORTED; out must not
 *   overlap x); w [C, 4] float32 (16-byte aligned); bias [C] float32 or NULL (none).
 *   Its output, viewed as [B, T, N, K] or [B, T, N, V], is the recurrence's q, k or v.
 *
 * m2rnn_gate_rmsnorm_bf16: epilogue.  For each of `rows` rows of D values (a token's
 *   readout over all heads, D = N V, the recurrence's y viewed as [B T, D]):
 *   z = y ⊙ SiLU(g_pre),  out = w_norm ⊙ z / sqrt(mean(z^2) + eps)
 *   (output gate first, then RMSNorm over the whole token).  y float32, g_pre and out
 *   bf16, w_norm [D] float32, eps >= 0; all 16-byte aligned; D % 8 == 0 (else
 *   UNSUPPORTED).  out is ready to be the W_o GEMM's operand.
 * Both: fp32 arithmetic, results rounded to bf16 (nearest even); memory-bound, every
 * element read and written once.
 */
m2rnn_status m2rnn_conv_silu_bf16(const uint16_t* x, const float* w, const float* bias,
                                  uint16_t* out, int B, int T, int C, void* stream);
m2rnn_status m2rnn_gate_rmsnorm_bf16(const float* y, const uint16_t* g_pre, const float* w_norm,
                                     float eps, uint16_t* out, long long rows, int D,
                                     void* stream);

/*
 * The block prologue fused into the bf16 forward (the notes' Sec. 2.3, Eq. (14)-(16)): the
 * recurrence of m2rnn_forward_bf16_qk on
 *   q = SiLU(conv(xq)), k = SiLU(conv(xk)), v = SiLU(conv(xv)),
 * each a causal depthwise conv of kernel 4 along t exactly as m2rnn_conv_silu_bf16 computes
 * it (same fp32 operations, the result rounded to bf16), so y and H_T are bit-identical to
 * m2rnn_conv_silu_bf16 on each projection followed by m2rnn_forward_bf16_qk.  The convolved
 * q, k, v are never written to memory.
 *   xq, xk  [B, T, Nqk, K] bf16, raw projections; conv taps wq, wk [Nqk*K][4] float32
 *   xv      [B, T, N, V] bf16; taps wv [N*V][4]
 *   bq, bk, bv: biases [Nqk*K] / [N*V] float32, or NULL for zero
 * Other arguments and errors as m2rnn_forward_bf16_qk, plus INVALID_ARG for a null tap
 * pointer (T > 0) or taps not 16-byte aligned.  Runs on the eight-row kernels, so it takes
 * K in {32, 64} and V in {16, 32, 48, 64} (UNSUPPORTED otherwise).  It saves the memory and
 * traffic of the convolved q, k, v but not time: on GB300 it runs slower than the separate
 * prologue plus forward (6.49 ms against 0.37 + 4.26 ms at B=8, T=16384, N=16, K=V=64).
 */
m2rnn_status m2rnn_forward_conv_bf16(const uint16_t* xq, const uint16_t* xk, const uint16_t* xv,
                                     const float* wq, const float* bq, const float* wk,
                                     const float* bk, const float* wv, const float* bv,
                                     const uint16_t* a, const float* alpha, const float* beta,
                                     const uint16_t* W, const float* w_r, const float* H0,
                                     float* y, float* H_T, int B, int T, int N, int Nqk, int K,
                                     int V, void* stream);

/* Name of a bf16 kernel variant (NULL for an unknown id).  Id 0 is "auto". */
const char* m2rnn_variant_name(int variant);

/* The variant m2rnn_forward_bf16 would pick for this shape on the current
 * device (>0), or 0 if no variant supports it. */
int m2rnn_pick_variant(int B, int T, int N, int K, int V);

/* 1 if bf16 kernel variant `variant` (> 0) can run this shape, else 0. */
int m2rnn_variant_supports(int variant, int B, int T, int N, int K, int V);

/*
 * The balanced schedule of the K = V = 128 tensor-core forward (variant
 * "tcgen05_k128_v128_balanced", chosen automatically when there are more
 * (batch, head) pairs than resident thread blocks).  Lay the B*N pairs' steps
 * end to end (pair p = b*N + n owns positions [p*T, (p+1)*T)); stretch `worker`
 * of `workers` (one thread block each) covers positions [*begin, *end).  A pair
 * cut by a boundary runs its
 * first steps at the start of the later block's stretch and its last steps at
 * the end of the earlier block's stretch (at least 129 of them: the handed-over
 * state travels through that pair's own y rows before they are written).
 * Host-only arithmetic, exposed so the schedule can be checked without a GPU.
 * Returns 0, or -1 for pairs, T or workers < 1, or worker outside [0, workers).
 */
int m2rnn_balanced_stretch(long long pairs, int T, long long workers, long long worker,
                           long long* begin, long long* end);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: M2RNN_ERR_TIMEOUT if a kernel's bounded wait gave up since the last
 * call, M2RNN_ERR_CUDA if the synchronisation itself failed, else M2RNN_OK.
 */
m2rnn_status m2rnn_stream_status(void* stream);

/* Static, human-readable name of a status code. */
const char* m2rnn_status_string(m2rnn_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int m2rnn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* M2RNN_H */
