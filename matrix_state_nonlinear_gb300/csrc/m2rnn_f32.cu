// m2rnn_f32.cu — fp32-operand forward recurrence (SIMT), any 1 <= K, V <= 128.
//
// Computes, per (batch b, head n) pair, the M²RNN recurrence of the M²RNN study
// notes (Sec. 2.1 Eq. (10)-(12), Sec. 2.2 Eq. (13)/(17)):
//   f_t = exp(-alpha_n softplus(a_t + beta_n)),  Z_t = tanh(H_{t-1} W + k_t v_t^T),
//   H_t = f_t H_{t-1} + (1 - f_t) Z_t,           y_t = H_t^T q_t + w_r ⊙ v_t.
// One thread block per pair (the notes' Sec. 2.6 work unit); W and two copies of
// the K x V state live in shared memory; every element is fp32 and tanh / exp /
// log1p are the accurate CUDA math functions.  This path serves small problems
// and the 1e-4 parity bar; the tensor-core paths carry the large workloads.
// With a non-null Hs the kernel also keeps every step's state, Hs[b][n][t] = H_t,
// for the backward pass (the notes' Sec. 2.6: states are kept, then scanned in
// reverse).
#include "m2rnn_internal.h"

namespace m2rnn {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, const float* __restrict__ a,
                   const float* __restrict__ alpha, const float* __restrict__ beta,
                   const float* __restrict__ W, const float* __restrict__ w_r,
                   const float* H0, float* __restrict__ y, float* H_T, float* __restrict__ Hs,
                   int T, int N, int K, int V, int Nqk) {
  extern __shared__ float smem[];
  float* Ws = smem;              // [V][V]
  float* Hbuf = Ws + V * V;      // [2][K][V]
  float* io = Hbuf + 2 * K * V;  // [2][K (k) + K (q) + V (v) + 2 (f, g)]
  const int io_stride = 2 * K + V + 2;

  const int pair = blockIdx.x;
  const int b = pair / N, n = pair % N;
  const int tid = threadIdx.x;
  const int KV = K * V;

  for (int e = tid; e < V * V; e += kThreads) Ws[e] = W[(size_t)n * V * V + e];
  const float* H0p = H0 ? H0 + (size_t)pair * KV : nullptr;
  for (int e = tid; e < KV; e += kThreads) Hbuf[e] = H0p ? H0p[e] : 0.f;
  const float al = alpha[n], be = beta[n];

  int cur = 0;
  for (int t = 0; t < T; ++t) {
    float* st = io + (t & 1) * io_stride;
    float* ks = st;
    float* qs = st + K;
    float* vs = st + 2 * K;
    const size_t row = ((size_t)b * T + t) * N + n;
    const size_t qrow = ((size_t)b * T + t) * Nqk + (Nqk == 1 ? 0 : n);  // shared q, k: head 0
    for (int i = tid; i < K; i += kThreads) {
      ks[i] = k[qrow * K + i];
      qs[i] = q[qrow * K + i];
    }
    for (int j = tid; j < V; j += kThreads) vs[j] = v[row * V + j];
    if (tid == 0) {
      // Eq. (17): f = exp(-alpha softplus(a + beta)); 1 - f via expm1 for accuracy.
      const float x = a[row] + be;
      const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
      st[2 * K + V] = expf(-al * sp);
      st[2 * K + V + 1] = -expm1f(-al * sp);
    }
    __syncthreads();
    const float f = st[2 * K + V], g = st[2 * K + V + 1];
    const float* Hc = Hbuf + cur * KV;
    float* Hn = Hbuf + (cur ^ 1) * KV;
    for (int e = tid; e < KV; e += kThreads) {
      const int i = e / V, j = e - (e / V) * V;
      float acc = ks[i] * vs[j];                       // rank-1 write k_t v_t^T
      const float* hrow = Hc + i * V;
      for (int l = 0; l < V; ++l) acc = fmaf(hrow[l], Ws[l * V + j], acc);  // H_{t-1} W
      const float hn = f * Hc[e] + g * tanhf(acc);     // Eq. (10)-(11)
      Hn[e] = hn;
      if (Hs) Hs[((size_t)pair * T + t) * KV + e] = hn;
    }
    __syncthreads();
    for (int j = tid; j < V; j += kThreads) {          // Eq. (12), sum over the K rows
      float s = 0.f;
      for (int i = 0; i < K; ++i) s = fmaf(Hn[i * V + j], qs[i], s);
      y[row * V + j] = s + w_r[(size_t)n * V + j] * vs[j];
    }
    cur ^= 1;
  }
  if (H_T) {
    __syncthreads();
    const float* Hc = Hbuf + cur * KV;
    for (int e = tid; e < KV; e += kThreads) H_T[(size_t)pair * KV + e] = Hc[e];
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const Problem& p, cudaStream_t stream) {
  const size_t smem =
      sizeof(float) * ((size_t)p.V * p.V + 2ull * p.K * p.V + 2ull * (2 * p.K + p.V + 2));
  cudaError_t err =
      cudaFuncSetAttribute(fwd_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)p.B * (unsigned)p.N;
  fwd_f32_kernel<<<grid, kThreads, smem, stream>>>(
      (const float*)p.q, (const float*)p.k, (const float*)p.v, (const float*)p.a, p.alpha, p.beta,
      (const float*)p.W, p.w_r, p.H0, p.y, p.H_T, static_cast<float*>(p.Hs), p.T, p.N, p.K, p.V,
      p.Nqk);
  return cudaGetLastError();
}

}  // namespace m2rnn
