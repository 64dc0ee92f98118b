// m2rnn_bwd_f32.cu — backward pass of the M²RNN recurrence (SIMT, fp32 arithmetic),
// any 1 <= K, V <= 128, inputs in fp32 or bf16.
//
// The reverse scan of the M²RNN study notes, Sec. 2.7, per (batch b, head n) pair,
// with u_t = dL/dy_t and C_T = dL/dH_T:
//   Z_t     = tanh(H_{t-1} W + k_t v_t^T)          (recomputed from the kept H_{t-1})
//   R_t     = C_t + q_t u_t^T
//   D_t     = ((1 - f_t) R_t) ⊙ (1 - Z_t ⊙ Z_t)
//   C_{t-1} = f_t R_t + D_t W^T
//   dL/df_t = <R_t, H_{t-1} - Z_t>,  dW += H_{t-1}^T D_t,
//   dk_t = D_t v_t,  dv_t = D_t^T k_t + w_r ⊙ u_t,  dq_t = H_t u_t,
// and through the gate of Eq. (13)/(17), x = a + beta:
//   da_t = dL/df_t · (-alpha f sigmoid(x)),  dalpha += dL/df_t · (-f softplus(x)),
//   dbeta += da_t,  dw_r += u_t ⊙ v_t.
// The states H_t come from the training forward (kept in HBM, the notes' Sec. 2.6):
// fp32 on the fp32 path, the bf16-rounded state on the bf16 path.
//
// One thread block per pair.  W and D_t live in shared memory; the running state
// gradient C and the pair's partial sums of dW, dw_r, dalpha, dbeta live in the
// caller's workspace (each element owned by one thread, so no atomics).  A second
// kernel sums the partials over the batch in a fixed order, so results are
// deterministic.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"

namespace m2rnn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld_in(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const uint16_t* p, size_t i) {
  return __uint_as_float((uint32_t)p[i] << 16);
}

// The value the kept state would hold: itself for fp32 states, its bf16 rounding
// (round to nearest even, as the tensor-core operand is formed) for bf16 states.
template <typename Th>
__device__ __forceinline__ float round_like(float x);
template <>
__device__ __forceinline__ float round_like<float>(float x) { return x; }
template <>
__device__ __forceinline__ float round_like<uint16_t>(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = x;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];  // fixed order
    red[kThreads / 32] = s;
  }
  __syncthreads();
  return red[kThreads / 32];
}

template <typename Tin, typename Th>
__global__ void __launch_bounds__(kThreads)
    bwd_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                    const Tin* __restrict__ a, const float* __restrict__ alpha,
                    const float* __restrict__ beta, const Tin* __restrict__ W,
                    const float* __restrict__ w_r, const float* __restrict__ H0,
                    const Th* __restrict__ Hs, const float* __restrict__ dy,
                    const float* __restrict__ dH_T, float* __restrict__ dq, float* __restrict__ dk,
                    float* __restrict__ dv, float* __restrict__ da, float* __restrict__ dH0,
                    float* __restrict__ ws, float* __restrict__ dqk_heads, int T, int N, int K,
                    int V, int Nqk) {
  extern __shared__ float smem[];
  float* Ws = smem;                 // [V][V]
  float* Ds = Ws + V * V;           // [K][V]  D_t
  float* ks = Ds + K * V;           // [K]
  float* qs = ks + K;               // [K]
  float* vs = qs + K;               // [V]
  float* us = vs + V;               // [V]     u_t = dy_t
  float* gate = us + V;             // f, 1 - f, sigmoid(x), softplus(x)
  float* red = gate + 4;            // [kThreads / 32 + 1]

  const int pair = blockIdx.x;
  const int b = pair / N, n = pair - (pair / N) * N;
  const int tid = threadIdx.x;
  const int KV = K * V, VV = V * V;
  float* Cw = ws + (size_t)pair * backward_pair_floats(K, V);  // C (K V)
  float* dWp = Cw + KV;                                        // dW partial (V V)
  float* dwr_p = dWp + VV;                                     // dw_r partial (V)
  float* ab_p = dwr_p + V;                                     // dalpha, dbeta partials

  for (int e = tid; e < VV; e += kThreads) {
    Ws[e] = ld_in(W, (size_t)n * VV + e);
    dWp[e] = 0.f;
  }
  for (int e = tid; e < KV; e += kThreads) Cw[e] = dH_T ? dH_T[(size_t)pair * KV + e] : 0.f;
  const float al = alpha[n], be = beta[n];
  const float wr = tid < V ? w_r[(size_t)n * V + tid] : 0.f;
  float dwr_acc = 0.f, dal_acc = 0.f, dbe_acc = 0.f;
  const bool shared_qk = Nqk == 1 && N > 1;

  for (int t = T - 1; t >= 0; --t) {
    const size_t row = ((size_t)b * T + t) * N + n;
    const size_t qrow = ((size_t)b * T + t) * Nqk + (Nqk == 1 ? 0 : n);
    for (int i = tid; i < K; i += kThreads) {
      ks[i] = ld_in(k, qrow * K + i);
      qs[i] = ld_in(q, qrow * K + i);
    }
    for (int j = tid; j < V; j += kThreads) {
      vs[j] = ld_in(v, row * V + j);
      us[j] = dy[row * V + j];
    }
    if (tid == 0) {  // gate of Eq. (13)/(17) and its derivative factors
      const float x = ld_in(a, row) + be;
      const float ex = expf(-fabsf(x));
      const float sp = fmaxf(x, 0.f) + log1pf(ex);
      gate[0] = expf(-al * sp);
      gate[1] = -expm1f(-al * sp);
      gate[2] = x >= 0.f ? 1.f / (1.f + ex) : ex / (1.f + ex);
      gate[3] = sp;
    }
    __syncthreads();
    const float f = gate[0], g = gate[1];
    // H_{t-1} from the kept states (H_0 itself for t = 0; the bf16 path keeps the
    // bf16-rounded states and rounds H_0 the same way), and H_t.
    const Th* Hp = t > 0 ? Hs + ((size_t)pair * T + t - 1) * KV : nullptr;
    const float* H0p = H0 ? H0 + (size_t)pair * KV : nullptr;
    const Th* Hc = Hs + ((size_t)pair * T + t) * KV;
    auto hprev = [&](size_t e) -> float {
      if (Hp) return ld_in(Hp, e);
      return H0p ? round_like<Th>(H0p[e]) : 0.f;
    };
    const bool have_prev = Hp || H0p;

    // Phase 1: Z_t, R_t, D_t and the partial <R_t, H_{t-1} - Z_t>.
    float dfl = 0.f;
    for (int e = tid; e < KV; e += kThreads) {
      const int i = e / V, j = e - (e / V) * V;
      float acc = ks[i] * vs[j];  // same order as the fp32 forward: rank-1, then l = 0..V-1
      if (have_prev)
        for (int l = 0; l < V; ++l) acc = fmaf(hprev((size_t)i * V + l), Ws[l * V + j], acc);
      const float Z = tanhf(acc);
      const float R = Cw[e] + qs[i] * us[j];
      Ds[e] = g * R * (1.f - Z * Z);
      Cw[e] = R;
      dfl += R * (hprev(e) - Z);
    }
    const float df = block_sum(dfl, red);  // also orders Ds writes before the reads below

    // Phase 2: C_{t-1} = f R_t + D_t W^T (same element ownership as phase 1).
    for (int e = tid; e < KV; e += kThreads) {
      const int i = e / V, l = e - (e / V) * V;
      const float* drow = Ds + i * V;
      const float* wrow = Ws + l * V;
      float acc = 0.f;
      for (int j = 0; j < V; ++j) acc = fmaf(drow[j], wrow[j], acc);
      Cw[e] = fmaf(f, Cw[e], acc);
    }
    // dW partial += H_{t-1}^T D_t.
    if (have_prev) {
      for (int e = tid; e < VV; e += kThreads) {
        const int l = e / V, j = e - (e / V) * V;
        float acc = dWp[e];
        for (int i = 0; i < K; ++i) acc = fmaf(hprev((size_t)i * V + l), Ds[i * V + j], acc);
        dWp[e] = acc;
      }
    }
    // dk_t = D_t v_t, dq_t = H_t u_t (per head; summed over heads later when shared).
    for (int i = tid; i < K; i += kThreads) {
      float sk = 0.f, sq = 0.f;
      for (int j = 0; j < V; ++j) {
        sk = fmaf(Ds[i * V + j], vs[j], sk);
        sq = fmaf(ld_in(Hc, (size_t)i * V + j), us[j], sq);
      }
      if (shared_qk) {
        dqk_heads[row * K + i] = sq;
        dqk_heads[(size_t)gridDim.x * T * K + row * K + i] = sk;
      } else {
        dq[row * K + i] = sq;
        dk[row * K + i] = sk;
      }
    }
    // dv_t = D_t^T k_t + w_r ⊙ u_t; dw_r partial += u_t ⊙ v_t.
    for (int j = tid; j < V; j += kThreads) {
      float s = 0.f;
      for (int i = 0; i < K; ++i) s = fmaf(Ds[i * V + j], ks[i], s);
      dv[row * V + j] = s + wr * us[j];
      dwr_acc = fmaf(us[j], vs[j], dwr_acc);
    }
    if (tid == 0) {
      const float d_a = df * (-al * f * gate[2]);
      da[row] = d_a;
      dal_acc += df * (-f * gate[3]);
      dbe_acc += d_a;
    }
    __syncthreads();  // io and Ds are rewritten by the next step
  }
  if (dH0)
    for (int e = tid; e < KV; e += kThreads) dH0[(size_t)pair * KV + e] = Cw[e];
  if (tid < V) dwr_p[tid] = dwr_acc;
  if (tid == 0) {
    ab_p[0] = dal_acc;
    ab_p[1] = dbe_acc;
  }
}

// Sum the per-pair partials over the batch: one block per head.
__global__ void __launch_bounds__(kThreads)
    bwd_reduce_params(const float* __restrict__ ws, float* __restrict__ dW,
                      float* __restrict__ dw_r, float* __restrict__ dalpha,
                      float* __restrict__ dbeta, int B, int N, int K, int V) {
  const int n = blockIdx.x;
  const size_t stride = backward_pair_floats(K, V);
  const int KV = K * V, VV = V * V;
  for (int e = threadIdx.x; e < VV + V + 2; e += blockDim.x) {
    float s = 0.f;
    for (int b = 0; b < B; ++b) s += ws[((size_t)b * N + n) * stride + KV + e];
    if (e < VV)
      dW[(size_t)n * VV + e] = s;
    else if (e < VV + V)
      dw_r[(size_t)n * V + e - VV] = s;
    else if (e == VV + V)
      dalpha[n] = s;
    else
      dbeta[n] = s;
  }
}

// Shared q, k: dq[b,t,0,:] = sum over heads of the per-head dq (same for dk).
__global__ void __launch_bounds__(kThreads)
    bwd_reduce_heads(const float* __restrict__ heads, float* __restrict__ dq,
                     float* __restrict__ dk, size_t BT, int N, int K, size_t half) {
  const size_t total = BT * K;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t bt = idx / K, i = idx - (idx / K) * K;
    float sq = 0.f, sk = 0.f;
    for (int n = 0; n < N; ++n) {
      sq += heads[(bt * N + n) * K + i];
      sk += heads[half + (bt * N + n) * K + i];
    }
    dq[idx] = sq;
    dk[idx] = sk;
  }
}

template <typename Tin, typename Th>
cudaError_t launch_simt(const BackwardProblem& p, cudaStream_t stream) {
  const size_t smem = sizeof(float) * ((size_t)p.V * p.V + (size_t)p.K * p.V + 2 * p.K +
                                       2 * p.V + 4 + kThreads / 32 + 1);
  cudaError_t err = cudaFuncSetAttribute(bwd_simt_kernel<Tin, Th>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned pairs = (unsigned)p.B * (unsigned)p.N;
  float* heads = p.ws + (size_t)p.B * p.N * backward_pair_floats(p.K, p.V);
  bwd_simt_kernel<Tin, Th><<<pairs, kThreads, smem, stream>>>(
      (const Tin*)p.q, (const Tin*)p.k, (const Tin*)p.v, (const Tin*)p.a, p.alpha, p.beta,
      (const Tin*)p.W, p.w_r, p.H0, (const Th*)p.Hs, p.dy, p.dH_T, p.dq, p.dk, p.dv, p.da, p.dH0, p.ws, heads,
      p.T, p.N, p.K, p.V, p.Nqk);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_reduce(const BackwardProblem& p, cudaStream_t stream) {
  bwd_reduce_params<<<(unsigned)p.N, kThreads, 0, stream>>>(p.ws, p.dW, p.dw_r, p.dalpha, p.dbeta,
                                                             p.B, p.N, p.K, p.V);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (p.Nqk == 1 && p.N > 1 && p.T > 0) {
    const size_t BT = (size_t)p.B * p.T;
    const size_t half = BT * p.N * p.K;
    const float* heads = p.ws + (size_t)p.B * p.N * backward_pair_floats(p.K, p.V);
    const size_t blocks = (BT * p.K + kThreads - 1) / kThreads;
    bwd_reduce_heads<<<(unsigned)(blocks < 4096 ? blocks : 4096), kThreads, 0, stream>>>(
        heads, p.dq, p.dk, BT, p.N, p.K, half);
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t launch_bwd_f32(const BackwardProblem& p, cudaStream_t stream) {
  cudaError_t err = launch_simt<float, float>(p, stream);
  return err == cudaSuccess ? launch_bwd_reduce(p, stream) : err;
}

cudaError_t launch_bwd_simt_bf16(const BackwardProblem& p, cudaStream_t stream) {
  cudaError_t err = launch_simt<uint16_t, uint16_t>(p, stream);
  return err == cudaSuccess ? launch_bwd_reduce(p, stream) : err;
}

}  // namespace m2rnn
