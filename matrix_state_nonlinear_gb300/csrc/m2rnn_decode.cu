// m2rnn_decode.cu — one decode step of the M²RNN recurrence (T = 1, state in / state
// out), bf16 operands, fp32 state, for serving with a fixed-size recurrent state.
//
// Per (batch b, head n) pair, the notes' Sec. 2.1 Eq. (10)-(12) and Sec. 2.2 Eq. (17)
// for a single token:
//   f = exp(-alpha softplus(a + beta)),  Z = tanh(H W + k v^T),
//   H' = f H + (1 - f) Z,  y = H'^T q + w_r ⊙ v.
// The step's arithmetic is the pipelined forward kernel's step, operation for
// operation: rank-1 term k v^T as the accumulator's initial value, bf16(H) W as
// m16n8k16 MMAs in ascending k-tile order, MUFU tanh, the same lerp, and the same
// readout reduction (per-warp shuffle reduce-scatter, then w_r ⊙ v plus the warps'
// partials in warp order).  T decode steps therefore reproduce a T-step forward pass
// bit for bit.
//
// No TMA, no producer warp, no pipelining: one block per pair, K / 16 warps; each
// warp loads its 16 state rows straight from global memory into registers, and the
// block stages W through shared memory for the B fragments.  The
// state update may be in place (H_in == H_out): every element is read and written
// by the same thread.  Large batches are bound by HBM traffic (the state is read and
// written once); small ones by launch latency.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kMaxWarps = 8;  // K <= 128

// MAXW: the most warps a launch uses (K / 16 <= MAXW).  Four-warp launches (K <= 64) with
// V <= 64 are register-capped so that six blocks fit on an SM: more state loads in flight.
// V = 128 keeps twice the state and accumulator per thread and is not capped.
template <int VT, int MAXW>
__global__ void __launch_bounds__(32 * MAXW, (MAXW <= 4 && VT <= 4) ? 6 : 1)
    decode_bf16_mma(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                    const uint16_t* __restrict__ v, const uint16_t* __restrict__ a,
                    const float* __restrict__ alpha, const float* __restrict__ beta,
                    const uint16_t* __restrict__ W, const float* __restrict__ w_r,
                    const float* H_in, float* H_out, float* __restrict__ y, int N, int Nqk, int K) {
  constexpr int V = 16 * VT, NT = 2 * VT, M = 4 * VT;
  __shared__ __align__(16) float ypart[MAXW][V];
  const int nw = K / 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  const size_t qrow = (size_t)b * Nqk + (Nqk == 1 ? 0 : n);
  const size_t row = (size_t)b * N + n;

  // W through shared memory: 16-byte coalesced loads, then the B fragments by
  // ldmatrix.trans (rows padded by 16 bytes so the eight row addresses of each 8 x 8
  // tile fall in distinct banks).
  constexpr int WS = V + 8;  // padded row length (bf16 elements)
  __shared__ __align__(16) uint16_t wsm[V * WS];
  const uint16_t* Wn = W + (size_t)n * V * V;
  for (int e = threadIdx.x; e < V * V / 8; e += blockDim.x) {
    const int r = e / (V / 8), ch = e - r * (V / 8);
    *reinterpret_cast<uint4*>(wsm + r * WS + 8 * ch) =
        *reinterpret_cast<const uint4*>(Wn + r * V + 8 * ch);
  }
  float2 h[NT][2];
  const float* hin = H_in ? H_in + (size_t)pair * K * V : nullptr;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    h[nt][0] = hin ? *reinterpret_cast<const float2*>(hin + (size_t)r0 * V + 8 * nt + 2 * c)
                   : make_float2(0.f, 0.f);
    h[nt][1] = hin ? *reinterpret_cast<const float2*>(hin + (size_t)r1 * V + 8 * nt + 2 * c)
                   : make_float2(0.f, 0.f);
  }
  __syncthreads();
  const int lr = lane & 7, lq = lane >> 3;
  const float2 fg = gate_fg(bf16_bits_to_float(a[row]), alpha[n], beta[n]);
  const float2 ff = make_float2(fg.x, fg.x), gg = make_float2(fg.y, fg.y);

  // P = k v^T + bf16(H) W
  float2 acc[NT][2];
  {
    const float kv0 = bf16_bits_to_float(k[qrow * K + r0]);
    const float kv1 = bf16_bits_to_float(k[qrow * K + r1]);
    const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 vv =
          bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(v + row * V + 8 * nt + 2 * c));
      acc[nt][0] = mul2(k0, vv);
      acc[nt][1] = mul2(k1, vv);
    }
  }
#pragma unroll
  for (int kt = 0; kt < VT; ++kt) {
    uint32_t af[4];
    af[0] = pack_bf16x2(h[2 * kt][0].x, h[2 * kt][0].y);
    af[1] = pack_bf16x2(h[2 * kt][1].x, h[2 * kt][1].y);
    af[2] = pack_bf16x2(h[2 * kt + 1][0].x, h[2 * kt + 1][0].y);
    af[3] = pack_bf16x2(h[2 * kt + 1][1].x, h[2 * kt + 1][1].y);
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {  // B fragments of n-tiles 2 np, 2 np + 1
      uint32_t wb[4];
      ldmatrix_x4_trans(wb, wsm + (16 * kt + lr + 8 * (lq & 1)) * WS + 16 * np + 8 * (lq >> 1));
      mma2(acc[2 * np], af, wb[0], wb[1]);
      mma2(acc[2 * np + 1], af, wb[2], wb[3]);
    }
  }
  // H' = f H + (1 - f) tanh(P)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float2 z = make_float2(tanh_mufu(acc[nt][r].x), tanh_mufu(acc[nt][r].y));
      h[nt][r] = fma2(gg, z, mul2(ff, h[nt][r]));
    }
  float* hout = H_out ? H_out + (size_t)pair * K * V : nullptr;
  if (hout) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(hout + (size_t)r0 * V + 8 * nt + 2 * c) = h[nt][0];
      *reinterpret_cast<float2*>(hout + (size_t)r1 * V + 8 * nt + 2 * c) = h[nt][1];
    }
  }
  // y = H'^T q + w_r ⊙ v: q-weighted sums of this thread's two rows, reduce-scattered
  // over the warp's 8 row groups (same stages and order as the forward kernel).
  const float qv0 = bf16_bits_to_float(q[qrow * K + r0]);
  const float qv1 = bf16_bits_to_float(q[qrow * K + r1]);
  const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
  float p[M];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float2 pp = fma2(q1, h[nt][1], mul2(q0, h[nt][0]));
    p[2 * nt] = pp.x;
    p[2 * nt + 1] = pp.y;
  }
#pragma unroll
  for (int stg = 0; stg < 3; ++stg) {
    const int mask = 16 >> stg;
    const int half = M >> (stg + 1);
    if (half >= 1) {
      const bool up = (lane & mask) != 0;
#pragma unroll
      for (int i = 0; i < (half >= 1 ? half : 1); ++i) {
        const float send = up ? p[i] : p[i + half];
        const float keep = up ? p[i + half] : p[i];
        p[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
      }
    } else {
      p[0] += __shfl_xor_sync(0xffffffffu, p[0], mask);
    }
  }
  if constexpr (M >= 8) {
    constexpr int cnt = M / 8;
#pragma unroll
    for (int i = 0; i < cnt; ++i) {
      const int m = cnt * g + i;
      ypart[warp][8 * (m >> 1) + 2 * c + (m & 1)] = p[i];
    }
  } else {
    if ((g & 1) == 0) {
      const int m = g >> 1;
      ypart[warp][8 * (m >> 1) + 2 * c + (m & 1)] = p[0];
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < V; j += blockDim.x) {
    const uint16_t vb = v[row * V + j];
    float o = w_r[(size_t)n * V + j] * bf16_bits_to_float(vb);
    for (int w = 0; w < nw; ++w) o += ypart[w][j];
    y[row * V + j] = o;
  }
}

}  // namespace

bool decode_supports(int K, int V) {
  return K >= 16 && K <= 16 * kMaxWarps && K % 16 == 0 &&
         (V == 16 || V == 32 || V == 64 || V == 128);
}

cudaError_t launch_decode_bf16(const Problem& p, cudaStream_t stream) {
  const unsigned grid = (unsigned)p.B * (unsigned)p.N;
  const unsigned threads = 32u * (unsigned)(p.K / 16);
  auto args = [&](auto kern) {
    kern<<<grid, threads, 0, stream>>>((const uint16_t*)p.q, (const uint16_t*)p.k,
                                       (const uint16_t*)p.v, (const uint16_t*)p.a, p.alpha, p.beta,
                                       (const uint16_t*)p.W, p.w_r, p.H0, p.H_T, p.y, p.N, p.Nqk,
                                       p.K);
  };
  const bool small = p.K <= 64;
  switch (p.V) {
    case 16: small ? args(decode_bf16_mma<1, 4>) : args(decode_bf16_mma<1, kMaxWarps>); break;
    case 32: small ? args(decode_bf16_mma<2, 4>) : args(decode_bf16_mma<2, kMaxWarps>); break;
    case 64: small ? args(decode_bf16_mma<4, 4>) : args(decode_bf16_mma<4, kMaxWarps>); break;
    case 128: small ? args(decode_bf16_mma<8, 4>) : args(decode_bf16_mma<8, kMaxWarps>); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace m2rnn
