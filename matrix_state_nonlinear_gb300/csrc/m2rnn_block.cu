// m2rnn_block.cu — the M²RNN block's elementwise stages around the recurrence
// (the notes' Sec. 2.3, Eq. (14)-(23)), as memory-bound fused kernels:
//
//  * prologue, applied to each of the q, k, v projections:
//      out[b,t,c] = SiLU( bias[c] + sum_{j=0..3} w[c][j] * x[b, t-3+j, c] ),
//    a depthwise causal Conv1D of kernel 4 (x at negative t is zero) followed by SiLU;
//  * epilogue, on the recurrence's readout y and the gate projection g_pre:
//      z = y ⊙ SiLU(g_pre),   out = w_norm ⊙ z / sqrt(mean(z^2) + eps),
//    the output gate first, then an RMSNorm whose statistic spans the whole token
//    (all heads; one scalar per token, as the notes' Appendix C uses it).
// The projections (W_q, W_k, W_v, W_g, W_f, W_o) are plain GEMMs outside.
//
// Both kernels read and write every element once with 16-byte vector accesses; the
// arithmetic is fp32 and the results are rounded to bf16 (round to nearest even),
// ready to be the next GEMM's operand.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kTaps = 4;
constexpr int kConvRows = 64;   // time steps per thread (sliding window)
constexpr int kConvThreads = 128;

// SiLU with the fast exponential and division intrinsics: a few ulp of fp32, far below
// the bf16 rounding of the result (for x -> -inf the quotient x / inf is 0).
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.f + __expf(-x)); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x);
  f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y);
  f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z);
  f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w);
  f[7] = bf16_hi(u.w);
}

// One thread: 8 consecutive channels over kConvRows consecutive steps of one batch
// row, keeping the last three inputs of each channel in registers.
__global__ void __launch_bounds__(kConvThreads)
    conv_silu_kernel(const uint16_t* __restrict__ x, const float* __restrict__ w,
                     const float* __restrict__ bias, uint16_t* __restrict__ out, int B, int T,
                     int C, int groups, int tiles) {
  // Consecutive threads take consecutive channel groups of the same time row (coalesced).
  const long long id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int cg = (int)(id % groups);
  const long long rest = id / groups;
  const int tile = (int)(rest % tiles);
  const long long b = rest / tiles;
  if (b >= B) return;
  const int c0 = 8 * cg;
  float wt[8][kTaps], bs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 wv = *reinterpret_cast<const float4*>(w + (size_t)(c0 + i) * kTaps);
    wt[i][0] = wv.x;
    wt[i][1] = wv.y;
    wt[i][2] = wv.z;
    wt[i][3] = wv.w;
    bs[i] = bias ? bias[c0 + i] : 0.f;
  }
  const int t0 = tile * kConvRows;
  const int t1 = min(T, t0 + kConvRows);
  const uint16_t* xb = x + (size_t)b * T * C + c0;
  uint16_t* ob = out + (size_t)b * T * C + c0;
  float h1[8], h2[8], h3[8];  // x[t-1], x[t-2], x[t-3]
  auto load = [&](int t, float (&f)[8]) {
    if (t >= 0) {
      unpack8(*reinterpret_cast<const uint4*>(xb + (size_t)t * C), f);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
  };
  load(t0 - 1, h1);
  load(t0 - 2, h2);
  load(t0 - 3, h3);
#pragma unroll 4
  for (int t = t0; t < t1; ++t) {
    float cur[8];
    load(t, cur);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      float s0 = bs[i], s1 = bs[i + 1];
      s0 = fmaf(wt[i][0], h3[i], s0);
      s0 = fmaf(wt[i][1], h2[i], s0);
      s0 = fmaf(wt[i][2], h1[i], s0);
      s0 = fmaf(wt[i][3], cur[i], s0);
      s1 = fmaf(wt[i + 1][0], h3[i + 1], s1);
      s1 = fmaf(wt[i + 1][1], h2[i + 1], s1);
      s1 = fmaf(wt[i + 1][2], h1[i + 1], s1);
      s1 = fmaf(wt[i + 1][3], cur[i + 1], s1);
      o[i / 2] = pack_bf16x2(silu_f(s0), silu_f(s1));
    }
    *reinterpret_cast<uint4*>(ob + (size_t)t * C) = make_uint4(o[0], o[1], o[2], o[3]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h3[i] = h2[i];
      h2[i] = h1[i];
      h1[i] = cur[i];
    }
  }
}

constexpr int kNormWarps = 8;

// One warp per token row: pass 1 forms z = y ⊙ SiLU(g) and sum(z^2); pass 2 recomputes z
// (the row is still in L1/L2) and writes the normalised bf16 output.
__global__ void __launch_bounds__(32 * kNormWarps)
    gate_rmsnorm_kernel(const float* __restrict__ y, const uint16_t* __restrict__ g_pre,
                        const float* __restrict__ w_norm, float eps, uint16_t* __restrict__ out,
                        long long rows, int D) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * kNormWarps + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* yr = y + r * D;
  const uint16_t* gr = g_pre + r * D;
  uint16_t* orow = out + r * D;
  auto zvals = [&](int e, float (&z)[8]) {
    const float4 y0 = *reinterpret_cast<const float4*>(yr + e);
    const float4 y1 = *reinterpret_cast<const float4*>(yr + e + 4);
    float gf[8];
    unpack8(*reinterpret_cast<const uint4*>(gr + e), gf);
    z[0] = y0.x * silu_f(gf[0]);
    z[1] = y0.y * silu_f(gf[1]);
    z[2] = y0.z * silu_f(gf[2]);
    z[3] = y0.w * silu_f(gf[3]);
    z[4] = y1.x * silu_f(gf[4]);
    z[5] = y1.y * silu_f(gf[5]);
    z[6] = y1.z * silu_f(gf[6]);
    z[7] = y1.w * silu_f(gf[7]);
  };
  float ss = 0.f;
  for (int e = 8 * lane; e < D; e += 256) {
    float z[8];
    zvals(e, z);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(z[i], z[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)D + eps);
  for (int e = 8 * lane; e < D; e += 256) {
    float z[8];
    zvals(e, z);
    const float4 w0 = *reinterpret_cast<const float4*>(w_norm + e);
    const float4 w1 = *reinterpret_cast<const float4*>(w_norm + e + 4);
    const uint4 o = make_uint4(pack_bf16x2(w0.x * z[0] * inv, w0.y * z[1] * inv),
                               pack_bf16x2(w0.z * z[2] * inv, w0.w * z[3] * inv),
                               pack_bf16x2(w1.x * z[4] * inv, w1.y * z[5] * inv),
                               pack_bf16x2(w1.z * z[6] * inv, w1.w * z[7] * inv));
    *reinterpret_cast<uint4*>(orow + e) = o;
  }
}

}  // namespace

cudaError_t launch_conv_silu(const uint16_t* x, const float* w, const float* bias, uint16_t* out,
                             int B, int T, int C, cudaStream_t stream) {
  const int groups = C / 8;
  const int tiles = (T + kConvRows - 1) / kConvRows;
  const long long total = (long long)groups * tiles * B;
  const unsigned blocks = (unsigned)((total + kConvThreads - 1) / kConvThreads);
  conv_silu_kernel<<<blocks, kConvThreads, 0, stream>>>(x, w, bias, out, B, T, C, groups, tiles);
  return cudaGetLastError();
}

cudaError_t launch_gate_rmsnorm(const float* y, const uint16_t* g_pre, const float* w_norm,
                                float eps, uint16_t* out, long long rows, int D,
                                cudaStream_t stream) {
  const unsigned blocks = (unsigned)((rows + kNormWarps - 1) / kNormWarps);
  gate_rmsnorm_kernel<<<blocks, 32 * kNormWarps, 0, stream>>>(y, g_pre, w_norm, eps, out, rows, D);
  return cudaGetLastError();
}

}  // namespace m2rnn
