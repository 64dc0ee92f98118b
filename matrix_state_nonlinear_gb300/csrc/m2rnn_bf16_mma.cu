// m2rnn_bf16_mma.cu — bf16-operand / fp32-state forward recurrence on the warp-level
// tensor-core MMA (mma.sync m16n8k16), one thread block per (batch, head) pair.
//
// The recurrence is Eq. (10)-(12) and (13)/(17) of the M²RNN study notes ("M²RNN:
// 矩阵状态非线性 RNN 的容量、表达力与系统代价", Sec. 2.1-2.2).  Sec. 2.6 of the notes
// describes the work split this kernel keeps: each (b, n) pair is an independent
// unit that holds H and W on chip and streams q, k, v and the gate in time order.
//
// Mapping.  Rows of H evolve independently given W and f (W mixes value columns,
// not key rows; notes Sec. 1.2), so warp w owns rows 16w .. 16w+15 of H for the
// whole sequence and never synchronises with the other warps inside a step:
//   * H (fp32) lives in registers in the m16n8 accumulator layout;
//   * the accumulator fragments of n-tiles 2j and 2j+1 are exactly the A
//     fragment of k-tile j, so the next step's bf16 operand is packed in
//     registers with no shared-memory trip;
//   * W (bf16) is the B operand: kept in registers for V <= 64, else read from
//     padded shared memory with ldmatrix.trans each step;
//   * the rank-1 term k_t v_t^T initialises the accumulators, then
//     P = k v^T + H_{t-1} W, Z = tanh(P) (MUFU), H = f H + (1 - f) Z;
//   * the readout H_t^T q_t is a q-weighted sum of each thread's two rows,
//     reduce-scattered over the 8 row groups of the warp with shuffles and
//     written as per-warp partials; partials of all warps, plus w_r ⊙ v_t, are
//     summed once per chunk and stored to y as float4.
// Inputs q, k, v arrive in chunks of Tc steps by TMA (double-buffered, mbarrier
// completion, bounded waits); gate logits a are prefetched into registers one
// chunk ahead and turned into (f, 1 - f) in shared memory.
//
// Any 1 <= K <= 128 and any V = 16, 32, ..., 128.  K rows are padded to Kp, the next
// multiple of 16 (one warp per 16 rows).  Padded rows start at zero and get a zero k and
// q, so their P = 0 W + 0 stays 0, tanh(0) = 0 keeps them at 0 for every t, and they add
// nothing to the readout; they are never stored.  With K not a multiple of 16 the q and
// k rows (K * 2 bytes, not a legal TMA stride in general) are staged by plain loads with
// the padding written as zeros; v still comes by TMA.  V whose readout slot count 4 V / 16
// is not a power of two pads the reduce-scatter with zero slots that are never stored.
#include <cuda_bf16.h>

#include <cstring>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

struct SmemLayout {
  int qs, ks, vs, stage_bytes;  // per stage (two stages, `stage_bytes` apart)
  int fg;                       // float2 [2][Tc]   (f, 1 - f)
  int ypart;                    // float  [Kp/16][Tc][V] per-warp readout partials
  int wr;                       // float  [V]
  int Ws;                       // bf16   [V][V + 8] (only when W is not in registers)
  int bar;                      // uint64 [3]
  int total;
};

__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }

// Kp: rows of H including the padding of a ragged K (a multiple of 16).
__host__ __device__ inline SmemLayout make_layout(int Kp, int V, int Tc, bool wreg) {
  SmemLayout L;
  L.qs = 0;
  L.ks = align128(Tc * Kp * 2);
  L.vs = L.ks + align128(Tc * Kp * 2);
  L.stage_bytes = L.vs + align128(Tc * V * 2);
  int o = 2 * L.stage_bytes;
  L.fg = o;
  o += align128(2 * Tc * 8);
  L.ypart = o;
  o += align128((Kp / 16) * Tc * V * 4);
  L.wr = o;
  o += align128(V * 4);
  L.Ws = o;
  if (!wreg) o += align128(V * (V + 8) * 2);
  L.bar = o;
  o += 64;
  L.total = o;
  return L;
}

// Eq. (17): f = exp(-alpha softplus(a + beta)); returns (f, 1 - f), 1 - f via expm1.
__device__ __forceinline__ float2 gate_pair(float a, float al, float be) {
  const float x = a + be;
  const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
  const float e = -al * sp;
  return make_float2(expf(e), -expm1f(e));
}

// kCache: also keep every state H_t, as the bf16 A fragments the next step's MMAs use
// (Hs [B N, T, K, V]), for the backward pass.
// kRagged: K is not a multiple of 16; q and k are staged by plain loads (qg, kg) into
// rows of Kp = blockDim.x / 2 with zero padding (the TMA maps tm_q, tm_k are unused).
template <int VT, bool WREG, bool kCache, bool kRagged>
__global__ void __launch_bounds__(256, 1)
    fwd_bf16_mma_rowwarp(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ qg,
                         const uint16_t* __restrict__ kg, const uint16_t* __restrict__ a,
                         const float* __restrict__ alpha, const float* __restrict__ beta,
                         const uint16_t* __restrict__ W, const float* __restrict__ w_r,
                         const float* H0, float* __restrict__ y, float* H_T,
                         uint16_t* __restrict__ Hs, int T, int N, int K, int Tc, int qk_hs,
                         int debug, int* status) {
  constexpr int V = 16 * VT;
  constexpr int NT = 2 * VT;  // n-tiles of 8 columns
  constexpr int M = 4 * VT;   // readout partial sums per thread
  // Reduce-scatter width: M rounded up to a power of two (slots M .. MP-1 stay zero).
  constexpr int MP = M <= 4 ? M : M <= 8 ? 8 : M <= 16 ? 16 : 32;
  constexpr int WS = V + 8;   // padded shared-memory row of W (bank-conflict-free ldmatrix)

  extern __shared__ __align__(128) uint8_t smem[];
  const int Kp = kRagged ? (int)(blockDim.x >> 1) : K;  // rows incl. padding (16 per warp)
  const SmemLayout L = make_layout(Kp, V, Tc, WREG);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int g = lane >> 2, c = lane & 3;
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + Tc - 1) / Tc;

  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  float2* fgs = reinterpret_cast<float2*>(smem + L.fg);
  float* ypart = reinterpret_cast<float*>(smem + L.ypart);
  float* wrs = reinterpret_cast<float*>(smem + L.wr);
  __nv_bfloat16* Ws = reinterpret_cast<__nv_bfloat16*>(smem + L.Ws);
  const float al = alpha[n], be = beta[n];
  const uint32_t stage_tx = (uint32_t)((kRagged ? 0 : 2 * K) + V) * (uint32_t)Tc * 2u;

  auto issue = [&](int cc) {  // one thread: TMA of chunk cc's q, k, v into stage cc & 1
    const int st = cc & 1;
    uint8_t* base = smem + st * L.stage_bytes;
    mbar_arrive_expect_tx(&bar[st], stage_tx);
    if constexpr (!kRagged) {
      tma_load_4d(base + L.qs, &tm_q, &bar[st], 0, n * qk_hs, cc * Tc, b);
      tma_load_4d(base + L.ks, &tm_k, &bar[st], 0, n * qk_hs, cc * Tc, b);
    }
    tma_load_4d(base + L.vs, &tm_v, &bar[st], 0, n, cc * Tc, b);
  };
  // Ragged K, every thread: chunk cc's q and k rows into stage cc & 1, rows K .. Kp-1 and
  // steps past T written as zeros.
  auto stage_qk = [&](int cc) {
    uint16_t* qd = reinterpret_cast<uint16_t*>(smem + (cc & 1) * L.stage_bytes + L.qs);
    uint16_t* kd = reinterpret_cast<uint16_t*>(smem + (cc & 1) * L.stage_bytes + L.ks);
    const size_t heads = qk_hs ? (size_t)N : 1;
    for (int idx = tid; idx < Tc * Kp; idx += nthreads) {
      const int s = idx / Kp, r = idx - s * Kp, t = cc * Tc + s;
      uint16_t qv = 0, kv = 0;
      if (t < T && r < K) {
        const size_t off = (((size_t)b * T + t) * heads + (size_t)n * qk_hs) * K + r;
        qv = qg[off];
        kv = kg[off];
      }
      qd[idx] = qv;
      kd[idx] = kv;
    }
  };

  if (tid == 0) {
    if constexpr (!kRagged) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
    }
    prefetch_tensormap(&tm_v);
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);  // never armed: the forced-timeout test hook waits on it
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int cc = 0; cc < 2 && cc < nchunks; ++cc) issue(cc);
  }
  if constexpr (kRagged)
    for (int cc = 0; cc < 2 && cc < nchunks; ++cc) stage_qk(cc);
  const size_t pair_row = (size_t)b * T;  // (b, t) row index base
  for (int cc = 0; cc < 2 && cc < nchunks; ++cc)
    for (int t = tid; t < Tc; t += nthreads) {
      const int tt = cc * Tc + t;
      const float av = tt < T ? bf16_bits_to_float(a[(pair_row + tt) * N + n]) : 0.f;
      fgs[cc * Tc + t] = gate_pair(av, al, be);
    }
  for (int j = tid; j < V; j += nthreads) wrs[j] = w_r[(size_t)n * V + j];

  // W: B fragments of m16n8k16 (k index = row l of W, n index = column j).
  const uint16_t* Wn = W + (size_t)n * V * V;
  uint32_t wb[WREG ? VT : 1][WREG ? NT : 1][2];
  if constexpr (WREG) {
#pragma unroll
    for (int kt = 0; kt < VT; ++kt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int col = 8 * nt + g;
        const int r = 16 * kt + 2 * c;
        wb[kt][nt][0] = (uint32_t)Wn[r * V + col] | ((uint32_t)Wn[(r + 1) * V + col] << 16);
        wb[kt][nt][1] =
            (uint32_t)Wn[(r + 8) * V + col] | ((uint32_t)Wn[(r + 9) * V + col] << 16);
      }
  } else {
    for (int e = tid; e < V * V / 8; e += nthreads) {  // 16-byte chunks of W rows
      const int r = e / (V / 8), c8 = (e - r * (V / 8)) * 8;
      *reinterpret_cast<uint4*>(Ws + r * WS + c8) =
          *reinterpret_cast<const uint4*>(Wn + (size_t)r * V + c8);
    }
  }

  // H (fp32) in the accumulator layout: rows r0 = 16 warp + g and r1 = r0 + 8,
  // columns 8 nt + 2c and 8 nt + 2c + 1.
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  const bool in0 = r0 < K, in1 = r1 < K;  // false only for the padding rows of a ragged K
  float h[NT][4];
  if (H0) {
    const float* h0p = H0 + (size_t)pair * K * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 u = in0 ? *reinterpret_cast<const float2*>(h0p + (size_t)r0 * V + 8 * nt + 2 * c)
                           : make_float2(0.f, 0.f);
      const float2 w = in1 ? *reinterpret_cast<const float2*>(h0p + (size_t)r1 * V + 8 * nt + 2 * c)
                           : make_float2(0.f, 0.f);
      h[nt][0] = u.x;
      h[nt][1] = u.y;
      h[nt][2] = w.x;
      h[nt][3] = w.y;
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) h[nt][0] = h[nt][1] = h[nt][2] = h[nt][3] = 0.f;
  }
  uint32_t af[VT][4];
#pragma unroll
  for (int kt = 0; kt < VT; ++kt) {
    af[kt][0] = pack_bf16x2(h[2 * kt][0], h[2 * kt][1]);
    af[kt][1] = pack_bf16x2(h[2 * kt][2], h[2 * kt][3]);
    af[kt][2] = pack_bf16x2(h[2 * kt + 1][0], h[2 * kt + 1][1]);
    af[kt][3] = pack_bf16x2(h[2 * kt + 1][2], h[2 * kt + 1][3]);
  }
  __syncthreads();

  const long long wait_limit = kWaitLimitCycles;
  for (int cc = 0; cc < nchunks; ++cc) {
    const int st = cc & 1;
    const uint32_t par = (uint32_t)(cc >> 1) & 1u;
    const int t0 = cc * Tc;
    const int steps = min(Tc, T - t0);
    const bool has_next = cc + 2 < nchunks;

    float a_next = 0.f;  // gate logit of chunk cc + 2, loaded now, used after the chunk
    if (has_next && tid < Tc) {
      const int tt = t0 + 2 * Tc + tid;
      if (tt < T) a_next = bf16_bits_to_float(a[(pair_row + tt) * N + n]);
    }

    bool ok = mbar_wait_bounded(&bar[st], par, wait_limit);
    if (debug & kDebugForceTimeout) ok = ok && mbar_wait_bounded(&bar[2], 0, kDebugWaitLimitCycles);
    if (__syncthreads_or(!ok)) {
      // Give copies still in flight a bounded chance to land before the block exits.
      if (tid == 0) {
        atomicExch(status, kStatusTimeout);
        mbar_wait_bounded(&bar[st], par, kDebugWaitLimitCycles);
        if (cc + 1 < nchunks)
          mbar_wait_bounded(&bar[st ^ 1], (uint32_t)((cc + 1) >> 1) & 1u, kDebugWaitLimitCycles);
      }
      return;
    }

    const uint8_t* sbase = smem + st * L.stage_bytes;
    const uint16_t* qs = reinterpret_cast<const uint16_t*>(sbase + L.qs);
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(sbase + L.ks);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(sbase + L.vs);
    const float2* fgc = fgs + st * Tc;
    float* yp = ypart + (size_t)warp * Tc * V;

    for (int s = 0; s < steps; ++s) {
      const float2 fg = fgc[s];
      const float k0 = bf16_bits_to_float(ks[s * Kp + r0]);
      const float k1 = bf16_bits_to_float(ks[s * Kp + r1]);
      const float q0 = bf16_bits_to_float(qs[s * Kp + r0]);
      const float q1 = bf16_bits_to_float(qs[s * Kp + r1]);

      // Rank-1 write k_t v_t^T as the accumulator's initial value (Eq. (10)).
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(vs + s * V + 8 * nt + 2 * c);
        const float v0 = bf16_lo(vv), v1 = bf16_hi(vv);
        acc[nt][0] = k0 * v0;
        acc[nt][1] = k0 * v1;
        acc[nt][2] = k1 * v0;
        acc[nt][3] = k1 * v1;
      }
      // + H_{t-1} W on the tensor cores.
#pragma unroll
      for (int kt = 0; kt < VT; ++kt) {
        if constexpr (WREG) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], af[kt], wb[kt][nt][0], wb[kt][nt][1]);
        } else {
#pragma unroll
          for (int np = 0; np < VT; ++np) {
            uint32_t r[4];
            const int row = 16 * kt + ((lane >> 3) & 1) * 8 + (lane & 7);
            const int col = 16 * np + (lane >> 4) * 8;
            ldmatrix_x4_trans(r, Ws + row * WS + col);
            mma_bf16_16816(acc[2 * np], af[kt], r[0], r[1]);
            mma_bf16_16816(acc[2 * np + 1], af[kt], r[2], r[3]);
          }
        }
      }
      // Z = tanh(P); H = f H + (1 - f) Z   (Eq. (10)-(11)).
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) h[nt][e] = fmaf(fg.y, tanh_mufu(acc[nt][e]), fg.x * h[nt][e]);
      // Next step's bf16 A operand, straight from the accumulator layout.
#pragma unroll
      for (int kt = 0; kt < VT; ++kt) {
        af[kt][0] = pack_bf16x2(h[2 * kt][0], h[2 * kt][1]);
        af[kt][1] = pack_bf16x2(h[2 * kt][2], h[2 * kt][3]);
        af[kt][2] = pack_bf16x2(h[2 * kt + 1][0], h[2 * kt + 1][1]);
        af[kt][3] = pack_bf16x2(h[2 * kt + 1][2], h[2 * kt + 1][3]);
      }
      if constexpr (kCache) {  // H_t in bf16, streaming stores (real rows only)
        uint16_t* hp = Hs + ((size_t)pair * T + t0 + s) * K * V;
#pragma unroll
        for (int kt = 0; kt < VT; ++kt) {
          if (in0) {
            __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r0 * V + 16 * kt + 2 * c), af[kt][0]);
            __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r0 * V + 16 * kt + 8 + 2 * c), af[kt][2]);
          }
          if (in1) {
            __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r1 * V + 16 * kt + 2 * c), af[kt][1]);
            __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r1 * V + 16 * kt + 8 + 2 * c), af[kt][3]);
          }
        }
      }
      // Readout (Eq. (12)): this thread's two rows, weighted by q, per column.
      float p[MP];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        p[2 * nt] = fmaf(q1, h[nt][2], q0 * h[nt][0]);
        p[2 * nt + 1] = fmaf(q1, h[nt][3], q0 * h[nt][1]);
      }
#pragma unroll
      for (int i = M; i < MP; ++i) p[i] = 0.f;
      // Reduce-scatter over the 8 row groups (lane bits 4, 3, 2).
#pragma unroll
      for (int stg = 0; stg < 3; ++stg) {
        const int mask = 16 >> stg;
        const int half = MP >> (stg + 1);
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
      // Lane (g, c) now holds the sums of value slots m = m0 .. m0 + cnt - 1,
      // slot m being column 8 (m >> 1) + 2c + (m & 1).
      float* yrow = yp + s * V;
      if constexpr (MP >= 8) {
        constexpr int cnt = MP / 8;
#pragma unroll
        for (int i = 0; i < cnt; ++i) {
          const int m = cnt * g + i;
          if (m < M) yrow[8 * (m >> 1) + 2 * c + (m & 1)] = p[i];
        }
      } else {
        if ((g & 1) == 0) {
          const int m = g >> 1;
          yrow[8 * (m >> 1) + 2 * c + (m & 1)] = p[0];
        }
      }
    }
    __syncthreads();

    // y_t = sum over warps of the partials + w_r ⊙ v_t, as float4 rows.
    {
      constexpr int V4 = V / 4;
      const int nw = Kp / 16;
      for (int idx = tid; idx < steps * V4; idx += nthreads) {
        const int s = idx / V4, j = (idx - s * V4) * 4;
        const uint2 vv = *reinterpret_cast<const uint2*>(vs + s * V + j);
        float4 o;
        o.x = wrs[j] * bf16_lo(vv.x);
        o.y = wrs[j + 1] * bf16_hi(vv.x);
        o.z = wrs[j + 2] * bf16_lo(vv.y);
        o.w = wrs[j + 3] * bf16_hi(vv.y);
        for (int w = 0; w < nw; ++w) {
          const float4 u = *reinterpret_cast<const float4*>(ypart + ((size_t)w * Tc + s) * V + j);
          o.x += u.x;
          o.y += u.y;
          o.z += u.z;
          o.w += u.w;
        }
        *reinterpret_cast<float4*>(y + ((pair_row + t0 + s) * N + n) * V + j) = o;
      }
    }
    __syncthreads();
    if (has_next) {
      if (tid == 0) issue(cc + 2);
      if constexpr (kRagged) stage_qk(cc + 2);
      if (tid < Tc) fgs[st * Tc + tid] = gate_pair(a_next, al, be);
    }
  }

  if (H_T) {
    float* hp = H_T + (size_t)pair * K * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (in0)
        *reinterpret_cast<float2*>(hp + (size_t)r0 * V + 8 * nt + 2 * c) = make_float2(h[nt][0], h[nt][1]);
      if (in1)
        *reinterpret_cast<float2*>(hp + (size_t)r1 * V + 8 * nt + 2 * c) = make_float2(h[nt][2], h[nt][3]);
    }
  }
}

bool make_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, int inner, int N, int T,
              int B, int Tc) {
  const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)N, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * N,
                                 (cuuint64_t)inner * 2 * N * T};
  const cuuint32_t box[4] = {(cuuint32_t)inner, 1u, (cuuint32_t)Tc, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int VT, bool WREG, bool kCache, bool kRagged>
cudaError_t launch_vt_cache(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  const int V = 16 * VT;
  const int Kp = (p.K + 15) & ~15;
  // Tc <= threads (one gate logit per thread and chunk), and the shared memory fits.
  int Tc = min(V <= 64 ? 64 : 32, 2 * Kp);
  SmemLayout L = make_layout(Kp, V, Tc, WREG);
  while (L.total > 227 * 1024 && Tc > 8) {
    Tc /= 2;
    L = make_layout(Kp, V, Tc, WREG);
  }
  CUtensorMap mq, mk, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  if (!kRagged && (!make_map(enc, &mq, p.q, p.K, p.Nqk, p.T, p.B, Tc) ||
                   !make_map(enc, &mk, p.k, p.K, p.Nqk, p.T, p.B, Tc)))
    return cudaErrorInvalidValue;
  if (!make_map(enc, &mv, p.v, V, p.N, p.T, p.B, Tc)) return cudaErrorInvalidValue;
  auto kern = fwd_bf16_mma_rowwarp<VT, WREG, kCache, kRagged>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)p.B * (unsigned)p.N;
  kern<<<grid, 2 * Kp, L.total, stream>>>(mq, mk, mv, (const uint16_t*)p.q, (const uint16_t*)p.k,
                                          (const uint16_t*)p.a, p.alpha, p.beta,
                                          (const uint16_t*)p.W, p.w_r, p.H0, p.y, p.H_T,
                                          static_cast<uint16_t*>(p.Hs), p.T, p.N, p.K, Tc,
                                          p.Nqk == 1 ? 0 : 1, p.debug, p.status);
  return cudaGetLastError();
}

template <int VT>
cudaError_t launch_vt(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  constexpr bool kWreg = VT <= 4;  // W as register B fragments up to V = 64, else shared memory
  const bool ragged = p.K % 16 != 0;
  if (p.Hs)
    return ragged ? launch_vt_cache<VT, kWreg, true, true>(p, enc, stream)
                  : launch_vt_cache<VT, kWreg, true, false>(p, enc, stream);
  return ragged ? launch_vt_cache<VT, kWreg, false, true>(p, enc, stream)
                : launch_vt_cache<VT, kWreg, false, false>(p, enc, stream);
}

}  // namespace

bool mma_rowwarp_supports(int K, int V) {
  return K >= 1 && K <= 128 && V >= 16 && V <= 128 && V % 16 == 0;
}

cudaError_t launch_fwd_bf16_mma_rowwarp(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  switch (p.V) {
    case 16: return launch_vt<1>(p, enc, stream);
    case 32: return launch_vt<2>(p, enc, stream);
    case 48: return launch_vt<3>(p, enc, stream);
    case 64: return launch_vt<4>(p, enc, stream);
    case 80: return launch_vt<5>(p, enc, stream);
    case 96: return launch_vt<6>(p, enc, stream);
    case 112: return launch_vt<7>(p, enc, stream);
    case 128: return launch_vt<8>(p, enc, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m2rnn
