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
// Two kernels with that arithmetic:
//  * decode_bf16_mma: one block per pair, ceil(K / 16) warps; each warp loads its 16 state
//    rows straight from global memory into registers, and the block stages W through shared
//    memory for the B fragments.  Any 1 <= K <= 128 and V = 16, 32, ..., 128: the rows past
//    K of the last warp are zero (zero state, k and q), stay zero through the step and are
//    not stored.  Small batches are bound by launch latency.
//  * decode_bf16_persist (K = V = 64, many pairs): persistent blocks stream the pairs'
//    states and operands through a TMA-filled shared-memory ring (below); large batches are
//    bound by HBM traffic (the state is read and written once).
// The state update may be in place (H_in == H_out): a pair's state is read before any of
// it is written, and no two pairs share state.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kMaxWarps = 8;  // K <= 128

// MAXW: the most warps a launch uses (ceil(K / 16) <= MAXW).  Four-warp launches (K <= 64)
// with V <= 64 are register-capped so that six blocks fit on an SM: more state loads in
// flight.  V > 64 keeps more state and accumulator per thread and is not capped.
// RAG: K is not a multiple of 16 (the last warp's rows past K are padding); not capped
// either, since the row masks would spill under the cap.
template <int VT, int MAXW, bool RAG>
__global__ void __launch_bounds__(32 * MAXW, (MAXW <= 4 && VT <= 4 && !RAG) ? 6 : 1)
    decode_bf16_mma(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                    const uint16_t* __restrict__ v, const uint16_t* __restrict__ a,
                    const float* __restrict__ alpha, const float* __restrict__ beta,
                    const uint16_t* __restrict__ W, const float* __restrict__ w_r,
                    const float* H_in, float* H_out, float* __restrict__ y, int N, int Nqk, int K) {
  constexpr int V = 16 * VT, NT = 2 * VT, M = 4 * VT;
  // Reduce-scatter width: M rounded up to a power of two (slots M .. MP-1 stay zero).
  constexpr int MP = M <= 4 ? M : M <= 8 ? 8 : M <= 16 ? 16 : 32;
  __shared__ __align__(16) float ypart[MAXW][V];
  const int nw = (K + 15) / 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  const bool in0 = !RAG || r0 < K, in1 = !RAG || r1 < K;  // false only for padding rows
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
    h[nt][0] = hin && in0 ? *reinterpret_cast<const float2*>(hin + (size_t)r0 * V + 8 * nt + 2 * c)
                          : make_float2(0.f, 0.f);
    h[nt][1] = hin && in1 ? *reinterpret_cast<const float2*>(hin + (size_t)r1 * V + 8 * nt + 2 * c)
                          : make_float2(0.f, 0.f);
  }
  __syncthreads();
  const int lr = lane & 7, lq = lane >> 3;
  const float2 fg = gate_fg(bf16_bits_to_float(a[row]), alpha[n], beta[n]);
  const float2 ff = make_float2(fg.x, fg.x), gg = make_float2(fg.y, fg.y);

  // P = k v^T + bf16(H) W
  float2 acc[NT][2];
  {
    const float kv0 = in0 ? bf16_bits_to_float(k[qrow * K + r0]) : 0.f;
    const float kv1 = in1 ? bf16_bits_to_float(k[qrow * K + r1]) : 0.f;
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
      if (in0) *reinterpret_cast<float2*>(hout + (size_t)r0 * V + 8 * nt + 2 * c) = h[nt][0];
      if (in1) *reinterpret_cast<float2*>(hout + (size_t)r1 * V + 8 * nt + 2 * c) = h[nt][1];
    }
  }
  // y = H'^T q + w_r ⊙ v: q-weighted sums of this thread's two rows, reduce-scattered
  // over the warp's 8 row groups (same stages and order as the forward kernel).
  const float qv0 = in0 ? bf16_bits_to_float(q[qrow * K + r0]) : 0.f;
  const float qv1 = in1 ? bf16_bits_to_float(q[qrow * K + r1]) : 0.f;
  const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
  float p[MP];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float2 pp = fma2(q1, h[nt][1], mul2(q0, h[nt][0]));
    p[2 * nt] = pp.x;
    p[2 * nt + 1] = pp.y;
  }
#pragma unroll
  for (int i = M; i < MP; ++i) p[i] = 0.f;
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
  if constexpr (MP >= 8) {
    constexpr int cnt = MP / 8;
#pragma unroll
    for (int i = 0; i < cnt; ++i) {
      const int m = cnt * g + i;
      if (m < M) ypart[warp][8 * (m >> 1) + 2 * c + (m & 1)] = p[i];
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

// ---------------------------------------------------------------- persistent form
// K = V = 64 with many pairs: each block walks the pairs blockIdx.x, + gridDim.x, ... and a
// producer warp streams every pair's state (fp32, two 128-byte-swizzled boxes of 32 columns),
// its head's W (bf16, one swizzled 64 x 64 box) and the q, k, v rows into a ring of
// kPS shared-memory stages with TMA, and writes the pair's gate (f, 1 - f) into the stage,
// so that the state loads of later pairs are in flight while four compute warps update the
// current one.  The per-element arithmetic and the
// readout order are those of decode_bf16_mma<4, 4, false> above (bit for bit); only the operands'
// path differs (shared memory filled by TMA instead of per-thread global loads).
constexpr int kPS = 2;                  // stages per block
constexpr int kPBlocks = 3;             // blocks per SM
constexpr int kPStage = 25 * 1024;      // state 16 KB + W 8 KB + q, k, v, gate; 1 KB aligned
constexpr int kPH = 0, kPW = 16384, kPQ = 24576, kPK = kPQ + 128, kPV = kPK + 128;
constexpr int kPG = kPV + 128;          // float2 (f, 1 - f), written by the producer
constexpr int kPYpart = kPS * kPStage;  // float [2][4][64] readout partials (double buffer)
constexpr int kPBar = kPYpart + 2 * 4 * 64 * 4;  // full[kPS], empty[kPS], never, abort flag
constexpr int kPSmem = kPBar + (2 * kPS + 2) * 8 + 1024;  // + slack to align the base to 1024

__global__ void __launch_bounds__(160, kPBlocks)
    decode_bf16_persist(const __grid_constant__ CUtensorMap tm_h,
                        const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ a,
                        const float* __restrict__ alpha, const float* __restrict__ beta,
                        const float* __restrict__ w_r, bool has_h, float* H_out,
                        float* __restrict__ y, int npairs, int N, int Nqk, int debug,
                        int* status) {
  constexpr int V = 64, NT = 8, M = 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* ypart = reinterpret_cast<float*>(smem + kPYpart);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPBar);
  uint64_t* empty = full + kPS;
  uint64_t* never = empty + kPS;  // never armed: the forced-timeout test hook waits on it
  volatile int* abort_flag = reinterpret_cast<volatile int*>(never + 1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long limit = kWaitLimitCycles;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 4) {  // ------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t tx = (has_h ? 16384u : 0u) + 8192u + 3u * 128u;
      bool ok = true;
      int issued = 0;
      // Gate inputs loaded one pair ahead; the gate goes into the stage with its operands
      // (the arrive below releases it to the compute warps).
      int pn = blockIdx.x;
      float an = 0.f, aln = 0.f, ben = 0.f;
      if (pn < npairs) {
        const int nn = pn - (pn / N) * N;
        an = bf16_bits_to_float(a[pn]);
        aln = alpha[nn];
        ben = beta[nn];
      }
      for (int i = 0; ok; ++i) {
        const int p = blockIdx.x + i * gridDim.x;
        if (p >= npairs) break;
        const int st = i % kPS, b = p / N, n = p - (p / N) * N;
        const float ac = an, alc = aln, bec = ben;
        pn = p + gridDim.x;
        if (pn < npairs) {
          const int nn = pn - (pn / N) * N;
          an = bf16_bits_to_float(a[pn]);
          aln = alpha[nn];
          ben = beta[nn];
        }
        // Gives up early once the compute warps have stopped (their own wait gave up).
        if (i >= kPS)
          ok = wait_or_abort_sleep(&empty[st], (uint32_t)((i / kPS) - 1) & 1u, limit, abort_flag);
        if (!ok) break;
        uint8_t* base = smem + st * kPStage;
        *reinterpret_cast<float2*>(base + kPG) = gate_fg(ac, alc, bec);
        mbar_arrive_expect_tx(&full[st], tx);
        tma_load_4d(base + kPW, &tm_w, &full[st], 0, 0, n, 0);
        if (has_h) {
          tma_load_4d(base + kPH, &tm_h, &full[st], 0, 0, p, 0);
          tma_load_4d(base + kPH + 8192, &tm_h, &full[st], 32, 0, p, 0);
        }
        tma_load_4d(base + kPQ, &tm_q, &full[st], 0, Nqk == 1 ? 0 : n, b, 0);
        tma_load_4d(base + kPK, &tm_k, &full[st], 0, Nqk == 1 ? 0 : n, b, 0);
        tma_load_4d(base + kPV, &tm_v, &full[st], 0, n, b, 0);
        issued = i + 1;
      }
      if (!ok) atomicExch(status, kStatusTimeout);
      // Every copy issued has landed before the block ends (normally the compute warps have
      // consumed them all; after a timeout they may not have).
      for (int i = issued - kPS > 0 ? issued - kPS : 0; i < issued; ++i)
        mbar_wait_bounded_sleep(&full[i % kPS], (uint32_t)(i / kPS) & 1u, kDebugWaitLimitCycles);
    }
    return;
  }

  // ------------------------------------------------------------------ compute warps
  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  const int lr = lane & 7, lq = lane >> 3;
  int p = blockIdx.x;
  for (int i = 0; p < npairs; ++i, p += gridDim.x) {
    const int st = i % kPS, n = p - (p / N) * N;
    // A joint decision, so that no warp is left alone at the named barrier below.
    bool wok = mbar_wait_bounded(&full[st], (uint32_t)(i / kPS) & 1u, limit);
    if ((debug & kDebugForceTimeout) && i == 0)
      wok = wok && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
    if (named_bar_or(2, 128, !wok)) {
      if (lane == 0) atomicExch(status, kStatusTimeout);
      if (threadIdx.x == 0) *abort_flag = 1;  // releases the producer's wait for a free stage
      break;
    }
    const uint8_t* base = smem + st * kPStage;
    const uint32_t wb0 = smem_u32(base + kPW);
    const uint16_t* qs = reinterpret_cast<const uint16_t*>(base + kPQ);
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(base + kPK);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(base + kPV);
    // State rows r0, r1, columns 8 nt + 2c, +1 from the swizzled boxes.
    float2 h[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t off = (uint32_t)((nt >> 2) * 8192 + ((((2 * (nt & 3) + (c >> 1)) ^ g)) << 4) +
                                      (c & 1) * 8);
      if (has_h) {
        h[nt][0] = *reinterpret_cast<const float2*>(base + kPH + r0 * 128 + off);
        h[nt][1] = *reinterpret_cast<const float2*>(base + kPH + r1 * 128 + off);
      } else {
        h[nt][0] = h[nt][1] = make_float2(0.f, 0.f);
      }
    }
    const float2 fg = *reinterpret_cast<const float2*>(base + kPG);
    const float2 ff = make_float2(fg.x, fg.x), gg = make_float2(fg.y, fg.y);
    // P = k v^T + bf16(H) W
    float2 acc[NT][2];
    {
      const float kv0 = bf16_bits_to_float(ks[r0]), kv1 = bf16_bits_to_float(ks[r1]);
      const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 vv = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vs + 8 * nt + 2 * c));
        acc[nt][0] = mul2(k0, vv);
        acc[nt][1] = mul2(k1, vv);
      }
    }
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t af[4];
      af[0] = pack_bf16x2(h[2 * kt][0].x, h[2 * kt][0].y);
      af[1] = pack_bf16x2(h[2 * kt][1].x, h[2 * kt][1].y);
      af[2] = pack_bf16x2(h[2 * kt + 1][0].x, h[2 * kt + 1][0].y);
      af[3] = pack_bf16x2(h[2 * kt + 1][1].x, h[2 * kt + 1][1].y);
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {  // B fragments of n-tiles 2 np, 2 np + 1
        uint32_t wbf[4];
        ldsm_x4_trans(wbf, sw128_addr(wb0, 16 * kt + lr + 8 * (lq & 1), 2 * np + (lq >> 1)));
        mma2(acc[2 * np], af, wbf[0], wbf[1]);
        mma2(acc[2 * np + 1], af, wbf[2], wbf[3]);
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
    float* hout = H_out + (size_t)p * 64 * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(hout + (size_t)r0 * V + 8 * nt + 2 * c) = h[nt][0];
      *reinterpret_cast<float2*>(hout + (size_t)r1 * V + 8 * nt + 2 * c) = h[nt][1];
    }
    // y = H'^T q + w_r ⊙ v (same reduction as decode_bf16_mma)
    const float qv0 = bf16_bits_to_float(qs[r0]), qv1 = bf16_bits_to_float(qs[r1]);
    const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
    float pr[M];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 pp = fma2(q1, h[nt][1], mul2(q0, h[nt][0]));
      pr[2 * nt] = pp.x;
      pr[2 * nt + 1] = pp.y;
    }
#pragma unroll
    for (int stg = 0; stg < 3; ++stg) {
      const int mask = 16 >> stg;
      const int half = M >> (stg + 1);
      const bool up = (lane & mask) != 0;
#pragma unroll
      for (int j = 0; j < half; ++j) {
        const float send = up ? pr[j] : pr[j + half];
        const float keep = up ? pr[j + half] : pr[j];
        pr[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
      }
    }
    float* yp = ypart + (i & 1) * 4 * 64;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int m = 2 * g + j;
      yp[warp * 64 + 8 * (m >> 1) + 2 * c + (m & 1)] = pr[j];
    }
    named_bar_sync(1, 128);
    if (threadIdx.x < V) {
      const int j = threadIdx.x;
      // Rounded product, then the warps' partials in warp order: no contraction into an FMA,
      // as in the kernels with a runtime warp count (the sums must match theirs bit for bit).
      float o = __fmul_rn(w_r[(size_t)n * V + j], bf16_bits_to_float(vs[j]));
#pragma unroll
      for (int w = 0; w < 4; ++w) o = __fadd_rn(o, yp[w * 64 + j]);
      y[(size_t)p * V + j] = o;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp has read stage st
  }
}

}  // namespace

bool decode_supports(int K, int V) {
  return K >= 1 && K <= 16 * kMaxWarps && V >= 16 && V <= 128 && V % 16 == 0;
}

bool make_map_dec(EncodeTiledFn enc, CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                  int esize, const cuuint64_t (&dims)[4], const cuuint32_t (&box)[4],
                  CUtensorMapSwizzle swz) {
  const cuuint64_t strides[3] = {dims[0] * esize, dims[0] * dims[1] * esize,
                                 dims[0] * dims[1] * dims[2] * esize};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The persistent form: K = V = 64, enough pairs to fill every SM twice over (unless
// `force`), and the 16-byte alignment TMA needs.  Returns false (nothing launched) when it
// does not apply.
bool launch_decode_persist(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                           cudaError_t* err, bool force) {
  const long long npairs = (long long)p.B * p.N;
  if (p.K != 64 || p.V != 64 || !enc || !p.status || (!force && npairs < 2048) ||
      npairs > 0x7fffffffLL)
    return false;
  if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.W) ||
      !aligned16(p.H_T) || (p.H0 && !aligned16(p.H0)))
    return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  CUtensorMap mh, mw, mq, mk, mv;
  memset(&mh, 0, sizeof(mh));
  const cuuint64_t dh[4] = {64, 64, (cuuint64_t)npairs, 1};
  const cuuint32_t bh[4] = {32, 64, 1, 1};
  const cuuint64_t dw[4] = {64, 64, (cuuint64_t)p.N, 1};
  const cuuint32_t bw[4] = {64, 64, 1, 1};
  const cuuint64_t dqk[4] = {64, (cuuint64_t)p.Nqk, (cuuint64_t)p.B, 1};
  const cuuint64_t dv[4] = {64, (cuuint64_t)p.N, (cuuint64_t)p.B, 1};
  const cuuint32_t brow[4] = {64, 1, 1, 1};
  if ((p.H0 && !make_map_dec(enc, &mh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.H0, 4, dh, bh,
                             CU_TENSOR_MAP_SWIZZLE_128B)) ||
      !make_map_dec(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.W, 2, dw, bw,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_dec(enc, &mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 2, dqk, brow,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_dec(enc, &mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, 2, dqk, brow,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_dec(enc, &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, 2, dv, brow,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  *err = cudaFuncSetAttribute(decode_bf16_persist, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kPSmem);
  if (*err != cudaSuccess) return true;
  const unsigned grid = (unsigned)std::min<long long>(npairs, (long long)kPBlocks * sms);
  decode_bf16_persist<<<grid, 160, kPSmem, stream>>>(
      mh, mw, mq, mk, mv, (const uint16_t*)p.a, p.alpha, p.beta, p.w_r, p.H0 != nullptr, p.H_T,
      p.y, (int)npairs, p.N, p.Nqk, p.debug, p.status);
  *err = cudaGetLastError();
  return true;
}

bool decode_persist_supports(const Problem& p) {
  return p.K == 64 && p.V == 64 && aligned16(p.q) && aligned16(p.k) && aligned16(p.v) &&
         aligned16(p.W) && aligned16(p.H_T) && (!p.H0 || aligned16(p.H0));
}

cudaError_t launch_decode_bf16(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                               int which) {
  cudaError_t perr = cudaSuccess;
  if (which != 1 && launch_decode_persist(p, enc, stream, &perr, which == 2)) return perr;
  if (which == 2) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)p.B * (unsigned)p.N;
  const unsigned threads = 32u * (unsigned)((p.K + 15) / 16);
  auto args = [&](auto kern) {
    kern<<<grid, threads, 0, stream>>>((const uint16_t*)p.q, (const uint16_t*)p.k,
                                       (const uint16_t*)p.v, (const uint16_t*)p.a, p.alpha, p.beta,
                                       (const uint16_t*)p.W, p.w_r, p.H0, p.H_T, p.y, p.N, p.Nqk,
                                       p.K);
  };
  const bool small = p.K <= 64, rag = p.K % 16 != 0;
  auto pick = [&](auto k4, auto k8, auto k4r, auto k8r) {
    if (rag) small ? args(k4r) : args(k8r);
    else small ? args(k4) : args(k8);
  };
#define M2RNN_DECODE_CASE(VT)                                                                  \
  case 16 * VT:                                                                                \
    pick(decode_bf16_mma<VT, 4, false>, decode_bf16_mma<VT, kMaxWarps, false>,                 \
         decode_bf16_mma<VT, 4, true>, decode_bf16_mma<VT, kMaxWarps, true>);                  \
    break;
  switch (p.V) {
    M2RNN_DECODE_CASE(1)
    M2RNN_DECODE_CASE(2)
    M2RNN_DECODE_CASE(3)
    M2RNN_DECODE_CASE(4)
    M2RNN_DECODE_CASE(5)
    M2RNN_DECODE_CASE(6)
    M2RNN_DECODE_CASE(7)
    M2RNN_DECODE_CASE(8)
#undef M2RNN_DECODE_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace m2rnn
