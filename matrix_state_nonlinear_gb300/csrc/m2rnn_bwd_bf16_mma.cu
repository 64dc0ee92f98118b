// m2rnn_bwd_bf16_mma.cu — backward pass of the M²RNN recurrence on the warp-level
// tensor-core MMA, K = V = 64, bf16 operands, fp32 gradients.
//
// The reverse scan of the M²RNN study notes, Sec. 2.7 (u_t = dL/dy_t, C_T = dL/dH_T):
//   Z_t = tanh(H_{t-1} W + k_t v_t^T)   recomputed from the kept bf16 state H_{t-1}
//   R_t = C_t + q_t u_t^T,   D_t = ((1 - f_t) R_t) ⊙ (1 - Z_t ⊙ Z_t)
//   C_{t-1} = f_t R_t + D_t W^T,   dL/df_t = <R_t, H_{t-1} - Z_t>
//   dW += H_{t-1}^T D_t,  dk_t = D_t v_t,  dv_t = D_t^T k_t + w_r ⊙ u_t,  dq_t = H_t u_t
// and the gate chain rule of Eq. (13)/(17).  The states are the ones the training
// forward kept (the notes' Sec. 2.6), rounded to bf16: exactly the tensor-core
// operand the forward multiplied by W, so H_{t-1} W and Z_t here repeat the
// forward's arithmetic bit for bit (same MMA sequence, same MUFU tanh).
//
// One thread block per (batch, head) pair: 4 compute warps own 16 rows of the
// state gradient C each (fp32, mma accumulator layout, in registers) and one
// producer warp.  Per step each compute warp runs three 16 x 64 x 64 MMA products:
//   * P_t = H_{t-1} W (+ k v^T): A fragments of H_{t-1} by ldmatrix from the TMA-loaded
//     state tile, B fragments of W by ldmatrix.trans from shared memory;
//   * C_{t-1} = f R_t + D_t W^T: A fragments packed from D_t in registers, W^T as
//     register-resident B fragments (the serial chain of the scan);
//   * dW += H_{t-1}^T D_t for its 32 x 32 block of dW: D_t of all rows goes through a
//     double-buffered shared tile (stmatrix), both operands by ldmatrix.trans.
// The producer warp TMA-loads, in reverse time order, chunks of Tc steps: the bf16
// state tiles (128-byte swizzle, so the ldmatrix rows hit distinct banks), q, k, v
// and dy; it computes the gate factors, and after a chunk sums the per-warp dv and
// dL/df partials into dv, da, dalpha, dbeta and dw_r.  All waits are bounded.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kK = 64, kV = 64;
constexpr int kNW = kK / 16;               // compute warps
constexpr int kNT = kV / 8;                // n-tiles of 8 columns
constexpr int kVT = kV / 16;               // k-tiles of 16 columns
constexpr int kTc = 4;                     // steps per chunk
constexpr int kThreads = 32 * (kNW + 1);
constexpr int kBar = 1;                    // named barrier of the compute warps
constexpr int kTile = kK * kV * 2;         // one bf16 K x V tile (64 rows of 128 bytes)

struct BwdLayout {
  int hs;        // [2][kTc] state tiles (TMA, 128-byte swizzle)
  int h0t;       // bf16(H_0) tile, same layout
  int dslot;     // [2] D_t tiles (stmatrix, same swizzle)
  int wsm;       // W (bf16, same swizzle)
  int in;        // [2] input stages: q, k [kTc][kK] bf16; v [kTc][kV] bf16; dy [kTc][kV] f32
  int in_stage, qs, ks, vs, dys;
  int gates;     // float4 [2][kTc]: f, 1 - f, sigmoid(x), softplus(x)
  int dfp;       // float [2][kNW][kTc]
  int dvp;       // float [2][kNW][kTc][kV]
  int bar;       // full[2], done[2], never; int abort
  int total;
};

__host__ __device__ inline BwdLayout bwd_layout() {
  BwdLayout L;
  int o = 0;
  L.hs = o;
  o += 2 * kTc * kTile;
  L.h0t = o;
  o += kTile;
  L.dslot = o;
  o += 2 * kTile;
  L.wsm = o;
  o += kV * kV * 2;
  L.qs = 0;
  L.ks = kTc * kK * 2;
  L.vs = L.ks + kTc * kK * 2;
  L.dys = L.vs + kTc * kV * 2;
  L.in_stage = (L.dys + kTc * kV * 4 + 127) & ~127;
  L.in = o;
  o += 2 * L.in_stage;
  L.gates = o;
  o += 2 * kTc * 16;
  L.dfp = o;
  o += 2 * kNW * kTc * 4;
  L.dvp = o;
  o += 2 * kNW * kTc * kV * 4;
  L.bar = o;
  o += 64;
  L.total = o + 1024;  // room to align the base to 1024 bytes
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_mma(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_dy, const uint16_t* __restrict__ a,
                 const float* __restrict__ alpha, const float* __restrict__ beta,
                 const uint16_t* __restrict__ W, const float* __restrict__ w_r,
                 const float* __restrict__ H0, const float* __restrict__ dH_T,
                 float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                 float* __restrict__ da, float* __restrict__ dH0, float* __restrict__ ws,
                 float* __restrict__ dqk_heads, int T, int N, int Nqk, int debug, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const BwdLayout L = bwd_layout();
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + kTc - 1) / kTc;
  const int nq = Nqk == 1 ? 0 : n;
  const bool shared_qk = Nqk == 1 && N > 1;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* done = full + 2;
  uint64_t* never = full + 4;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 5);
  float4* gates = reinterpret_cast<float4*>(smem + L.gates);
  float* dfp = reinterpret_cast<float*>(smem + L.dfp);
  float* dvp = reinterpret_cast<float*>(smem + L.dvp);
  float* wsp = ws + (size_t)pair * backward_pair_floats(kK, kV);
  float* dWp = wsp + kK * kV;
  float* dwr_p = dWp + kV * kV;
  float* ab_p = dwr_p + kV;
  const long long limit = kWaitLimitCycles;

  if (tid == 0) {
    mbar_init(&full[0], 32);
    mbar_init(&full[1], 32);
    mbar_init(&done[0], 32 * kNW);
    mbar_init(&done[1], 32 * kNW);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // W and bf16(H_0) into swizzled tiles (16-byte chunks; 64 rows x 8 chunks each).
  const uint16_t* Wn = W + (size_t)n * kV * kV;
  const float* h0p = H0 ? H0 + (size_t)pair * kK * kV : nullptr;
  for (int e = tid; e < kV * 8; e += kThreads) {
    const int row = e >> 3, ch = e & 7;
    const uint4 wv = *reinterpret_cast<const uint4*>(Wn + row * kV + 8 * ch);
    *reinterpret_cast<uint4*>(smem + (sw128_addr(sbase + L.wsm, row, ch) - sbase)) = wv;
    uint4 hv = make_uint4(0u, 0u, 0u, 0u);
    if (h0p) {
      const float4 x0 = *reinterpret_cast<const float4*>(h0p + row * kV + 8 * ch);
      const float4 x1 = *reinterpret_cast<const float4*>(h0p + row * kV + 8 * ch + 4);
      hv = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                      pack_bf16x2(x1.z, x1.w));
    }
    *reinterpret_cast<uint4*>(smem + (sw128_addr(sbase + L.h0t, row, ch) - sbase)) = hv;
  }
  __syncthreads();

  auto stage_of = [&](int p) { return p & 1; };
  auto chunk_of = [&](int p) { return nchunks - 1 - p; };  // reverse time order

  if (warp == kNW) {
    // ======================================================= producer warp
    const float al = alpha[n], be = beta[n];
    const uint32_t tx = (uint32_t)(kTc * kTile + 2 * kTc * kK * 2 + kTc * kV * 2 + kTc * kV * 4);
    const float2 wr = *reinterpret_cast<const float2*>(w_r + (size_t)n * kV + 2 * lane);
    auto arm = [&](int p) {
      const int st = stage_of(p), t0 = chunk_of(p) * kTc;
      if (lane < kTc) {  // gate factors of Eq. (13)/(17) and their derivatives
        const int t = t0 + lane;
        const float x = (t < T ? bf16_bits_to_float(a[((size_t)b * T + t) * N + n]) : 0.f) + be;
        const float ex = expf(-fabsf(x));
        const float sp = fmaxf(x, 0.f) + log1pf(ex);
        const float sg = x >= 0.f ? 1.f / (1.f + ex) : ex / (1.f + ex);
        gates[st * kTc + lane] = make_float4(expf(-al * sp), -expm1f(-al * sp), sg, sp);
      }
      __syncwarp();
      if (lane != 0) {
        mbar_arrive(&full[st]);
      } else {
        uint8_t* in = smem + L.in + st * L.in_stage;
        mbar_arrive_expect_tx(&full[st], tx);
        tma_load_4d(smem + L.hs + st * kTc * kTile, &tm_h, &full[st], 0, 0, t0, pair);
        tma_load_4d(in + L.qs, &tm_q, &full[st], 0, nq, t0, b);
        tma_load_4d(in + L.ks, &tm_k, &full[st], 0, nq, t0, b);
        tma_load_4d(in + L.vs, &tm_v, &full[st], 0, n, t0, b);
        tma_load_4d(in + L.dys, &tm_dy, &full[st], 0, n, t0, b);
      }
    };
    if (lane == 0) {
      prefetch_tensormap(&tm_h);
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_dy);
    }
    int issued = 0;
    for (; issued < 2 && issued < nchunks; ++issued) arm(issued);
    float2 dwr = make_float2(0.f, 0.f);
    float dal = 0.f, dbe = 0.f;
    for (int p = 0; p < nchunks; ++p) {
      const int st = stage_of(p), t0 = chunk_of(p) * kTc;
      const int steps = min(kTc, T - t0);
      const bool ok = wait_or_abort(&done[st], (uint32_t)(p >> 1) & 1u, limit, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicExch(status, kStatusTimeout);
          for (int pi = p; pi < issued; ++pi)  // let copies in flight land
            mbar_wait_bounded(&full[stage_of(pi)], (uint32_t)(pi >> 1) & 1u, kDebugWaitLimitCycles);
        }
        break;
      }
      const uint8_t* in = smem + L.in + st * L.in_stage;
      const float* dys = reinterpret_cast<const float*>(in + L.dys);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(in + L.vs);
      for (int s = 0; s < steps; ++s) {  // columns 2 lane, 2 lane + 1
        const size_t row = ((size_t)b * T + t0 + s) * N + n;
        const float2 u = *reinterpret_cast<const float2*>(dys + s * kV + 2 * lane);
        float2 acc = make_float2(wr.x * u.x, wr.y * u.y);
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
          const float2 pw =
              *reinterpret_cast<const float2*>(dvp + ((st * kNW + w) * kTc + s) * kV + 2 * lane);
          acc.x += pw.x;
          acc.y += pw.y;
        }
        *reinterpret_cast<float2*>(dv + row * kV + 2 * lane) = acc;
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(vs + s * kV + 2 * lane);
        dwr.x = fmaf(u.x, bf16_lo(vv), dwr.x);
        dwr.y = fmaf(u.y, bf16_hi(vv), dwr.y);
      }
      if (lane < steps) {
        float df = 0.f;
#pragma unroll
        for (int w = 0; w < kNW; ++w) df += dfp[(st * kNW + w) * kTc + lane];
        const float4 gt = gates[st * kTc + lane];
        const float d_a = df * (-al * gt.x * gt.z);
        da[((size_t)b * T + t0 + lane) * N + n] = d_a;
        dal = fmaf(df, -gt.x * gt.w, dal);
        dbe += d_a;
      }
      __syncwarp();
      if (issued < nchunks) arm(issued++);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {  // fixed-order tree: deterministic
      dal += __shfl_xor_sync(0xffffffffu, dal, o);
      dbe += __shfl_xor_sync(0xffffffffu, dbe, o);
    }
    *reinterpret_cast<float2*>(dwr_p + 2 * lane) = dwr;
    if (lane == 0) {
      ab_p[0] = dal;
      ab_p[1] = dbe;
    }
    return;
  }

  // ========================================================= compute warps
  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  // ldmatrix row addressing: lane L supplies row (L & 7) + 8 * bit of matrix L >> 3.
  const int lr = lane & 7, lq = lane >> 3;

  // W^T as B fragments of C += D W^T (k = column j of W, n = row l of W).
  uint32_t wtb[kVT][kNT][2];
#pragma unroll
  for (int kj = 0; kj < kVT; ++kj)
#pragma unroll
    for (int nl = 0; nl < kNT; ++nl) {
      const uint16_t* wrow = Wn + (8 * nl + g) * kV + 16 * kj + 2 * c;
      wtb[kj][nl][0] = *reinterpret_cast<const uint32_t*>(wrow);
      wtb[kj][nl][1] = *reinterpret_cast<const uint32_t*>(wrow + 8);
    }
  // State gradient C_T = dH_T for rows r0, r1 (accumulator layout).
  float2 C[kNT][2];
  const float* dhp = dH_T ? dH_T + (size_t)pair * kK * kV : nullptr;
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    C[nt][0] = dhp ? *reinterpret_cast<const float2*>(dhp + r0 * kV + 8 * nt + 2 * c)
                   : make_float2(0.f, 0.f);
    C[nt][1] = dhp ? *reinterpret_cast<const float2*>(dhp + r1 * kV + 8 * nt + 2 * c)
                   : make_float2(0.f, 0.f);
  }
  // This warp's 32 x 32 block of dW: rows 32 mb + 16 mt (+ g, g + 8), columns 32 nb + 8 nt.
  const int mb = warp >> 1, nb = warp & 1;
  float2 dWa[2][4][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) dWa[mt][nt][0] = dWa[mt][nt][1] = make_float2(0.f, 0.f);

  bool ok = wait_or_abort(&full[0], 0u, limit, abort_flag);
  if (debug & kDebugForceTimeout) ok = ok && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
  bool aborted = named_bar_or(kBar, 32 * kNW, !ok);

  for (int p = 0; p < nchunks && !aborted; ++p) {
    const int st = stage_of(p), cidx = chunk_of(p), t0 = cidx * kTc;
    const int steps = min(kTc, T - t0);
    if (p > 0) {
      const bool w_ok = wait_or_abort(&full[st], (uint32_t)(p >> 1) & 1u, limit, abort_flag);
      if (named_bar_or(kBar, 32 * kNW, !w_ok)) {
        aborted = true;
        break;
      }
    }
    const uint8_t* in = smem + L.in + st * L.in_stage;
    const uint16_t* qs = reinterpret_cast<const uint16_t*>(in + L.qs);
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(in + L.ks);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(in + L.vs);
    const float* dys = reinterpret_cast<const float*>(in + L.dys);
    for (int s = steps - 1; s >= 0; --s) {
      const int t = t0 + s;
      if (s == 0 && cidx > 0) {  // H_{t-1} is the last state of the next chunk to process
        const bool w_ok = wait_or_abort(&full[stage_of(p + 1)], (uint32_t)((p + 1) >> 1) & 1u,
                                        limit, abort_flag);
        if (named_bar_or(kBar, 32 * kNW, !w_ok)) {
          aborted = true;
          break;
        }
      }
      const uint32_t hcur = sbase + L.hs + (st * kTc + s) * kTile;
      const uint32_t hprev = s > 0 ? hcur - kTile
                             : cidx > 0 ? sbase + L.hs + (stage_of(p + 1) * kTc + kTc - 1) * kTile
                                        : sbase + L.h0t;
      const uint32_t dsl = sbase + L.dslot + (t & 1) * kTile;
      const float4 gt = gates[st * kTc + s];
      const float2 ff = make_float2(gt.x, gt.x), gg = make_float2(gt.y, gt.y);

      // ---- P_t = k_t v_t^T + H_{t-1} W (the forward's operands and order)
      uint32_t ah[kVT][4];
#pragma unroll
      for (int kt = 0; kt < kVT; ++kt)
        ldsm_x4(ah[kt], sw128_addr(hprev, 16 * warp + lr + 8 * (lq & 1), 2 * kt + (lq >> 1)));
      float2 P[kNT][2];
      {
        const float kv0 = bf16_bits_to_float(ks[s * kK + r0]);
        const float kv1 = bf16_bits_to_float(ks[s * kK + r1]);
        const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const float2 vv =
              bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vs + s * kV + 8 * nt + 2 * c));
          P[nt][0] = mul2(k0, vv);
          P[nt][1] = mul2(k1, vv);
        }
      }
#pragma unroll
      for (int kt = 0; kt < kVT; ++kt)
#pragma unroll
        for (int np = 0; np < kNT / 2; ++np) {
          uint32_t wb[4];  // b0, b1 of n-tile 2 np, then of n-tile 2 np + 1
          ldsm_x4_trans(wb, sw128_addr(sbase + L.wsm, 16 * kt + lr + 8 * (lq & 1), 2 * np + (lq >> 1)));
          mma2(P[2 * np], ah[kt], wb[0], wb[1]);
          mma2(P[2 * np + 1], ah[kt], wb[2], wb[3]);
        }

      // ---- Z, R, D (in place of P), dL/df partial, C <- f R
      const float qv0 = bf16_bits_to_float(qs[s * kK + r0]);
      const float qv1 = bf16_bits_to_float(qs[s * kK + r1]);
      const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
      float dfl = 0.f;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const float2 u = *reinterpret_cast<const float2*>(dys + s * kV + 8 * nt + 2 * c);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          // H_{t-1} at (row r, columns 8 nt + 2c, +1): A fragment register 2 (nt & 1) + r of k-tile nt / 2
          const uint32_t hb = ah[nt >> 1][2 * (nt & 1) + r];
          const float2 h = bf16x2_to_float2(hb);
          const float2 z = make_float2(tanh_mufu(P[nt][r].x), tanh_mufu(P[nt][r].y));
          const float2 R = fma2(r ? q1 : q0, u, C[nt][r]);
          const float2 one_m_z2 = make_float2(fmaf(-z.x, z.x, 1.f), fmaf(-z.y, z.y, 1.f));
          P[nt][r] = mul2(mul2(gg, R), one_m_z2);   // D_t
          dfl = fmaf(R.x, h.x - z.x, dfl);
          dfl = fmaf(R.y, h.y - z.y, dfl);
          C[nt][r] = mul2(ff, R);
        }
      }

      // ---- dk_t = D v_t (row sums), dv partial = D^T k_t over this warp's rows
      float pdv[2 * kNT];
      float sk0 = 0.f, sk1 = 0.f;
      {
        const float kv0 = bf16_bits_to_float(ks[s * kK + r0]);
        const float kv1 = bf16_bits_to_float(ks[s * kK + r1]);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const float2 vv =
              bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vs + s * kV + 8 * nt + 2 * c));
          sk0 = fmaf(P[nt][0].x, vv.x, fmaf(P[nt][0].y, vv.y, sk0));
          sk1 = fmaf(P[nt][1].x, vv.x, fmaf(P[nt][1].y, vv.y, sk1));
          pdv[2 * nt] = fmaf(kv1, P[nt][1].x, kv0 * P[nt][0].x);
          pdv[2 * nt + 1] = fmaf(kv1, P[nt][1].y, kv0 * P[nt][0].y);
        }
      }

      // ---- D_t as bf16 A fragments; publish to the shared D tile; C += D W^T
      uint32_t ad[kVT][4];
#pragma unroll
      for (int kj = 0; kj < kVT; ++kj) {
        ad[kj][0] = pack_bf16x2(P[2 * kj][0].x, P[2 * kj][0].y);
        ad[kj][1] = pack_bf16x2(P[2 * kj][1].x, P[2 * kj][1].y);
        ad[kj][2] = pack_bf16x2(P[2 * kj + 1][0].x, P[2 * kj + 1][0].y);
        ad[kj][3] = pack_bf16x2(P[2 * kj + 1][1].x, P[2 * kj + 1][1].y);
        stsm_x4(sw128_addr(dsl, 16 * warp + lr + 8 * (lq & 1), 2 * kj + (lq >> 1)), ad[kj]);
      }
#pragma unroll
      for (int kj = 0; kj < kVT; ++kj)
#pragma unroll
        for (int nl = 0; nl < kNT; ++nl) mma2(C[nl], ad[kj], wtb[kj][nl][0], wtb[kj][nl][1]);

      // ---- reductions: dk, dv partials, dL/df partial, dq = H_t u_t
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        sk0 += __shfl_xor_sync(0xffffffffu, sk0, o);
        sk1 += __shfl_xor_sync(0xffffffffu, sk1, o);
      }
#pragma unroll
      for (int stg = 0; stg < 3; ++stg) {  // reduce-scatter over the 8 row groups
        const int mask = 16 >> stg, half = kNT >> stg;
        const bool up = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = up ? pdv[i] : pdv[i + half];
          const float keep = up ? pdv[i + half] : pdv[i];
          pdv[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
      // Lane (g, c) now holds columns 8 g + 2c, 8 g + 2c + 1.
      *reinterpret_cast<float2*>(dvp + ((st * kNW + warp) * kTc + s) * kV + 8 * g + 2 * c) =
          make_float2(pdv[0], pdv[1]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dfl += __shfl_xor_sync(0xffffffffu, dfl, o);
      if (lane == 0) dfp[(st * kNW + warp) * kTc + s] = dfl;
      float sq0 = 0.f, sq1 = 0.f;
      {
        uint32_t hc[kVT][4];
#pragma unroll
        for (int kt = 0; kt < kVT; ++kt)
          ldsm_x4(hc[kt], sw128_addr(hcur, 16 * warp + lr + 8 * (lq & 1), 2 * kt + (lq >> 1)));
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const float2 u = *reinterpret_cast<const float2*>(dys + s * kV + 8 * nt + 2 * c);
          const float2 h0 = bf16x2_to_float2(hc[nt >> 1][2 * (nt & 1)]);
          const float2 h1 = bf16x2_to_float2(hc[nt >> 1][2 * (nt & 1) + 1]);
          sq0 = fmaf(h0.x, u.x, fmaf(h0.y, u.y, sq0));
          sq1 = fmaf(h1.x, u.x, fmaf(h1.y, u.y, sq1));
        }
      }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        sq0 += __shfl_xor_sync(0xffffffffu, sq0, o);
        sq1 += __shfl_xor_sync(0xffffffffu, sq1, o);
      }
      if (c == 0) {
        const size_t qrow = ((size_t)b * T + t) * (shared_qk ? N : Nqk) + (shared_qk ? n : nq);
        float* dqo = shared_qk ? dqk_heads : dq;
        float* dko = shared_qk ? dqk_heads + (size_t)gridDim.x * T * kK : dk;
        dqo[qrow * kK + r0] = sq0;
        dqo[qrow * kK + r1] = sq1;
        dko[qrow * kK + r0] = sk0;
        dko[qrow * kK + r1] = sk1;
      }

      // ---- dW += H_{t-1}^T D_t (this warp's 32 x 32 block, all 64 rows of step t)
      named_bar_sync(kBar, 32 * kNW);
#pragma unroll
      for (int kt = 0; kt < kK / 16; ++kt) {
        uint32_t ha[2][4], db[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          ldsm_x4_trans(ha[mt], sw128_addr(hprev, 16 * kt + lr + 8 * (lq >> 1),
                                           4 * mb + 2 * mt + (lq & 1)));
#pragma unroll
        for (int np = 0; np < 2; ++np)
          ldsm_x4_trans(db[np], sw128_addr(dsl, 16 * kt + lr + 8 * (lq & 1),
                                           4 * nb + 2 * np + (lq >> 1)));
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            mma2(dWa[mt][2 * np], ha[mt], db[np][0], db[np][1]);
            mma2(dWa[mt][2 * np + 1], ha[mt], db[np][2], db[np][3]);
          }
      }
    }
    if (aborted) break;
    mbar_arrive(&done[st]);
  }
  if (aborted) {
    *abort_flag = 1;
    if (lane == 0) atomicExch(status, kStatusTimeout);
    return;
  }
  if (dH0) {
    float* hp = dH0 + (size_t)pair * kK * kV;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      *reinterpret_cast<float2*>(hp + r0 * kV + 8 * nt + 2 * c) = C[nt][0];
      *reinterpret_cast<float2*>(hp + r1 * kV + 8 * nt + 2 * c) = C[nt][1];
    }
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int l = 32 * mb + 16 * mt + g, j = 32 * nb + 8 * nt + 2 * c;
      *reinterpret_cast<float2*>(dWp + l * kV + j) = dWa[mt][nt][0];
      *reinterpret_cast<float2*>(dWp + (l + 8) * kV + j) = dWa[mt][nt][1];
    }
}

bool make_map(EncodeTiledFn enc, CUtensorMap* map, CUtensorMapDataType dt, const void* base,
              int esize, const cuuint64_t (&dims)[4], const cuuint32_t (&box)[4],
              CUtensorMapSwizzle swz) {
  const cuuint64_t strides[3] = {dims[0] * esize, dims[0] * dims[1] * esize,
                                 dims[0] * dims[1] * dims[2] * esize};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool bwd_mma_supports(int K, int V) { return K == kK && V == kV; }

cudaError_t launch_bwd_bf16_mma(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                int* status, cudaStream_t stream) {
  const BwdLayout L = bwd_layout();
  const cuuint64_t B = (cuuint64_t)p.B, T = (cuuint64_t)p.T, N = (cuuint64_t)p.N;
  CUtensorMap mh, mq, mk, mv, mdy;
  const cuuint64_t dh[4] = {kV, kK, T, B * N};
  const cuuint32_t bh[4] = {kV, kK, kTc, 1};
  const cuuint64_t dqk[4] = {kK, (cuuint64_t)p.Nqk, T, B};
  const cuuint32_t bqk[4] = {kK, 1, kTc, 1};
  const cuuint64_t dvv[4] = {kV, N, T, B};
  const cuuint32_t bvv[4] = {kV, 1, kTc, 1};
  if (!make_map(enc, &mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.Hs, 2, dh, bh,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(enc, &mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 2, dqk, bqk,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(enc, &mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, 2, dqk, bqk,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(enc, &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, 2, dvv, bvv,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(enc, &mdy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dy, 4, dvv, bvv,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(bwd_bf16_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  float* heads = p.ws + (size_t)p.B * p.N * backward_pair_floats(kK, kV);
  bwd_bf16_mma<<<(unsigned)(p.B * p.N), kThreads, L.total, stream>>>(
      mh, mq, mk, mv, mdy, (const uint16_t*)p.a, p.alpha, p.beta, (const uint16_t*)p.W, p.w_r,
      p.H0, p.dH_T, p.dq, p.dk, p.dv, p.da, p.dH0, p.ws, heads, p.T, p.N, p.Nqk, debug, status);
  err = cudaGetLastError();
  return err == cudaSuccess ? launch_bwd_reduce(p, stream) : err;
}

}  // namespace m2rnn
