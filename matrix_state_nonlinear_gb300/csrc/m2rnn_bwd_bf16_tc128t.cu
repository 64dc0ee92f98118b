// m2rnn_bwd_bf16_tc128t.cu — backward pass of the M²RNN recurrence for V = 128 and K <= 64 (a
// multiple of 16), every product of a step on the 5th-generation tensor cores, taken transposed
// so that the tensor-memory lanes run over the 128 value columns.
//
// Reverse scan of the M²RNN study notes, Sec. 2.7 (gate of Eq. (13)/(17)), on the kept bf16
// states S_t = bf16(H_t).  Per step t, from C_t = dL/dH_t (C_{T-1} = dH_T):
//   P_t = S_{t-1} W + k_t v_t^T (recomputed),  Z_t = tanh(P_t),
//   R_t = C_t + q_t u_t^T,  D_t = ((1 - f_t) R_t) ⊙ (1 - Z_t^2),
//   C_{t-1} = f_t R_t + D_t W^T,  dW += S_{t-1}^T D_t,  dL/df_t = <R_t, S_{t-1} - Z_t>,
//   dk_t = D_t v_t,  dv_t = D_t^T k_t + w_r ⊙ u_t,  dq_t = S_t u_t.
// The same scan as the V = 128 kernel whose products run over the state rows (rows padded to
// 128 there), with the two per-step products of the recurrence transposed:
//   P_{t-1}^T = W^T S_{t-2}^T + v_{t-1} k_{t-1}^T   (M = 128 columns j, N = K rows i)
//   G_t^T = W D_t^T                                  (M = 128, N = K)
// so that all 128 tensor-memory lanes hold real columns: thread (column j = 32 (warp & 3) + lane,
// row half warp >> 2) keeps f R of its <= 32 rows in fp32 and does the elementwise work of those
// rows, half the padded kernel's 64 entries at K = 64.  D_t is kept as its transpose (row j,
// column i, 128-byte swizzle), which every product reads in the form it needs: N-major for G^T,
// K-major for dW (= S^T D) and for dv (= D^T k), M-major for dk (= D v); the state tiles (row i)
// are read K-major for P^T and dq (= S u) and M-major for dW.  dL/df takes S_{t-1} by column
// from the state tile (one two-byte load per row; consecutive lanes read consecutive columns).
// Issue order, commits, the state ring, the input ring and the abort handling are those of the
// padded kernel.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 128;         // value width: the products' M (and dW's N)
constexpr int kR = 128;         // rows of the padded state tiles (state rows K .. 127 stay zero)
constexpr int kCompute = 256;   // 8 compute warps: lane quadrant (warp & 3) x row half (warp >> 2)
constexpr int kThreads = kCompute + 32;  // + the issuer warp
constexpr int kBarCompute = 1;  // named barrier of the compute warps
constexpr int kTile = kR * kV * 2;         // one bf16 128 x 128 tile: [2 column halves][128][128 B]
constexpr int kSmallTile = 16 * kV * 2;    // an N = 16 B operand: [2 K-blocks][16 rows][128 B]
constexpr int kSlots = 3;                  // state ring

// Tensor-memory columns.
constexpr uint32_t kTmemCols = 512;
// P^T and G^T take K <= 64 columns each; dW 128; dk, dv, dq 16 each.
constexpr uint32_t kColP = 0, kColG = 64, kColW = 128, kColDk = 256, kColDv = 272, kColDq = 288;

// Shared memory layout (bytes from a 1024-aligned base).
constexpr int kOffWt = 0;                          // W^T: row j, column l holds W[l][j]
constexpr int kOffD = kOffWt + kTile;              // D_t^T (bf16), row j, column i; [2] by t & 1
constexpr int kOffS = kOffD + 2 * kTile;           // state slots [kSlots]
constexpr int kOffBv = kOffS + kSlots * kTile;     // dk's B: row 0 = v_t
constexpr int kOffBk = kOffBv + kSmallTile;        // dv's B: row 0 = k_t (K index = row i)
constexpr int kOffBu = kOffBk + kSmallTile;        // dq's B: rows 0, 1 = bf16 hi, lo of u_{t-1}
constexpr int kOffAx = kOffBu + kSmallTile;        // rank-1 A (column 0 = v): [128 x 16] cores
constexpr int kOffBx = kOffAx + 4096;              // rank-1 B (column 0 = k): same layout
constexpr int kInBytes = kV * 4 + kV * 2 + 2 * kR * 2;  // u (f32), v, q, k (bf16)
constexpr int kOffIn = kOffBx + 4096;              // per-step inputs [3] by t % 3
constexpr int kInU = 0, kInV = kV * 4, kInQ = kInV + kV * 2, kInK = kInQ + kR * 2;
constexpr int kOffGate = kOffIn + 3 * kInBytes;    // float4 [3]: f, 1 - f, sigmoid(x), softplus(x)
constexpr int kOffDf = kOffGate + 3 * 16;          // float [2][8]: dL/df partials per warp
constexpr int kOffBar = kOffDf + 2 * 8 * 4;        // gp, rest, dready, full[kSlots], never; abort; slot
constexpr int kSmemBytes = kOffBar + 64 + 1024;    // + slack to align the base to 1024

__device__ __forceinline__ uint32_t sw128_off(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}
__device__ __forceinline__ uint32_t core_off(int r, int k) {  // no-swizzle, K = 16
  return (uint32_t)((r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// Gate of Eq. (13)/(17) and the factors of its derivative: f, 1 - f, sigmoid(x), softplus(x)
// with x = a + beta.
__device__ __forceinline__ float4 gate4(float a, float al, float be) {
  const float x = a + be;
  const float ex = expf(-fabsf(x));
  const float sp = fmaxf(x, 0.f) + log1pf(ex);
  const float sg = x >= 0.f ? 1.f / (1.f + ex) : ex / (1.f + ex);
  return make_float4(expf(-al * sp), -expm1f(-al * sp), sg, sp);
}


__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_tc128t(const __grid_constant__ CUtensorMap tm_h, const uint16_t* __restrict__ q,
                    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                    const uint16_t* __restrict__ a, const float* __restrict__ alpha,
                    const float* __restrict__ beta, const uint16_t* __restrict__ W,
                    const float* __restrict__ w_r, const float* __restrict__ H0,
                    const float* __restrict__ dy, const float* __restrict__ dH_T,
                    float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                    float* __restrict__ da, float* __restrict__ dH0, float* __restrict__ ws,
                    float* __restrict__ dqk_heads, int T, int N, int Nqk, int K, int debug,
                    int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool issuer = warp == kCompute / 32;
  const int qd = warp & 3, rh = (warp >> 2) & 1;
  const int j = 32 * qd + lane;   // column of this thread (and tensor-memory lane)
  const int r0 = 32 * rh;         // first of its rows
  const int nr = min(max(K - r0, 0), 32);  // its rows: r0 .. r0 + nr - 1 (a multiple of 16)
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const bool shared_qk = Nqk == 1 && N > 1;
  const int nq = Nqk == 1 ? 0 : n;
  const int krows = K >> 4;       // 16-row groups of the state
  const float al = alpha[n], be = beta[n];

  uint8_t* sWt = smem + kOffWt;
  uint8_t* sD = smem + kOffD;
  uint8_t* sBv = smem + kOffBv;
  uint8_t* sBk = smem + kOffBk;
  uint8_t* sBu = smem + kOffBu;
  uint8_t* sAx = smem + kOffAx;
  uint8_t* sBx = smem + kOffBx;
  float4* gates = reinterpret_cast<float4*>(smem + kOffGate);
  float* dfpart = reinterpret_cast<float*>(smem + kOffDf);
  uint64_t* gp_bar = reinterpret_cast<uint64_t*>(smem + kOffBar);  // G_t and P_{t-1} done
  uint64_t* rest_bar = gp_bar + 1;  // the whole batch done (dW, dk, dv, dq too)
  uint64_t* dready = gp_bar + 2;    // the compute warps' operands of a batch are written
  uint64_t* sfull = gp_bar + 3;     // [kSlots]
  uint64_t* never = gp_bar + 3 + kSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gp_bar + 4 + kSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gp_bar + 4 + kSlots) + 1;
  auto slot_of = [](int s) { return (s + 1) % kSlots; };  // state s >= -1
  auto state_tile = [&](int s) { return smem + kOffS + slot_of(s) * kTile; };
  auto state_parity = [&](int s) { return (uint32_t)((T - 1 - s) / kSlots) & 1u; };
  auto in_buf = [&](int t) { return smem + kOffIn + (t % 3) * kInBytes; };
  const long long limit = kWaitLimitCycles;

  // Copies of step t's inputs into in_buf(t) (threads 0 .. 63); thread 64 loads a_t.
  float a_pref = 0.f;
  auto fetch_inputs = [&](int t) {
    uint8_t* dst = in_buf(t);
    const size_t row = ((size_t)b * T + t) * N + n;
    const size_t qrow = ((size_t)b * T + t) * Nqk + nq;
    if (tid < 32) {
      cp_async16(dst + kInU + 16 * tid, dy + row * kV + 4 * tid);
    } else if (tid < 48) {
      cp_async16(dst + kInV + 16 * (tid - 32), v + row * kV + 8 * (tid - 32));
    } else if (tid < 64) {
      const int c = tid - 48;  // 16-byte chunks of q then k (K / 8 each)
      if (c < (K >> 3)) {
        cp_async16(dst + kInQ + 16 * c, q + qrow * K + 8 * c);
        cp_async16(dst + kInK + 16 * c, k + qrow * K + 8 * c);
      }
    } else if (tid == 64) {
      a_pref = bf16_bits_to_float(a[row]);
    }
    cp_async_commit();
  };
  auto put_gate = [&](int t) {
    if (tid == 64) gates[t % 3] = gate4(a_pref, al, be);
  };
  // The bf16 of H_0 (or zeros) as state -1, element by element over the compute threads;
  // thread 0 completes the slot's phase.
  auto put_h0 = [&]() {
    uint8_t* tile = state_tile(-1);
    const float* hp = H0 ? H0 + (size_t)pair * K * kV : nullptr;
    for (int e = tid; e < K * kV; e += kCompute) {
      const int i = e >> 7, c = e & 127;
      *reinterpret_cast<uint16_t*>(tile + sw128_off(i, c, kR)) =
          __bfloat16_as_ushort(__float2bfloat16_rn(hp ? hp[e] : 0.f));
    }
    fence_proxy_async_smem();
    named_bar_sync(kBarCompute, kCompute);
    if (tid == 0) mbar_arrive(&sfull[slot_of(-1)]);
  };
  // TMA of state s >= 0 into its slot (one lane).
  auto load_state = [&](int s) {
    uint64_t* bar = &sfull[slot_of(s)];
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * 64 * K * 2));
    tma_load_4d(state_tile(s), &tm_h, bar, 0, 0, s, pair);
    tma_load_4d(state_tile(s) + kR * 128, &tm_h, bar, 64, 0, s, pair);
  };

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    prefetch_tensormap(&tm_h);
    mbar_init(gp_bar, 1);
    mbar_init(rest_bar, 1);
    mbar_init(dready, kCompute / 32);
    for (int s = 0; s < kSlots; ++s) mbar_init(&sfull[s], 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  // Zero the D^T tiles, the state slots and the small tiles (padding stays 0).
  for (int e = tid; e < (kOffIn - kOffD) / 16; e += kThreads)
    reinterpret_cast<uint4*>(sD)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // the zeros before any TMA write into the same tiles
  // W^T tile: row j, column l holds W[l][j].
  const uint16_t* Wn = W + (size_t)n * kV * kV;
  for (int e = tid; e < kV * kV; e += kThreads) {
    const int l = e >> 7, jj = e & 127;
    *reinterpret_cast<uint16_t*>(sWt + sw128_off(jj, l, kR)) = Wn[e];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t idesc_p = umma_idesc_bf16(kV, K, false);             // W^T K-major, S K-major
  const uint32_t idesc_g = umma_idesc_bf16_ab(kV, K, true, true);     // W M-major, D^T N-major
  const uint32_t idesc_w = umma_idesc_bf16_ab(kV, kV, true, false);   // S M-major, D^T K-major
  const uint32_t idesc_dv = umma_idesc_bf16(kV, 16, false);           // D^T K-major, k row
  const uint32_t idesc_dk = umma_idesc_bf16(kR, 16, true);            // D^T M-major, v row
  const uint32_t idesc_dq = umma_idesc_bf16(kR, 16, false);           // S K-major, u rows
  // Descriptor bases: a tile at byte offset `off` from the 1024-aligned base has the base's
  // start-address field plus off / 16.  K-major tiles step 32 bytes per K = 16 inside a
  // 64-column block (the next block is 16 KB on, 2 KB in a 16-row tile); M/N-major reads step
  // 16 rows (2 KB), their second 64-wide M/N block 16 KB on.
  const uint64_t kbase = umma_desc(smem_u32(smem), 16, 1024, 2);
  const uint64_t mbase = umma_desc(smem_u32(smem), 16384, 1024, 2);
  auto at = [](uint64_t base, int off) { return base + (uint64_t)(off >> 4); };
  const uint64_t dAx = umma_desc(smem_u32(sAx), 128, 256, 0);
  const uint64_t dBx = umma_desc(smem_u32(sBx), 128, 256, 0);

  if (issuer) {
    // ======================================================= issuer warp
    // Batch t (t = T first: dq_{T-1} and P_{T-1} only) after the compute warps' signal; the
    // state ring as in the padded kernel.
    const bool leader = lane == 0;
    bool ok = true;
    if (leader) {
      for (int s = T - 1; s >= T - 3 && s >= 0; --s) load_state(s);
    }
    uint32_t dready_ph = 0, rest_ph = 0;
    for (int t = T; t >= 0 && ok; --t) {
      if (t < T && t - 3 >= 0) {
        ok = __all_sync(0xffffffffu,
                        wait_or_abort(rest_bar, rest_ph & 1u, limit, abort_flag));
        ++rest_ph;
        if (!ok) break;
        if (leader) load_state(t - 3);
      }
      bool w = wait_or_abort(dready, dready_ph & 1u, limit, abort_flag);
      ++dready_ph;
      if (t >= 1) w = w && wait_or_abort(&sfull[slot_of(t - 2)], state_parity(t - 2), limit,
                                         abort_flag);
      if (t >= 1) w = w && wait_or_abort(&sfull[slot_of(t - 1)], state_parity(t - 1), limit,
                                         abort_flag);
      if (t == T && (debug & kDebugForceTimeout))
        w = w && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      const int doff = kOffD + (t & 1) * kTile;
      const int s1 = kOffS + slot_of(t - 1) * kTile;
      if (t < T) {  // G_t^T = W D_t^T: A = the W^T tile read M-major, B = D^T read N-major
        umma4_if<128, 128>(leader, tmem + kColG, at(mbase, kOffWt), at(mbase, doff), idesc_g,
                           0u);
        umma4_if<128, 128>(leader, tmem + kColG, at(mbase, kOffWt + 8192),
                           at(mbase, doff + 8192), idesc_g, 1u);
      }
      if (t >= 1) {  // P_{t-1}^T = W^T S_{t-2}^T + v_{t-1} k_{t-1}^T
        const int s2 = kOffS + slot_of(t - 2) * kTile;
        umma4_if<2, 2>(leader, tmem + kColP, at(kbase, kOffWt), at(kbase, s2), idesc_p, 0u);
        umma4_if<2, 2>(leader, tmem + kColP, at(kbase, kOffWt + 16384), at(kbase, s2 + 16384),
                       idesc_p, 1u);
        umma_bf16_if(leader, tmem + kColP, dAx, dBx, idesc_p, 1u);
      }
      umma_commit_if(leader, gp_bar);
      if (t < T) {
        // dW += S_{t-1}^T D_t over the krows 16-row groups (A = S M-major, B = D^T K-major).
        const uint32_t acc0 = t < T - 1 ? 1u : 0u;
        if (krows == 4) {
          umma4_if<128, 2>(leader, tmem + kColW, at(mbase, s1), at(kbase, doff), idesc_w, acc0);
        } else {
          for (int kk = 0; kk < krows; ++kk)
            umma_bf16_if(leader, tmem + kColW, at(mbase, s1 + kk * 2048),
                         at(kbase, doff + kk * 32), idesc_w, kk == 0 ? acc0 : 1u);
        }
        // dk_t = D_t v_t: A = D^T read M-major (M = rows i), K = the 128 columns
        umma4_if<128, 2>(leader, tmem + kColDk, at(mbase, doff), at(kbase, kOffBv), idesc_dk, 0u);
        umma4_if<128, 2>(leader, tmem + kColDk, at(mbase, doff + 8192), at(kbase, kOffBv + 2048),
                         idesc_dk, 1u);
        // dv_t = D_t^T k_t: A = D^T K-major (M = columns j), K = the rows
        if (krows == 4) {
          umma4_if<2, 2>(leader, tmem + kColDv, at(kbase, doff), at(kbase, kOffBk), idesc_dv, 0u);
        } else {
          for (int kk = 0; kk < krows; ++kk)
            umma_bf16_if(leader, tmem + kColDv, at(kbase, doff + kk * 32),
                         at(kbase, kOffBk + kk * 32), idesc_dv, kk == 0 ? 0u : 1u);
        }
      }
      if (t >= 1) {  // dq_{t-1} = S_{t-1} u_{t-1}
        umma4_if<2, 2>(leader, tmem + kColDq, at(kbase, s1), at(kbase, kOffBu), idesc_dq, 0u);
        umma4_if<2, 2>(leader, tmem + kColDq, at(kbase, s1 + 16384), at(kbase, kOffBu + 2048),
                       idesc_dq, 1u);
      }
      umma_commit_if(leader, rest_bar);
    }
    if (!ok && leader) {
      *abort_flag = 1;
      atomicExch(status, kStatusTimeout);
    }
  } else {
    // ======================================================= compute warps
    const uint32_t t_lane = tmem + ((uint32_t)(32 * qd) << 16);
    // The running f R of this thread's column over its rows (pairs of rows): C_{T-1} = dH_T
    // (or 0), no G yet.
    float2 cf[16];
    {
      const float* gp = dH_T ? dH_T + (size_t)pair * K * kV + j : nullptr;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = r0 + 2 * u;
        cf[u] = (gp && 2 * u < nr) ? make_float2(gp[(size_t)i * kV], gp[(size_t)(i + 1) * kV])
                                   : make_float2(0.f, 0.f);
      }
    }
    float dwr_acc = 0.f, dal_acc = 0.f, dbe_acc = 0.f;
    const float wr_j = w_r[(size_t)n * kV + j];
    if (T <= 2) put_h0();
    fetch_inputs(T - 1);

    // Small operands of the batch issued after step t (t = T: the first batch): the rank-1 of
    // step t - 1 (v over the product rows j, k over the state rows), dq_{t-1}'s u rows, and for
    // t < T dk_t's v and dv_t's k rows.
    auto put_small = [&](int t) {
      if (t - 1 >= 0) {
        const uint8_t* in1 = in_buf(t - 1);
        if (rh == 0) {
          *reinterpret_cast<uint16_t*>(sAx + core_off(j, 0)) =
              reinterpret_cast<const uint16_t*>(in1 + kInV)[j];
        } else if (j < K) {
          *reinterpret_cast<uint16_t*>(sBx + core_off(j, 0)) =
              reinterpret_cast<const uint16_t*>(in1 + kInK)[j];
        }
        if (tid < 64) {  // u_{t-1} as bf16 hi (row 0) and lo (row 1) parts
          const float2 x = reinterpret_cast<const float2*>(in1 + kInU)[tid];
          const uint32_t hi = pack_bf16x2(x.x, x.y);
          const float2 hf = bf16x2_to_float2(hi);
          *reinterpret_cast<uint32_t*>(sBu + sw128_off(0, 2 * tid, 16)) = hi;
          *reinterpret_cast<uint32_t*>(sBu + sw128_off(1, 2 * tid, 16)) =
              pack_bf16x2(x.x - hf.x, x.y - hf.y);
        }
      }
      if (t < T) {
        const uint8_t* in0 = in_buf(t);
        if (rh == 0) {  // dv's B row 0: k_t over the rows (K index = row i)
          if (j < K)
            *reinterpret_cast<uint16_t*>(sBk + sw128_off(0, j, 16)) =
                reinterpret_cast<const uint16_t*>(in0 + kInK)[j];
        } else {        // dk's B row 0: v_t over the columns
          *reinterpret_cast<uint16_t*>(sBv + sw128_off(0, j, 16)) =
              reinterpret_cast<const uint16_t*>(in0 + kInV)[j];
        }
      }
      fence_proxy_async_smem();
    };
    // Every compute warp has written its operands of the next batch: one arrive per warp.
    auto signal = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dready);
    };
    // dq_t and dk_{t+1} (row half 0: tensor-memory lane = row i = j, rows < K) and dv_{t+1}
    // (row half 1: lane = column j).
    auto small_outputs = [&](int t) {
      const int tn = t + 1;
      if (rh == 0) {
        float dq0 = 0.f, dq1 = 0.f, dkn = 0.f;
        if (t >= 0) {
          dq0 = tmem_ld1(t_lane + kColDq);
          dq1 = tmem_ld1(t_lane + kColDq + 1);
        }
        if (tn < T) dkn = tmem_ld1(t_lane + kColDk);
        if (j < K) {
          const int hs = shared_qk ? N : Nqk, hq = shared_qk ? n : nq;
          float* dqo = shared_qk ? dqk_heads : dq;
          float* dko = shared_qk ? dqk_heads + (size_t)gridDim.x * T * K : dk;
          if (t >= 0) dqo[(((size_t)b * T + t) * hs + hq) * K + j] = dq0 + dq1;
          if (tn < T) dko[(((size_t)b * T + tn) * hs + hq) * K + j] = dkn;
        }
      } else if (tn < T) {
        const float dvn = tmem_ld1(t_lane + kColDv);
        const float un = reinterpret_cast<const float*>(in_buf(tn) + kInU)[j];
        dv[(((size_t)b * T + tn) * N + n) * kV + j] = fmaf(wr_j, un, dvn);
      }
    };

    // First batch's operands (step T - 1's inputs).
    cp_async_wait_all();
    named_bar_sync(kBarCompute, kCompute);
    put_small(T);
    put_gate(T - 1);
    signal();

    bool abort = false, has_g = false;
    uint32_t gp_ph = 0, rest_ph = 0;
    for (int t = T - 1; t >= 0; --t) {
      // G_{t+1}^T and P_t^T (the first commit of the batch issued after step t + 1).
      bool ok = wait_or_abort(gp_bar, gp_ph & 1u, limit, abort_flag);
      ++gp_ph;
      tc_fence_before();
      abort = named_bar_or(kBarCompute, kCompute, !ok);
      if (abort) break;
      tc_fence_after();
      if (t >= 1) fetch_inputs(t - 1);  // into the buffer step t + 2 used

      // ---- elementwise step t
      const uint8_t* in0 = in_buf(t);
      const float4 gt = gates[t % 3];
      // ff = f_t; ngg = -(1 - f_t), paired with Z^2 - 1 below (no negated operand)
      const float2 ff = make_float2(gt.x, gt.x), ngg = make_float2(-gt.y, -gt.y);
      const float uj = reinterpret_cast<const float*>(in0 + kInU)[j];
      const float2 u2 = make_float2(uj, uj);
      const uint16_t* qrow = reinterpret_cast<const uint16_t*>(in0 + kInQ);
      const uint8_t* sprev = state_tile(t - 1);
      uint8_t* dcur = sD + (t & 1) * kTile;
      // Every thread observes the load of S_{t-1} before reading it.
      ok = wait_or_abort(&sfull[slot_of(t - 1)], state_parity(t - 1), limit, abort_flag);
      float2 dfp = make_float2(0.f, 0.f);
#pragma unroll
      for (int piece = 0; piece < 2; ++piece) {
        if (16 * piece < nr) {  // warp-uniform
          const int ib = r0 + 16 * piece;  // rows ib .. ib + 15
          float pv[16], gv[16];
          tmem_ld16_nowait(t_lane + kColP + ib, pv);
          if (has_g) tmem_ld16_nowait(t_lane + kColG + ib, gv);
          const uint4 qa = *reinterpret_cast<const uint4*>(qrow + ib);
          const uint4 qb = *reinterpret_cast<const uint4*>(qrow + ib + 8);
          const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
          uint32_t sw[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t s_lo = *reinterpret_cast<const uint16_t*>(
                sprev + sw128_off(ib + 2 * e, j, kR));
            const uint32_t s_hi = *reinterpret_cast<const uint16_t*>(
                sprev + sw128_off(ib + 2 * e + 1, j, kR));
            sw[e] = s_lo | (s_hi << 16);
          }
          tmem_wait_ld();
          uint32_t dpk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int u = 8 * piece + e;  // row pair (ib + 2e, ib + 2e + 1)
            const float2 z = make_float2(tanh_mufu(pv[2 * e]), tanh_mufu(pv[2 * e + 1]));
            const float2 c = has_g ? add2(cf[u], make_float2(gv[2 * e], gv[2 * e + 1])) : cf[u];
            const float2 r = fma2(bf16x2_to_float2(qw[e]), u2, c);     // R = C + q u^T
            const float2 zz1 = fma2(z, z, make_float2(-1.f, -1.f));   // Z^2 - 1
            const float2 d = mul2(mul2(ngg, r), zz1);                 // D = (1 - f) R (1 - Z^2)
            dfp = fma2(r, sub2(bf16x2_to_float2(sw[e]), z), dfp);     // <R, S_{t-1} - Z>
            cf[u] = mul2(ff, r);                                      // f R, for C_{t-1}
            dpk[e] = pack_bf16x2(d.x, d.y);
          }
          // D^T row j, columns ib .. ib + 15.
          *reinterpret_cast<uint4*>(dcur + sw128_off(j, ib, kR)) =
              make_uint4(dpk[0], dpk[1], dpk[2], dpk[3]);
          *reinterpret_cast<uint4*>(dcur + sw128_off(j, ib + 8, kR)) =
              make_uint4(dpk[4], dpk[5], dpk[6], dpk[7]);
        }
      }
      has_g = true;
      // dL/df_t partial of the warp; dw_r += u_t ⊙ v_t (row half 1: one thread per column).
      float dsum = dfp.x + dfp.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
      if (lane == 0) dfpart[(t & 1) * 8 + warp] = dsum;
      if (rh == 1)
        dwr_acc = fmaf(uj, bf16_bits_to_float(reinterpret_cast<const uint16_t*>(in0 + kInV)[j]),
                       dwr_acc);

      // The second commit of the batch issued after step t + 1 (dW_{t+1}, dk_{t+1}, dv_{t+1},
      // dq_t): its outputs, and the operand tiles it read are free again.
      ok = wait_or_abort(rest_bar, rest_ph & 1u, limit, abort_flag) && ok;
      ++rest_ph;
      cp_async_wait_all();  // step t - 1's inputs
      tc_fence_before();
      abort = named_bar_or(kBarCompute, kCompute, !ok);
      if (abort) break;
      tc_fence_after();
      small_outputs(t);
      put_small(t);
      if (t >= 1) put_gate(t - 1);
      if (t == 2) put_h0();  // state 2's slot is free: state -1 for batches 1 and 0
      signal();
      if (tid == 32) {  // da_t and the dalpha, dbeta sums
        float df = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) df += dfpart[(t & 1) * 8 + w];
        const float d_a = df * (-al * gt.x * gt.z);
        da[((size_t)b * T + t) * N + n] = d_a;
        dal_acc = fmaf(df, -gt.x * gt.w, dal_acc);
        dbe_acc += d_a;
      }
    }

    if (!abort) {
      // The last batch: G_0^T, then dW_0, dk_0, dv_0.
      bool ok2 = wait_or_abort(gp_bar, gp_ph & 1u, limit, abort_flag);
      ok2 = wait_or_abort(rest_bar, rest_ph & 1u, limit, abort_flag) && ok2;
      tc_fence_before();
      abort = named_bar_or(kBarCompute, kCompute, !ok2);
      tc_fence_after();
      if (!abort) {
        small_outputs(-1);
        // dH_0 = C_{-1} = f_0 R_0 + G_0.
        if (dH0) {
          float* hp = dH0 + (size_t)pair * K * kV + j;
#pragma unroll
          for (int piece = 0; piece < 2; ++piece) {
            if (16 * piece < nr) {
              const int ib = r0 + 16 * piece;
              float gv[16];
              tmem_ld16_nowait(t_lane + kColG + ib, gv);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float2 c = add2(cf[8 * piece + e], make_float2(gv[2 * e], gv[2 * e + 1]));
                hp[(size_t)(ib + 2 * e) * kV] = c.x;
                hp[(size_t)(ib + 2 * e + 1) * kV] = c.y;
              }
            }
          }
        }
        // This pair's dW (tensor-memory lane l, columns j'), dw_r, dalpha and dbeta partials.
        float* wsp = ws + (size_t)pair * backward_pair_floats(K, kV);
        float* dWp = wsp + (size_t)K * kV;
        float* dwr_p = dWp + kV * kV;
        float* ab_p = dwr_p + kV;
        const int c0 = 64 * rh;
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          float wv[16];
          tmem_ld16_nowait(t_lane + kColW + c0 + 16 * piece, wv);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(dWp + (size_t)j * kV + c0 + 16 * piece + e) =
                make_float4(wv[e], wv[e + 1], wv[e + 2], wv[e + 3]);
        }
        if (rh == 1) dwr_p[j] = dwr_acc;
        if (tid == 32) {
          ab_p[0] = dal_acc;
          ab_p[1] = dbe_acc;
        }
      }
    }
    if (abort && tid == 0) {
      *abort_flag = 1;
      atomicExch(status, kStatusTimeout);
    }
    cp_async_wait_all();
  }

  // Before tensor memory is released every issued product and TMA load must be done: wait
  // (bounded) for the last phase of each barrier that may still complete.
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    mbar_wait_bounded(gp_bar, 0u, kDebugWaitLimitCycles);
    mbar_wait_bounded(gp_bar, 1u, kDebugWaitLimitCycles);
    mbar_wait_bounded(rest_bar, 0u, kDebugWaitLimitCycles);
    mbar_wait_bounded(rest_bar, 1u, kDebugWaitLimitCycles);
    for (int s = 0; s < kSlots; ++s) {
      mbar_wait_bounded(&sfull[s], 0u, kDebugWaitLimitCycles);
      mbar_wait_bounded(&sfull[s], 1u, kDebugWaitLimitCycles);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool bwd_tc128t_supports(int K, int V) { return V == kV && K >= 16 && K <= 64 && K % 16 == 0; }

cudaError_t launch_bwd_bf16_tc128t(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                   int* status, cudaStream_t stream) {
  if (!bwd_tc128t_supports(p.K, p.V) || p.T < 1) return cudaErrorInvalidValue;
  // Kept states [B N, T, K, V] bf16: a box of 64 columns x K rows of one step (128-byte
  // swizzle, the K-major operand layout).
  CUtensorMap mh;
  const cuuint64_t dims[4] = {(cuuint64_t)kV, (cuuint64_t)p.K, (cuuint64_t)p.T,
                              (cuuint64_t)p.B * p.N};
  const cuuint64_t strides[3] = {(cuuint64_t)kV * 2, (cuuint64_t)kV * 2 * p.K,
                                 (cuuint64_t)kV * 2 * p.K * p.T};
  const cuuint32_t box[4] = {64u, (cuuint32_t)p.K, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  if (enc(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p.Hs), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(bwd_bf16_tc128t,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  float* heads = p.ws + (size_t)p.B * p.N * backward_pair_floats(p.K, p.V);
  bwd_bf16_tc128t<<<(unsigned)(p.B * p.N), kThreads, kSmemBytes, stream>>>(
      mh, (const uint16_t*)p.q, (const uint16_t*)p.k, (const uint16_t*)p.v, (const uint16_t*)p.a,
      p.alpha, p.beta, (const uint16_t*)p.W, p.w_r, p.H0, p.dy, p.dH_T, p.dq, p.dk, p.dv, p.da,
      p.dH0, p.ws, heads, p.T, p.N, p.Nqk, p.K, debug, status);
  err = cudaGetLastError();
  return err == cudaSuccess ? launch_bwd_reduce(p, stream) : err;
}

}  // namespace m2rnn
