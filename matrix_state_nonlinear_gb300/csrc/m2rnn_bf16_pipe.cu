// m2rnn_bf16_pipe.cu — software-pipelined bf16-operand / fp32-state forward recurrence
// on the warp-level tensor-core MMA, for K <= 64 and V in {16, 32, 64} (W held in
// registers).
//
// Same recurrence and mapping as the row-warp kernel (M²RNN study notes, Sec. 2.1
// Eq. (10)-(12), Sec. 2.2 Eq. (13)/(17); one thread block per (batch, head) pair,
// warp w owns rows 16w .. 16w+15 of H in registers), with two changes that let the
// MUFU tanh and the tensor-core MMA of one warp run at the same time:
//
//  * Step wavefront.  The bf16 A fragment of k-tile j of H_t is packed from the
//    accumulators of n-tiles 2j and 2j+1 alone, so the MMA of step t+1 for k-tile
//    j can start as soon as those two n-tiles of step t have been through
//    tanh and the gate lerp.  Each step therefore runs, for j = 0 .. V/16-1:
//      tanh + lerp of n-tiles 2j, 2j+1 (step t)  ->  pack A_j  ->  MMA(step t+1, k-tile j)
//    and the MMAs of k-tile j overlap the tanh of k-tile j+1.  Two accumulator
//    sets alternate: P_t being consumed, P_{t+1} being built (initialised with the
//    rank-1 term k_{t+1} v_{t+1}^T).
//
//  * Deferred readout.  The q-weighted row sums of H_t are formed at the end of step
//    t, but their shuffle reduce-scatter runs one stage per k-tile phase of step
//    t+1, so the dependent shuffle chain overlaps that step's MUFU and MMA work
//    instead of stalling the in-order issue of one warp.
//
//  * Inputs one step ahead (plain forward).  A step's shared-memory operands (gates and
//    q of step t, k and v of step t+1) are loaded into registers during the step before,
//    so that no step waits on a shared-memory load.
//
//  * Producer warp.  An extra warp issues the TMA loads of q, k, v chunks,
//    computes the gates (f, 1 - f) of a chunk before its load is armed, and sums
//    the per-warp readout partials (+ w_r ⊙ v) into y after the compute warps
//    finish a chunk.  Compute warps and the producer meet only through
//    mbarriers (full: inputs and gates ready; done: a chunk's partials written),
//    never through a block-wide barrier inside the time loop.
//
// fp32 elementwise math uses the packed f32x2 instructions (two lanes of work per
// issue slot); tanh is the MUFU tanh.approx.f32.
#include <cuda_bf16.h>

#include <cstring>
#include <type_traits>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

struct PipeLayout {
  int qs, ks, vs, stage_bytes;  // TMA destinations, two stages `stage_bytes` apart
  int fg;                       // float2 [2][Tc]          (f, 1 - f) per step
  int ypart;                    // float  [2][nw][Tc+1][V] per-warp readout partials (row Tc: scratch
                                //                          target of the empty first pending readout)
  int wr;                       // float  [V]
  int bar;                      // uint64 full[2], done[2], never-armed[1]; int abort
  int hring;                    // state-keeping forward, V = 64: [nw][2 slots][2 steps][16 rows][64]
                                //   bf16, 128-byte swizzled, staged for TMA stores (+1024 to align)
  int total;
};

__host__ __device__ inline int al128(int x) { return (x + 127) & ~127; }

__host__ __device__ inline PipeLayout pipe_layout(int K, int V, int Tc, bool ring = false) {
  PipeLayout L;
  const int nw = K / 16;
  L.qs = 0;
  L.ks = al128(Tc * K * 2);
  L.vs = L.ks + al128(Tc * K * 2);
  L.stage_bytes = L.vs + al128(Tc * V * 2);
  int o = 2 * L.stage_bytes;
  L.fg = o;
  o += al128(2 * Tc * 8);
  L.ypart = o;
  o += al128(2 * nw * (Tc + 1) * V * 4);
  L.wr = o;
  o += al128(V * 4);
  L.bar = o;
  o += 128;
  L.hring = o;
  if (ring) o += nw * 4 * 16 * V * 2 + 1024;
  L.total = o;
  return L;
}

template <int VT, bool kCache>
__global__ void __launch_bounds__(160, 1)
    fwd_bf16_mma_pipe(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_hs,
                      const __grid_constant__ CUtensorMap tm_hs1, const uint16_t* __restrict__ a,
                      const float* __restrict__ alpha, const float* __restrict__ beta,
                      const uint16_t* __restrict__ W, const float* __restrict__ w_r,
                      const float* H0, float* __restrict__ y, float* H_T, uint16_t* __restrict__ Hs,
                      int T, int N, int K, int Tc, int qk_hs, int debug, int* status) {
  constexpr int V = 16 * VT;
  constexpr int NT = 2 * VT;  // n-tiles of 8 columns
  constexpr int M = 4 * VT;   // readout partial sums per thread

  extern __shared__ __align__(128) uint8_t smem[];
  const int nw = K / 16;  // compute warps; warp nw is the producer
  // V = 64 keeps the states through a shared-memory ring and TMA tensor stores.
  constexpr bool kRing = kCache && VT == 4;
  const PipeLayout L = pipe_layout(K, V, Tc, kRing);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + Tc - 1) / Tc;
  const size_t row_base = (size_t)b * T;  // (b, t) row index base

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* done = full + 2;
  uint64_t* never = full + 4;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 5);
  float2* fgs = reinterpret_cast<float2*>(smem + L.fg);
  float* ypart = reinterpret_cast<float*>(smem + L.ypart);
  float* wrs = reinterpret_cast<float*>(smem + L.wr);
  const long long limit = kWaitLimitCycles;

  if (tid == 0) {
    // Every lane of the producer (full) and of each compute warp (done) arrives, so
    // each thread's own shared-memory writes are released by its own arrive.
    mbar_init(&full[0], 32);
    mbar_init(&full[1], 32);
    mbar_init(&done[0], 32 * nw);
    mbar_init(&done[1], 32 * nw);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int j = tid; j < V; j += blockDim.x) wrs[j] = w_r[(size_t)n * V + j];
  __syncthreads();

  // ======================================================= producer warp
  if (warp == nw) {
    const float al = alpha[n], be = beta[n];
    const uint32_t stage_tx = (uint32_t)(2 * K + V) * (uint32_t)Tc * 2u;
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    // Gates of chunk cc into fg[cc & 1], then arm full[cc & 1] and start the TMA.
    auto arm = [&](int cc) {
      const int st = cc & 1;
      for (int s = lane; s < Tc; s += 32) {
        const int t = cc * Tc + s;
        const float av = t < T ? bf16_bits_to_float(a[(row_base + t) * N + n]) : 0.f;
        fgs[st * Tc + s] = gate_fg(av, al, be);
      }
      __syncwarp();
      if (lane != 0) {
        mbar_arrive(&full[st]);
      } else {
        uint8_t* base = smem + st * L.stage_bytes;
        mbar_arrive_expect_tx(&full[st], stage_tx);
        tma_load_4d(base + L.qs, &tm_q, &full[st], 0, n * qk_hs, cc * Tc, b);
        tma_load_4d(base + L.ks, &tm_k, &full[st], 0, n * qk_hs, cc * Tc, b);
        tma_load_4d(base + L.vs, &tm_v, &full[st], 0, n, cc * Tc, b);
      }
    };
    int issued = 0;
    for (; issued < 2 && issued < nchunks; ++issued) arm(issued);

    for (int cc = 0; cc < nchunks; ++cc) {
      const int st = cc & 1;
      const bool dok = kRing ? wait_or_abort(&done[st], (uint32_t)(cc >> 1) & 1u, limit, abort_flag)
                             : wait_or_abort_sleep(&done[st], (uint32_t)(cc >> 1) & 1u, limit,
                                                   abort_flag);
      if (!dok) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicExch(status, kStatusTimeout);
          // Let TMA copies still in flight land before the block's shared memory goes away.
          for (int ci = cc; ci < issued; ++ci)
            if (kRing)
              mbar_wait_bounded(&full[ci & 1], (uint32_t)(ci >> 1) & 1u, kDebugWaitLimitCycles);
            else
              mbar_wait_bounded_sleep(&full[ci & 1], (uint32_t)(ci >> 1) & 1u,
                                      kDebugWaitLimitCycles);
        }
        return;
      }
      // y_t = sum of the per-warp partials + w_r ⊙ v_t, float4 per lane.
      const int t0 = cc * Tc;
      const int steps = min(Tc, T - t0);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + st * L.stage_bytes + L.vs);
      const float* yp = ypart + (size_t)st * nw * (Tc + 1) * V;
      constexpr int V4 = V / 4;
      for (int idx = lane; idx < steps * V4; idx += 32) {
        const int s = idx / V4, j = (idx - s * V4) * 4;
        const uint2 vv = *reinterpret_cast<const uint2*>(vs + s * V + j);
        const float4 w4 = *reinterpret_cast<const float4*>(wrs + j);
        float4 o = make_float4(w4.x * bf16_lo(vv.x), w4.y * bf16_hi(vv.x), w4.z * bf16_lo(vv.y),
                               w4.w * bf16_hi(vv.y));
        for (int w = 0; w < nw; ++w) {
          const float4 u = *reinterpret_cast<const float4*>(yp + ((size_t)w * (Tc + 1) + s) * V + j);
          o.x += u.x;
          o.y += u.y;
          o.z += u.z;
          o.w += u.w;
        }
        *reinterpret_cast<float4*>(y + ((row_base + t0 + s) * N + n) * V + j) = o;
      }
      __syncwarp();
      if (issued < nchunks) arm(issued++);
    }
    return;
  }

  // ======================================================= compute warps
  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;

  // W as m16n8k16 B fragments (k index = row l of W, n index = column j).
  const uint16_t* Wn = W + (size_t)n * V * V;
  uint32_t wb[VT][NT][2];
#pragma unroll
  for (int kt = 0; kt < VT; ++kt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = 8 * nt + g, r = 16 * kt + 2 * c;
      wb[kt][nt][0] = (uint32_t)Wn[r * V + col] | ((uint32_t)Wn[(r + 1) * V + col] << 16);
      wb[kt][nt][1] = (uint32_t)Wn[(r + 8) * V + col] | ((uint32_t)Wn[(r + 9) * V + col] << 16);
    }

  // H_0 (fp32) in the accumulator layout: h[nt][0] = row r0, h[nt][1] = row r1,
  // columns 8 nt + 2c and 8 nt + 2c + 1.
  float2 h[NT][2];
  if (H0) {
    const float* hp = H0 + (size_t)pair * K * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      h[nt][0] = *reinterpret_cast<const float2*>(hp + (size_t)r0 * V + 8 * nt + 2 * c);
      h[nt][1] = *reinterpret_cast<const float2*>(hp + (size_t)r1 * V + 8 * nt + 2 * c);
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) h[nt][0] = h[nt][1] = make_float2(0.f, 0.f);
  }

  bool ok = kRing ? wait_or_abort(&full[0], 0u, limit, abort_flag)
                  : wait_or_abort_sleep(&full[0], 0u, limit, abort_flag);
  if (debug & kDebugForceTimeout)
    ok = ok && (kRing ? mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles)
                      : mbar_wait_bounded_sleep(never, 0u, kDebugWaitLimitCycles));
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicExch(status, kStatusTimeout);
    return;
  }

  // P_0 = k_0 v_0^T + H_0 W.
  float2 acc[NT][2];
  uint32_t af[VT][4];
  {
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(smem + L.ks);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + L.vs);
    const float2 k0 = make_float2(bf16_bits_to_float(ks[r0]), bf16_bits_to_float(ks[r0]));
    const float2 k1 = make_float2(bf16_bits_to_float(ks[r1]), bf16_bits_to_float(ks[r1]));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 vv = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vs + 8 * nt + 2 * c));
      acc[nt][0] = mul2(k0, vv);
      acc[nt][1] = mul2(k1, vv);
    }
#pragma unroll
    for (int kt = 0; kt < VT; ++kt) {
      af[kt][0] = pack_bf16x2(h[2 * kt][0].x, h[2 * kt][0].y);
      af[kt][1] = pack_bf16x2(h[2 * kt][1].x, h[2 * kt][1].y);
      af[kt][2] = pack_bf16x2(h[2 * kt + 1][0].x, h[2 * kt + 1][0].y);
      af[kt][3] = pack_bf16x2(h[2 * kt + 1][1].x, h[2 * kt + 1][1].y);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma2(acc[nt], af[kt], wb[kt][nt][0], wb[kt][nt][1]);
    }
  }

  // One time step.  On entry `cur` holds P_t (complete) and h holds H_{t-1}; on
  // exit h holds H_t and `nxt` holds P_{t+1} (its last MMAs may still be in flight).
  // Program order interleaves each MMA of step t+1 with one MUFU tanh of step t, so
  // that in-order issue keeps the tensor pipe and the MUFU busy together.
  float2 nxt[NT][2];
  bool aborted = false;
  // Reduce-scatter stage `stg` of a pending readout (lane bits 4, 3, 2), and its store.
  auto red_stage = [&](float (&p)[M], int stg) {
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
  };
  auto red_store = [&](float (&p)[M], float* yrow) {
    if constexpr (M >= 8) {
      constexpr int cnt = M / 8;
#pragma unroll
      for (int i = 0; i < cnt; ++i) {
        const int m = cnt * g + i;
        yrow[8 * (m >> 1) + 2 * c + (m & 1)] = p[i];
      }
    } else {
      if ((g & 1) == 0) {
        const int m = g >> 1;
        yrow[8 * (m >> 1) + 2 * c + (m & 1)] = p[0];
      }
    }
  };
  auto yrow_of = [&](int cc, int s) {
    return ypart + (((size_t)(cc & 1) * nw + warp) * (Tc + 1) + s) * V;
  };
  // A step's shared-memory inputs, loaded one step ahead so that their latency overlaps
  // the previous step: the gates and q of step t, k and v of step t + 1.
  struct StepIn {
    float2 fg;
    uint16_t k0, k1, q0, q1;
    uint32_t v[NT];
  };
  // Inputs of the step after (cc, s): gates and q of step s + 1, k and v of step s + 2
  // (either may be in the next chunk's stage; past the end of the sequence they are
  // stale and never used).
  auto fetch = [&](StepIn& in, int cc, int s, int steps) {
    const int st = cc & 1;
    const bool n1 = s + 1 >= steps, n2 = s + 2 >= steps;
    const int st1 = n1 ? st ^ 1 : st, s1 = n1 ? s + 1 - steps : s + 1;
    const int st2 = n2 ? st ^ 1 : st, s2 = n2 ? s + 2 - steps : s + 2;
    in.fg = fgs[st1 * Tc + s1];
    const uint8_t* b1 = smem + st1 * L.stage_bytes;
    const uint8_t* b2 = smem + st2 * L.stage_bytes;
    const uint16_t* qs = reinterpret_cast<const uint16_t*>(b1 + L.qs) + s1 * K;
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(b2 + L.ks) + s2 * K;
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(b2 + L.vs) + s2 * V;
    in.q0 = qs[r0];
    in.q1 = qs[r1];
    in.k0 = ks[r0];
    in.k1 = ks[r1];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      in.v[nt] = *reinterpret_cast<const uint32_t*>(vs + 8 * nt + 2 * c);
  };
  auto step = [&](float2 (&cur)[NT][2], float2 (&nx)[NT][2], int cc, int s, int steps,
                  float (&pin)[M], float (&pout)[M], StepIn& in, bool odd) {
    // odd: the second step of a two-step trip (a literal at every call, folded when inlined)
    float* pin_row = yrow_of(cc, s > 0 ? s - 1 : Tc);
    const int st = cc & 1;
    const uint8_t* sbase = smem + st * L.stage_bytes;
    // Step t+1 is the first of the next chunk when s is the chunk's last step (its
    // inputs were waited for before this step).  Selects, not branches, so that a
    // step body stays one basic block the compiler can schedule as a whole.
    const bool last = s == steps - 1;
    const uint8_t* nbase = last ? smem + (st ^ 1) * L.stage_bytes : sbase;
    const int sn = last ? 0 : s + 1;
    // The state-keeping form loads its inputs within the step (one step ahead it ran
    // slower: 6.49 against 6.25 ms at the headline shape); the plain forward uses the
    // registers loaded during the step before.
    StepIn cin;
    if constexpr (!kRing) {
      cin = in;
      fetch(in, cc, s, steps);
    }
    float2 fg;
    if constexpr (kRing)
      fg = fgs[st * Tc + s];
    else
      fg = cin.fg;
    const float2 ff = make_float2(fg.x, fg.x), gg = make_float2(fg.y, fg.y);

    // Rank-1 k_{t+1} v_{t+1}^T initialises P_{t+1}.  (After the last step of the
    // sequence this reads stale inputs; the result is never used.)
    if constexpr (kRing) {
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(nbase + L.ks) + sn * K;
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(nbase + L.vs) + sn * V;
      const float kv0 = bf16_bits_to_float(ks[r0]), kv1 = bf16_bits_to_float(ks[r1]);
      const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 vv = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vs + 8 * nt + 2 * c));
        nx[nt][0] = mul2(k0, vv);
        nx[nt][1] = mul2(k1, vv);
      }
    } else {
      const float kv0 = bf16_bits_to_float(cin.k0), kv1 = bf16_bits_to_float(cin.k1);
      const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 vv = bf16x2_to_float2(cin.v[nt]);
        nx[nt][0] = mul2(k0, vv);
        nx[nt][1] = mul2(k1, vv);
      }
    }
    // k-tile 0 of H_t.
    {
      float z[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 pv = cur[e >> 2][(e >> 1) & 1];
        z[e] = tanh_mufu((e & 1) ? pv.y : pv.x);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
        h[e >> 1][e & 1] = fma2(gg, make_float2(z[2 * e], z[2 * e + 1]), mul2(ff, h[e >> 1][e & 1]));
      af[0][0] = pack_bf16x2(h[0][0].x, h[0][0].y);
      af[0][1] = pack_bf16x2(h[0][1].x, h[0][1].y);
      af[0][2] = pack_bf16x2(h[1][0].x, h[1][0].y);
      af[0][3] = pack_bf16x2(h[1][1].x, h[1][1].y);
    }
    red_stage(pin, 0);
    // Phases kt = 0 .. VT-1: MMAs of step t+1 on k-tile kt, interleaved with the
    // tanh of k-tile kt+1 of step t.
#pragma unroll
    for (int kt = 0; kt < VT; ++kt) {
      float z[8];
      constexpr int E = NT > 8 ? NT : 8;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (e < NT) mma2(nx[e], af[kt], wb[kt][e][0], wb[kt][e][1]);
        if (kt + 1 < VT && e < 8) {
          const float2 pv = cur[2 * (kt + 1) + (e >> 2)][(e >> 1) & 1];
          z[e] = tanh_mufu((e & 1) ? pv.y : pv.x);
        }
      }
      if (kt + 1 < VT) {
        const int n0 = 2 * (kt + 1);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          h[n0 + (e >> 1)][e & 1] =
              fma2(gg, make_float2(z[2 * e], z[2 * e + 1]), mul2(ff, h[n0 + (e >> 1)][e & 1]));
        af[kt + 1][0] = pack_bf16x2(h[n0][0].x, h[n0][0].y);
        af[kt + 1][1] = pack_bf16x2(h[n0][1].x, h[n0][1].y);
        af[kt + 1][2] = pack_bf16x2(h[n0 + 1][0].x, h[n0 + 1][0].y);
        af[kt + 1][3] = pack_bf16x2(h[n0 + 1][1].x, h[n0 + 1][1].y);
      }
      if (kt == 0) red_stage(pin, 1);
      if (kt == (VT > 1 ? 1 : 0)) {
        red_stage(pin, 2);
        red_store(pin, pin_row);
      }
    }

    // Readout of H_t (Eq. (12)): q-weighted sums of this thread's two rows.
    const uint16_t* qs = reinterpret_cast<const uint16_t*>(sbase + L.qs) + s * K;
    float qv0, qv1;
    if constexpr (kRing) {
      qv0 = bf16_bits_to_float(qs[r0]);
      qv1 = bf16_bits_to_float(qs[r1]);
    } else {
      qv0 = bf16_bits_to_float(cin.q0);
      qv1 = bf16_bits_to_float(cin.q1);
    }
    const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
    float p[M];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 pp = fma2(q1, h[nt][1], mul2(q0, h[nt][0]));
      p[2 * nt] = pp.x;
      p[2 * nt + 1] = pp.y;
    }
    // This step's partial sums are reduced during the next step (or at chunk end).
#pragma unroll
    for (int i = 0; i < M; ++i) pout[i] = p[i];
    if constexpr (kRing) {
      // Keep H_t for the backward pass as the bf16 A fragments just packed from it
      // (exactly the tensor-core operand step t+1 uses): stmatrix into this warp's half of
      // a two-step slot of a 2-slot swizzled ring; after the second step of the trip, one
      // fence and one TMA store of the warp's 16 rows for both steps (the odd last step of a
      // sequence is stored alone, after the loop's tail step).  A slot is rewritten only
      // after the store issued from it two trips earlier has read it.  No branch on the
      // lane: the wait and the commit run on every lane (lanes 1-31 only ever hold empty
      // groups) and the store is predicated on lane 0, so the step body stays one basic
      // block (with `if (lane == 0)` blocks the step took 930 instead of 790 cycles).
      const int t = cc * Tc + s;
      const uint32_t rbase = (smem_u32(smem) + L.hring + 1023u) & ~1023u;
      const uint32_t pslot = rbase + (uint32_t)((warp * 2 + ((t >> 1) & 1)) * 2 * 16 * V * 2);
      const uint32_t sb = pslot + (odd ? 16u * V * 2u : 0u);
      if (!odd) {
        bulk_wait_group_read<1>();  // every lane: only lane 0 holds groups
        __syncwarp();
      }
      const int lr = lane & 7, lq = lane >> 3;
#pragma unroll
      for (int kt = 0; kt < VT; ++kt)
        stsm_x4(sw128_addr(sb, lr + 8 * (lq & 1), 2 * kt + (lq >> 1)), af[kt]);
      if (odd) {
        fence_proxy_async_smem();
        __syncwarp();
        tma_store_4d_if(lane == 0, &tm_hs, pslot, 0, 16 * warp, t - 1, pair);
        bulk_commit_group();
      }
    } else if constexpr (kCache) {
      // Keep H_t for the backward pass as the bf16 A fragments just packed from it:
      // exactly the tensor-core operand step t+1 uses (streaming stores).
      uint16_t* hp = Hs + ((size_t)pair * T + (size_t)cc * Tc + s) * K * V;
#pragma unroll
      for (int kt = 0; kt < VT; ++kt) {
        __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r0 * V + 16 * kt + 2 * c), af[kt][0]);
        __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r1 * V + 16 * kt + 2 * c), af[kt][1]);
        __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r0 * V + 16 * kt + 8 + 2 * c), af[kt][2]);
        __stcs(reinterpret_cast<unsigned int*>(hp + (size_t)r1 * V + 16 * kt + 8 + 2 * c), af[kt][3]);
      }
    }
  };

  float pA[M], pB[M];
#pragma unroll
  for (int i = 0; i < M; ++i) pA[i] = pB[i] = 0.f;
  StepIn in;  // inputs of step 0: fetched as "the step after step -1"
  if constexpr (!kRing) fetch(in, 0, -1, nchunks > 1 ? Tc : T);
  for (int cc = 0; cc < nchunks; ++cc) {
    const int steps = min(Tc, T - cc * Tc);
    // The chunk's last step reads k_{t+1}, v_{t+1} from the next chunk: wait for it
    // before the two-step trip (or the odd tail) that contains that step.
    auto wait_next = [&]() {
      if (cc + 1 < nchunks &&
          !(kRing ? wait_or_abort(&full[(cc + 1) & 1], (uint32_t)((cc + 1) >> 1) & 1u, limit,
                                  abort_flag)
                  : wait_or_abort_sleep(&full[(cc + 1) & 1], (uint32_t)((cc + 1) >> 1) & 1u,
                                        limit, abort_flag)))
        aborted = true;
    };
    int s = 0;
    bool tail = false;
    for (; s + 1 < steps; s += 2) {  // two steps per trip: the accumulator sets swap roles
      if (s + 2 >= steps) wait_next();
      if (aborted) break;
      step(acc, nxt, cc, s, steps, pA, pB, in, false);
      step(nxt, acc, cc, s + 1, steps, pB, pA, in, true);
    }
    if (s < steps && !aborted) {  // odd tail of the last chunk
      wait_next();
      step(acc, nxt, cc, s, steps, pA, pB, in, false);
      tail = true;
      if constexpr (kRing) {  // the last state alone: a one-step store of the pair slot's first half
        const int t = cc * Tc + s;
        const uint32_t rbase = (smem_u32(smem) + L.hring + 1023u) & ~1023u;
        const uint32_t pslot = rbase + (uint32_t)((warp * 2 + ((t >> 1) & 1)) * 2 * 16 * V * 2);
        fence_proxy_async_smem();
        __syncwarp();
        tma_store_4d_if(lane == 0, &tm_hs1, pslot, 0, 16 * warp, t, pair);
        bulk_commit_group();
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] = nxt[nt][0];
        acc[nt][1] = nxt[nt][1];
      }
    }
    if (aborted) {
      *abort_flag = 1;
      if (lane == 0) atomicExch(status, kStatusTimeout);
      if constexpr (kRing) {
        if (lane == 0) bulk_wait_group<0>();  // stores still reading the ring
      }
      return;
    }
    {  // flush the chunk's last pending readout
      float* row = yrow_of(cc, steps - 1);
      if (tail) {
        red_stage(pB, 0); red_stage(pB, 1); red_stage(pB, 2); red_store(pB, row);
      } else {
        red_stage(pA, 0); red_stage(pA, 1); red_stage(pA, 2); red_store(pA, row);
      }
    }
    mbar_arrive(&done[cc & 1]);
  }

  if (H_T) {
    float* hp = H_T + (size_t)pair * K * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(hp + (size_t)r0 * V + 8 * nt + 2 * c) = h[nt][0];
      *reinterpret_cast<float2*>(hp + (size_t)r1 * V + 8 * nt + 2 * c) = h[nt][1];
    }
  }
  if constexpr (kRing) {
    if (lane == 0) bulk_wait_group<0>();  // every state store complete before the block ends
  }
}

bool make_map_pipe(EncodeTiledFn enc, CUtensorMap* map, const void* base, int inner, int N, int T,
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

template <int VT>
cudaError_t launch_pipe_vt(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  const int V = 16 * VT;
  const bool ring = p.Hs && VT == 4;
  int Tc = 64;
  PipeLayout L = pipe_layout(p.K, V, Tc, ring);
  while (L.total > 227 * 1024 && Tc > 8) {
    Tc /= 2;
    L = pipe_layout(p.K, V, Tc, ring);
  }
  CUtensorMap mq, mk, mv, mh, mh1;
  if (!make_map_pipe(enc, &mq, p.q, p.K, p.Nqk, p.T, p.B, Tc) ||
      !make_map_pipe(enc, &mk, p.k, p.K, p.Nqk, p.T, p.B, Tc) ||
      !make_map_pipe(enc, &mv, p.v, V, p.N, p.T, p.B, Tc))
    return cudaErrorInvalidValue;
  memset(&mh, 0, sizeof(mh));
  memset(&mh1, 0, sizeof(mh1));
  if (ring) {  // kept states [B N, T, K, V] bf16, stored 16 rows at a time, 128-byte swizzle
    const cuuint64_t dims[4] = {(cuuint64_t)V, (cuuint64_t)p.K, (cuuint64_t)p.T,
                                (cuuint64_t)p.B * p.N};
    const cuuint64_t strides[3] = {(cuuint64_t)V * 2, (cuuint64_t)V * 2 * p.K,
                                   (cuuint64_t)V * 2 * p.K * p.T};
    // two steps per store (box of 2 time steps), and one for an odd last step
    const cuuint32_t box[4] = {(cuuint32_t)V, 16u, 2u, 1u};
    const cuuint32_t box1[4] = {(cuuint32_t)V, 16u, 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    if (enc(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.Hs, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&mh1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.Hs, dims, strides, box1, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = p.Hs ? fwd_bf16_mma_pipe<VT, true> : fwd_bf16_mma_pipe<VT, false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)p.B * (unsigned)p.N;
  const int threads = 32 * (p.K / 16 + 1);
  kern<<<grid, threads, L.total, stream>>>(mq, mk, mv, mh, mh1, (const uint16_t*)p.a, p.alpha, p.beta,
                                           (const uint16_t*)p.W, p.w_r, p.H0, p.y, p.H_T,
                                           static_cast<uint16_t*>(p.Hs), p.T,
                                           p.N, p.K, Tc, p.Nqk == 1 ? 0 : 1, p.debug, p.status);
  return cudaGetLastError();
}

}  // namespace

bool mma_pipe_supports(int K, int V) {
  // At most 4 compute warps + the producer (160 threads) keep the whole working
  // set (H, two accumulator sets, A and W fragments) in registers without spills.
  return K >= 16 && K <= 64 && K % 16 == 0 && (V == 16 || V == 32 || V == 64);
}

cudaError_t launch_fwd_bf16_mma_pipe(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  switch (p.V) {
    case 16: return launch_pipe_vt<1>(p, enc, stream);
    case 32: return launch_pipe_vt<2>(p, enc, stream);
    case 64: return launch_pipe_vt<4>(p, enc, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace m2rnn
