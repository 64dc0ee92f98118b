// m2rnn_bwd_bf16_tcc.cu — backward pass of the M²RNN recurrence, K = V = 64, with every
// product of a step on the 5th-generation tensor cores, the serial chain included.
//
// Reverse scan of the M²RNN study notes, Sec. 2.7 (gate of Eq. (13)/(17)), on the kept bf16
// states.  Per step t, from C_t = dL/dH_t (C_{T-1} = dH_T):
//   P_t = H_{t-1} W + k_t v_t^T (recomputed),  Z_t = tanh(P_t),
//   R_t = C_t + q_t u_t^T,  D_t = ((1 - f_t) R_t) ⊙ (1 - Z_t^2),
//   C_{t-1} = f_t R_t + D_t W^T,  dW += H_{t-1}^T D_t,
//   dk_t = D_t v_t,  dv_t = D_t^T k_t + w_r ⊙ u_t,  dq_t = H_t u_t,  dL/df_t = <R_t, H_{t-1} - Z_t>.
// The issuer warp puts three tcgen05.mma products per step on the tensor core (M = 64,
// four K = 16 steps, fp32 accumulators in tensor memory).  The whole warp runs the issuing
// loop, so the descriptors stay warp-uniform, and one elected lane issues each MMA and
// commit (an issuer in a one-lane branch issued ~1.6x slower):
//   * G_t = D_t W^T, the chain product, as soon as every compute warp has written its part
//     of D_t^T (A = the D_t^T tile read M-major, B = the W^T tile read N-major);
//   * dW += H_{t-1}^T D_t into one accumulator over the whole sequence (same D_t^T tile);
//   * P_t = H_{t-1} [W | u], up to two steps ahead of the scan (kept state tile; B = the W^T
//     tile followed by 16 rows that hold u_{t-1} split into bf16 high and low parts, written
//     by the issuer just before the product).  Columns 64 .. 79 of the result give
//     dq_{t-1} = H_{t-1} u_{t-1} with fp32 accuracy in u; dq_{T-1} comes from one extra
//     N = 16 product on H_{T-1} at the start.
// Eight compute warps each own a 16-row block (the tensor-memory lane quarter of their
// sub-partition) and a 32-column half.  The halves never exchange data: the chain product
// reads all of D_t from shared memory.  Within a step a warp first loads the step's shared
// operands (no wait for the tensor core), then does the work that only needs P_t (rank-1
// term, tanh, 1 - Z^2, H_{t-1} - Z; dq_{t-1} read from the same slot), then waits for
// G_{t+1}, forms R_t, D_t and f_t R_t, writes D_t^T and signals, and reduces dk, dv and
// dL/df while the tensor core computes the next chain product.  Arrives and duplicated
// stores are predicated or done by every lane rather than branched, so the step's code
// stays in few basic blocks.  Waits that a commit already implies are skipped: a commit
// completes only when every earlier product of the issuing thread has.
//
// Roles: warps 0-7 compute, warp 8 producer (TMA, gates, per-chunk dv, dk, dq, da, dL/df
// sums, dalpha, dbeta, dw_r), warp 9 tensor-core issuer.  mbarriers: full (TMA), done
// (compute warps finished a chunk), mmadone (the chunk's products finished), pready /
// pfree (P slots), dtready / dtfree (D^T slots), gready (G slots), qdone (the dq_{T-1}
// product).  Every wait is bounded.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kK = 64, kV = 64;
constexpr int kNW = 4;                   // 16-row blocks
constexpr int kCW = 8;                   // compute warps: row block w % 4, column half w / 4
constexpr int kProducer = kCW, kIssuer = kCW + 1;
constexpr int kThreads = 32 * (kCW + 2);
constexpr int kTc = 8;                   // steps per chunk (= the 8 u rows: t0 % 8 == 0)
static_assert(kTc == 8, "the u rows of the P product are indexed by t % 8");
constexpr int kStages = 2;               // chunk stages in flight (TMA ring)
constexpr int kS = 3;                    // P slots in tensor memory (issue up to kS - 1 ahead)
constexpr int kTile = kK * kV * 2;       // one bf16 64 x 64 tile (64 rows of 128 bytes)
constexpr int kStageTiles = kTc + 1;     // states t0 - 1 .. t0 + Tc - 1
constexpr int kPN = kV + 16;             // P product width: W's 64 columns + 16 columns of u
constexpr uint32_t kPCols = 96;          // tensor-memory columns per P slot
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDwCol = kS * kPCols; // P slots: columns 0 .. 287; dW: 288 .. 351
constexpr uint32_t kGCol = kDwCol + 64;  // G slots: 352 .. 479

struct Layout {
  int hs, h0t, wt, dt, in, in_stage, qs, ks, vs, dys, gates, dfp, dvp, dkp, dqp, bar, total;
};

__host__ __device__ inline Layout layout_tcc() {
  Layout L;
  int o = 0;
  L.hs = o;                        // kept states, [kStages][kStageTiles] swizzled tiles
  o += kStages * kStageTiles * kTile;
  L.h0t = o;                       // bf16(H_0): the state before step 0
  o += kTile;
  L.wt = o;                        // W^T: row j holds W[0..63][j]; rows 64 .. 79 follow it:
  o += kTile + 2 * 1024;           // u_tau split as bf16 hi (row 64 + tau % 8) + lo (row 72 + ...)
  L.dt = o;                        // D_t^T, two slots: row j holds D_t[0..63][j]
  o += 2 * kTile;
  L.qs = 0;                        // per-stage inputs: q, k, v (bf16), dy (fp32)
  L.ks = kTc * kK * 2;
  L.vs = L.ks + kTc * kK * 2;
  L.dys = L.vs + kTc * kV * 2;
  L.in_stage = (L.dys + kTc * kV * 4 + 127) & ~127;
  L.in = o;
  o += kStages * L.in_stage;
  L.gates = o;                     // float4 [kStages][kTc]: f, 1 - f, sigmoid(a + beta), softplus
  o += kStages * kTc * 16;
  L.dfp = o;                       // float [kStages][kCW][kTc][8]: dL/df partials (per lane & 7)
  o += kStages * kCW * kTc * 8 * 4;
  L.dvp = o;                       // float [kStages][kNW][kTc][kV]: dv partials per row block
  o += kStages * kNW * kTc * kV * 4;
  L.dkp = o;                       // float [kStages][2 halves][kTc][kK]: dk partials
  o += kStages * 2 * kTc * kK * 4;
  L.dqp = o;                       // float [kStages][kTc][kK]: dq_t
  o += kStages * kTc * kK * 4;
  L.bar = o;
  o += 256;
  L.total = o + 1024;              // slack for aligning the base to 1024 bytes
  return L;
}

struct Bars {
  uint64_t* full;     // [kStages]
  uint64_t* done;     // [kStages]
  uint64_t* mmadone;  // [kStages]
  uint64_t* pready;   // [kS]
  uint64_t* pfree;    // [kS]
  uint64_t* dtready;  // [2]
  uint64_t* dtfree;   // [2]
  uint64_t* gready;   // [2]
  uint64_t* qdone;    // the dq_{T-1} product
  uint64_t* never;
  volatile int* abort_flag;
  uint32_t* tmem_slot;
};

__device__ inline Bars bars_at(uint8_t* p) {
  Bars B;
  uint64_t* b = reinterpret_cast<uint64_t*>(p);
  B.full = b;
  B.done = b + kStages;
  B.mmadone = b + 2 * kStages;
  B.pready = b + 3 * kStages;
  B.pfree = B.pready + kS;
  B.dtready = B.pfree + kS;
  B.dtfree = B.dtready + 2;
  B.gready = B.dtfree + 2;
  B.qdone = B.gready + 2;
  B.never = B.qdone + 1;
  B.abort_flag = reinterpret_cast<volatile int*>(B.never + 1);
  B.tmem_slot = reinterpret_cast<uint32_t*>(B.never + 2);
  return B;
}

__host__ __device__ constexpr int stage_of(int p) { return p % kStages; }
__host__ __device__ constexpr uint32_t phase_of(int p) { return (uint32_t)(p / kStages) & 1u; }

// Processing order: chunks from last to first, steps within a chunk from last to first.
struct Cursor {
  int p, s, steps, u;  // processed-chunk index, step in chunk, steps of the chunk, step count
};
__device__ inline int chunk_steps(int p, int nchunks, int T) {
  return min(kTc, T - (nchunks - 1 - p) * kTc);
}
__device__ inline void cursor_next(Cursor& c, int nchunks, int T) {
  ++c.u;
  if (c.s > 0) {
    --c.s;
  } else {
    ++c.p;
    if (c.p < nchunks) {
      c.steps = chunk_steps(c.p, nchunks, T);
      c.s = c.steps - 1;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_tcc(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_dy, const uint16_t* __restrict__ a,
                 const float* __restrict__ alpha, const float* __restrict__ beta,
                 const uint16_t* __restrict__ W, const float* __restrict__ w_r,
                 const float* __restrict__ H0, const float* __restrict__ dH_T,
                 float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                 float* __restrict__ da, float* __restrict__ dH0, float* __restrict__ ws,
                 float* __restrict__ dqk_heads, int T, int N, int Nqk, int debug, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Layout L = layout_tcc();
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.x, b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + kTc - 1) / kTc;
  const int nq = Nqk == 1 ? 0 : n;
  const bool shared_qk = Nqk == 1 && N > 1;
  const Bars Bs = bars_at(smem + L.bar);
  float4* gates = reinterpret_cast<float4*>(smem + L.gates);
  float* dfp = reinterpret_cast<float*>(smem + L.dfp);
  float* dvp = reinterpret_cast<float*>(smem + L.dvp);
  float* dkp = reinterpret_cast<float*>(smem + L.dkp);
  float* dqp = reinterpret_cast<float*>(smem + L.dqp);
  float* wsp = ws + (size_t)pair * backward_pair_floats(kK, kV);
  float* dWp = wsp + kK * kV;
  float* dwr_p = dWp + kV * kV;
  float* ab_p = dwr_p + kV;
  const long long limit = kWaitLimitCycles;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&Bs.full[i], 32);
      mbar_init(&Bs.done[i], 32 * kCW);
      mbar_init(&Bs.mmadone[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&Bs.dtready[i], kCW);
      mbar_init(&Bs.dtfree[i], 1);
      mbar_init(&Bs.gready[i], 1);
    }
    for (int i = 0; i < kS; ++i) {
      mbar_init(&Bs.pready[i], 1);
      mbar_init(&Bs.pfree[i], kCW);
    }
    mbar_init(Bs.qdone, 1);
    mbar_init(Bs.never, 1);
    *Bs.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(Bs.tmem_slot, kTmemCols);
  // W^T and bf16(H_0) into swizzled tiles.
  const uint16_t* Wn = W + (size_t)n * kV * kV;
  const float* h0p = H0 ? H0 + (size_t)pair * kK * kV : nullptr;
  for (int e = tid; e < kV * 8; e += kThreads) {
    const int row = e >> 3, ch = e & 7;
    uint32_t wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      wv[i] = (uint32_t)Wn[(8 * ch + 2 * i) * kV + row] |
              ((uint32_t)Wn[(8 * ch + 2 * i + 1) * kV + row] << 16);
    *reinterpret_cast<uint4*>(smem + (sw128_addr(sbase + L.wt, row, ch) - sbase)) =
        make_uint4(wv[0], wv[1], wv[2], wv[3]);
    uint4 hv = make_uint4(0u, 0u, 0u, 0u);
    if (h0p) {
      const float4 x0 = *reinterpret_cast<const float4*>(h0p + row * kV + 8 * ch);
      const float4 x1 = *reinterpret_cast<const float4*>(h0p + row * kV + 8 * ch + 4);
      hv = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                      pack_bf16x2(x1.z, x1.w));
    }
    *reinterpret_cast<uint4*>(smem + (sw128_addr(sbase + L.h0t, row, ch) - sbase)) = hv;
  }
  for (int e = tid; e < 16 * 8; e += kThreads)  // u rows: zero until first written
    *reinterpret_cast<uint4*>(smem + L.wt + kTile + 16 * e) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // the tiles are read by the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *Bs.tmem_slot;

  // State tile of state t - 1 for step s of processed chunk p (stage st), or the H_0 tile.
  auto hprev_tile = [&](int st, int s, int p) -> uint32_t {
    const int t = (nchunks - 1 - p) * kTc + s;
    return t == 0 ? sbase + L.h0t : sbase + L.hs + (st * kStageTiles + s) * kTile;
  };

  if (warp == kProducer) {
    // ======================================================= producer warp
    const float al = alpha[n], be = beta[n];
    const uint32_t tx =
        (uint32_t)(kStageTiles * kTile + 2 * kTc * kK * 2 + kTc * kV * 2 + kTc * kV * 4);
    const float2 wr = *reinterpret_cast<const float2*>(w_r + (size_t)n * kV + 2 * lane);
    auto arm = [&](int p) {
      const int st = stage_of(p), t0 = (nchunks - 1 - p) * kTc;
      if (lane < kTc) {
        const int t = t0 + lane;
        const float x = (t < T ? bf16_bits_to_float(a[((size_t)b * T + t) * N + n]) : 0.f) + be;
        const float ex = expf(-fabsf(x));
        const float sp = fmaxf(x, 0.f) + log1pf(ex);
        const float sg = x >= 0.f ? 1.f / (1.f + ex) : ex / (1.f + ex);
        gates[st * kTc + lane] = make_float4(expf(-al * sp), -expm1f(-al * sp), sg, sp);
      }
      __syncwarp();
      if (lane != 0) {
        mbar_arrive(&Bs.full[st]);
      } else {
        uint8_t* in = smem + L.in + st * L.in_stage;
        mbar_arrive_expect_tx(&Bs.full[st], tx);
        // states t0 - 1 .. t0 + Tc - 1 (t0 - 1 = -1 is zero-filled and not used)
        tma_load_4d(smem + L.hs + st * kStageTiles * kTile, &tm_h, &Bs.full[st], 0, 0, t0 - 1,
                    pair);
        tma_load_4d(in + L.qs, &tm_q, &Bs.full[st], 0, nq, t0, b);
        tma_load_4d(in + L.ks, &tm_k, &Bs.full[st], 0, nq, t0, b);
        tma_load_4d(in + L.vs, &tm_v, &Bs.full[st], 0, n, t0, b);
        tma_load_4d(in + L.dys, &tm_dy, &Bs.full[st], 0, n, t0, b);
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
    for (; issued < kStages && issued < nchunks; ++issued) arm(issued);
    float2 dwr = make_float2(0.f, 0.f);
    float dal = 0.f, dbe = 0.f;
    bool ok = true;
    for (int p = 0; p < nchunks; ++p) {
      const int st = stage_of(p), t0 = (nchunks - 1 - p) * kTc;
      const int steps = min(kTc, T - t0);
      const uint32_t par = phase_of(p);
      ok = wait_or_abort(&Bs.done[st], par, limit, Bs.abort_flag);
      ok = ok && wait_or_abort(&Bs.mmadone[st], par, limit, Bs.abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint8_t* in = smem + L.in + st * L.in_stage;
      const float* dys = reinterpret_cast<const float*>(in + L.dys);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(in + L.vs);
      for (int s = 0; s < steps; ++s) {
        // dv_t = w_r ⊙ u_t + the row blocks' D_t^T k_t partials; lane: columns 2 lane, +1
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
        // dk_t (the two column halves' partial sums) and dq_t; lane: rows 2 lane, +1
        const size_t qrow =
            ((size_t)b * T + t0 + s) * (shared_qk ? N : Nqk) + (shared_qk ? n : nq);
        float* dqo = shared_qk ? dqk_heads : dq;
        float* dko = shared_qk ? dqk_heads + (size_t)gridDim.x * T * kK : dk;
        const float* pk0 = dkp + ((st * 2 + 0) * kTc + s) * kK;
        const float* pk1 = dkp + ((st * 2 + 1) * kTc + s) * kK;
        const float2 k0v = *reinterpret_cast<const float2*>(pk0 + 2 * lane);
        const float2 k1v = *reinterpret_cast<const float2*>(pk1 + 2 * lane);
        *reinterpret_cast<float2*>(dko + qrow * kK + 2 * lane) =
            make_float2(k0v.x + k1v.x, k0v.y + k1v.y);
        *reinterpret_cast<float2*>(dqo + qrow * kK + 2 * lane) =
            *reinterpret_cast<const float2*>(dqp + (st * kTc + s) * kK + 2 * lane);
      }
      // dL/df_t: the 8 warps' 8 partials of each step, summed by the whole warp; lane s keeps
      // step s's total.
      float df = 0.f;
      for (int s = 0; s < steps; ++s) {
        const int w = lane >> 2, j = 2 * (lane & 3);
        const float2 pp = *reinterpret_cast<const float2*>(dfp + ((st * kCW + w) * kTc + s) * 8 + j);
        float sum = pp.x + pp.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == s) df = sum;
      }
      if (lane < steps) {  // da_t, and the sums for dalpha, dbeta
        const float4 gt = gates[st * kTc + lane];
        const float d_a = df * (-al * gt.x * gt.z);
        da[((size_t)b * T + t0 + lane) * N + n] = d_a;
        dal = fmaf(df, -gt.x * gt.w, dal);
        dbe += d_a;
      }
      __syncwarp();
      if (issued < nchunks) arm(issued++);
    }
    if (!ok) {
      if (lane == 0) {
        *Bs.abort_flag = 1;
        atomicExch(status, kStatusTimeout);
        for (int i = 0; i < kStages; ++i)  // let copies in flight land
          for (int ph = 0; ph < 2; ++ph)
            mbar_wait_bounded(&Bs.full[i], (uint32_t)ph, kDebugWaitLimitCycles);
      }
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        dal += __shfl_xor_sync(0xffffffffu, dal, o);
        dbe += __shfl_xor_sync(0xffffffffu, dbe, o);
      }
      *reinterpret_cast<float2*>(dwr_p + 2 * lane) = dwr;
      if (lane == 0) {
        ab_p[0] = dal;
        ab_p[1] = dbe;
      }
    }
  } else if (warp == kIssuer) {
    // ======================================================= tensor-core issuer
    // The whole warp runs the loop (the descriptors stay warp-uniform); one elected lane
    // issues each MMA and commit.  Wait outcomes are made warp-uniform with __all_sync.
    const bool leader = elect_one_sync();
    const uint32_t idesc_p = umma_idesc_bf16(kK, kPN, false);         // A = H, B = [W^T; u rows]
    const uint32_t idesc_q = umma_idesc_bf16(kK, 16, false);          // A = H, B = the u rows
    const uint32_t idesc_w = umma_idesc_bf16(kV, kV, true);           // A = H^T (M-major view)
    const uint32_t idesc_g = umma_idesc_bf16_ab(kK, kV, true, true);  // A = D, B = W^T N-major
    // Descriptors of a tile at byte offset `off` from sbase: the base's address field plus
    // off / 16 (shared-memory offsets stay below 256 KB, so the field does not overflow).
    const uint64_t d_k0 = umma_desc(sbase, 16, 1024, 2);     // K-major 128-byte-swizzled
    const uint64_t d_m0 = umma_desc(sbase, kTile, 1024, 2);  // MN-major, one 64-wide atom
    const uint64_t d_wt = d_k0 + (uint64_t)(L.wt >> 4);      // W^T, K-major
    const uint64_t d_wn = d_m0 + (uint64_t)(L.wt >> 4);      // the same tile, N-major
    const uint64_t d_u = d_k0 + (uint64_t)((L.wt + kTile) >> 4);  // the u rows alone
    auto hprev_off = [&](int st, int s, int p) -> int {  // the state tile before step s
      const int t = (nchunks - 1 - p) * kTc + s;
      return t == 0 ? L.h0t : L.hs + (st * kStageTiles + s) * kTile;
    };
    // u_tau (fp32, step s_u of the dy block of stage st_u) into rows 64 + tau % 8 (bf16 of u)
    // and 72 + tau % 8 (bf16 of the remainder) of the B operand [W^T; u rows], so that the
    // product H_{t-1} [W | u] also yields H_{t-1} u_{t-1} = dq_{t-1} to fp32 accuracy in u.
    // Row r of the u groups: 128-byte-swizzled like the W^T rows above it (rows 64 + r and
    // 72 + r, r < 8, so the swizzle term is r); this lane's 4 bytes at column 2 lane.
    uint8_t* const urow0 = smem + L.wt + kTile + (lane & 3) * 4;
    const float* const dys0 = reinterpret_cast<const float*>(smem + L.in + L.dys) + 2 * lane;
    auto put_u = [&](int st_u, int s_u, int row) {
      const float2 x = *reinterpret_cast<const float2*>(dys0 + (st_u * L.in_stage) / 4 + s_u * kV);
      const uint32_t hi = pack_bf16x2(x.x, x.y);
      const float2 hf = bf16x2_to_float2(hi);
      const uint32_t lo = pack_bf16x2(x.x - hf.x, x.y - hf.y);
      uint8_t* const dst = urow0 + row * 128 + (((lane >> 2) ^ row) << 4);
      *reinterpret_cast<uint32_t*>(dst) = hi;
      *reinterpret_cast<uint32_t*>(dst + 8 * 128) = lo;
      fence_proxy_async_smem();
    };
    Cursor cp{0, chunk_steps(0, nchunks, T) - 1, chunk_steps(0, nchunks, T), 0};
    Cursor cw = cp;
    bool ok = true;
    int full_seen = -1;  // chunks whose TMA completion was waited for
    // dq_{T-1} = H_{T-1} u_{T-1}: no P product has H_{T-1} as its A operand.  Into the second
    // G slot, which is first written by the chain product of step 1.
    {
      const int steps0 = chunk_steps(0, nchunks, T);
      ok = __all_sync(0xffffffffu, wait_or_abort(&Bs.full[0], 0u, limit, Bs.abort_flag));
      if (ok) {
        full_seen = 0;
        put_u(0, steps0 - 1, (T - 1) & 7);
        __syncwarp();
        tc_fence_after();
        umma4_if<2, 2>(leader, tmem + kGCol + 64, d_k0 + (uint64_t)((L.hs + steps0 * kTile) >> 4),
                       d_u, idesc_q, 0u);
        umma_commit_if(leader, Bs.qdone);
      }
    }
    const bool q_issued = ok;
    int pslot = 0;        // cp.u % kS
    uint32_t pround = 0;  // cp.u / kS
    while (ok && cw.u < T) {
      // P_t = H_{t-1} W for the steps ahead, into slot u % kS.
      while (ok && cp.u < T && cp.u < cw.u + kS) {
        const int slot = pslot;
        // u_{t-1} sits in the next processed chunk when t is the first step of its chunk.
        const bool cross = cp.s == 0 && cp.p + 1 < nchunks;
        bool w = true;
        if (cp.p > full_seen)
          w = wait_or_abort(&Bs.full[stage_of(cp.p)], phase_of(cp.p), limit, Bs.abort_flag);
        if (cross && cp.p + 1 > full_seen)
          w = w && wait_or_abort(&Bs.full[stage_of(cp.p + 1)], phase_of(cp.p + 1), limit,
                                 Bs.abort_flag);
        // The slot, and (as its product completed before) the u rows the product of step
        // u - 8 read: both are free once the warps have read P of step u - kS.
        if (cp.u >= kS)
          w = w && wait_or_abort(&Bs.pfree[slot], (pround - 1u) & 1u, limit, Bs.abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        full_seen = cross ? cp.p + 1 : max(full_seen, cp.p);
        if (cp.s > 0 || cross)  // t > 0: u_{t-1} into row (t - 1) % 8
          put_u(cross ? stage_of(cp.p + 1) : stage_of(cp.p), cross ? kTc - 1 : cp.s - 1,
                (cp.s + 7) & 7);
        __syncwarp();
        tc_fence_after();
        umma4_if<2, 2>(leader, tmem + kPCols * (uint32_t)slot,
                       d_k0 + (uint64_t)(hprev_off(stage_of(cp.p), cp.s, cp.p) >> 4), d_wt,
                       idesc_p, 0u);
        umma_commit_if(leader, &Bs.pready[slot]);
        cursor_next(cp, nchunks, T);
        if (++pslot == kS) {
          pslot = 0;
          ++pround;
        }
      }
      if (!ok) break;
      // D_t^T of step cw.u written by every compute warp: the chain product first.
      ok = __all_sync(0xffffffffu, wait_or_abort(&Bs.dtready[cw.u & 1], (uint32_t)(cw.u >> 1) & 1u,
                                                 limit, Bs.abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint64_t dto = (uint64_t)((L.dt + (cw.u & 1) * kTile) >> 4);
      // D_t (M-major view of D_t^T) x W^T (N-major): the chain product
      umma4_if<128, 128>(leader, tmem + kGCol + (uint32_t)(64 * (cw.u & 1)), d_m0 + dto, d_wn,
                         idesc_g, 0u);
      umma_commit_if(leader, &Bs.gready[cw.u & 1]);
      // dW += H_{t-1}^T D_t  (A = H_{t-1} M-major view, B = D_t^T K-major).
      umma4_if<128, 2>(leader, tmem + kDwCol,
                       d_m0 + (uint64_t)(hprev_off(stage_of(cw.p), cw.s, cw.p) >> 4), d_k0 + dto,
                       idesc_w, cw.u > 0 ? 1u : 0u);
      umma_commit_if(leader, &Bs.dtfree[cw.u & 1]);
      umma_commit_if(leader && cw.s == 0, &Bs.mmadone[stage_of(cw.p)]);  // the stage may be reused
      cursor_next(cw, nchunks, T);
    }
    if (!ok && lane == 0) {
      *Bs.abort_flag = 1;
      atomicExch(status, kStatusTimeout);
    }
    // Before the tensor memory is released every issued MMA must have finished: a commit
    // completes when all earlier MMAs of the issuing thread have, so wait for the last
    // commit of each kind (bounded).
    if (q_issued) mbar_wait_bounded(Bs.qdone, 0u, limit);
    if (cp.u > 0)
      mbar_wait_bounded(&Bs.pready[(cp.u - 1) % kS], (uint32_t)((cp.u - 1) / kS) & 1u, limit);
    if (cw.u > 0)
      mbar_wait_bounded(&Bs.dtfree[(cw.u - 1) & 1], (uint32_t)((cw.u - 1) >> 1) & 1u, limit);
  } else {
    // ======================================================= compute warps
    const int rb = warp & 3, ch = warp >> 2;
    const int g = lane >> 2, c = lane & 3;
    const int r0 = 16 * rb + g, r1 = r0 + 8;
    const int c0 = 32 * ch;
    const int lr = lane & 7, lq = lane >> 3;
    const uint32_t t_lanes = tmem + ((uint32_t)(32 * rb) << 16);

    // C: rows r0 / r1, columns c0 + 8 nt + 2c, +1.  Holds C_t at the start of step t's
    // chain part and f_t R_t after it (C_{t-1} = f_t R_t + G_t).
    float2 C[4][2];
    const float* dhp = dH_T ? dH_T + (size_t)pair * kK * kV : nullptr;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      C[nt][0] = dhp ? *reinterpret_cast<const float2*>(dhp + r0 * kV + c0 + 8 * nt + 2 * c)
                     : make_float2(0.f, 0.f);
      C[nt][1] = dhp ? *reinterpret_cast<const float2*>(dhp + r1 * kV + c0 + 8 * nt + 2 * c)
                     : make_float2(0.f, 0.f);
    }
    bool ok = true;
    if (debug & kDebugForceTimeout) ok = mbar_wait_bounded(Bs.never, 0u, kDebugWaitLimitCycles);
    // dq_t of the coming step; lanes 0-15 hold rows 16 rb + lane.  First dq_{T-1}, whose
    // product was issued before P_{T-1} (so the pready commit of step 0 covers it).
    float dqc = 0.f;
    if (ok) {
      ok = wait_or_abort(&Bs.pready[0], 0u, limit, Bs.abort_flag);
      if (ok) {
        tc_fence_after();
        const uint32_t col = kGCol + 64 + (uint32_t)((T - 1) & 7);
        const uint32_t qh = tmem_ld_32x32b_x1(t_lanes + col);
        const uint32_t ql = tmem_ld_32x32b_x1(t_lanes + col + 8);
        tmem_wait_ld();
        dqc = __uint_as_float(qh) + __uint_as_float(ql);
      }
    }
    int u = 0;
    for (int p = 0; p < nchunks && ok; ++p) {
      const int st = stage_of(p), t0 = (nchunks - 1 - p) * kTc;
      const int steps = min(kTc, T - t0);
      ok = wait_or_abort(&Bs.full[st], phase_of(p), limit, Bs.abort_flag);
      const uint8_t* in = smem + L.in + st * L.in_stage;
      const uint16_t* qs = reinterpret_cast<const uint16_t*>(in + L.qs);
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(in + L.ks);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(in + L.vs);
      const float* dys = reinterpret_cast<const float*>(in + L.dys);
      for (int s = steps - 1; s >= 0 && ok; --s, ++u) {
        const uint32_t hprev = hprev_tile(st, s, p);
        const float4 gt = gates[st * kTc + s];
        // ff = f_t; ngg = -(1 - f_t), paired with Z^2 - 1 below (one fma, no negation)
        const float2 ff = make_float2(gt.x, gt.x), ngg = make_float2(-gt.y, -gt.y);

        // ---- shared-memory operands of the step (the stage is resident)
        const float kv0 = bf16_bits_to_float(ks[s * kK + r0]);
        const float kv1 = bf16_bits_to_float(ks[s * kK + r1]);
        const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
        const float qv0 = bf16_bits_to_float(qs[s * kK + r0]);
        const float qv1 = bf16_bits_to_float(qs[s * kK + r1]);
        const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
        float2 vv[4], uu[4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          vv[nt] = bf16x2_to_float2(
              *reinterpret_cast<const uint32_t*>(vs + s * kV + c0 + 8 * nt + 2 * c));
          uu[nt] = *reinterpret_cast<const float2*>(dys + s * kV + c0 + 8 * nt + 2 * c);
        }
        uint32_t ah[2][4];  // H_{t-1}, this half's two k-tiles
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2)
          ldsm_x4(ah[q2], sw128_addr(hprev, 16 * rb + lr + 8 * (lq & 1), 4 * ch + 2 * q2 + (lq >> 1)));
        // ---- P_t (this half's 32 columns) from tensor memory, + k_t v_t^T.  From step 2 on
        // P_t is complete already: it was issued before the chain product of step u - 2,
        // whose commit the previous step waited for.
        const int slot = u % kS;
        if (u < 2) {
          ok = wait_or_abort(&Bs.pready[slot], (uint32_t)(u / kS) & 1u, limit, Bs.abort_flag);
          if (!ok) break;
          tc_fence_after();
        }
        // dq_t: the two column halves store one half of the rows each.
        if ((lane >> 3) == ch) dqp[(st * kTc + s) * kK + 16 * rb + lane] = dqc;
        uint32_t pr[16];
        tmem_ld_16x256b_x4(t_lanes + kPCols * (uint32_t)slot + (uint32_t)c0, pr);
        // dq_{t-1} = H_{t-1} u_{t-1} from the u columns of the same product (hi + lo parts)
        const uint32_t qcol = kPCols * (uint32_t)slot + kV + (uint32_t)((s + 7) & 7);
        const uint32_t qh = tmem_ld_32x32b_x1(t_lanes + qcol);
        const uint32_t ql = tmem_ld_32x32b_x1(t_lanes + qcol + 8);
        tmem_wait_ld();
        dqc = __uint_as_float(qh) + __uint_as_float(ql);
        tc_fence_before();
        __syncwarp();
        mbar_arrive_if(lane == 0, &Bs.pfree[slot]);
        float2 zz1[4][2], hmz[4][2], R[4][2];
        const float2 mone = make_float2(-1.f, -1.f);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float2 pv = fma2(r ? k1 : k0, vv[nt],
                                   make_float2(__uint_as_float(pr[4 * nt + 2 * r]),
                                               __uint_as_float(pr[4 * nt + 2 * r + 1])));
            const float2 z = make_float2(tanh_mufu(pv.x), tanh_mufu(pv.y));
            const float2 h = bf16x2_to_float2(ah[nt >> 1][2 * (nt & 1) + r]);
            zz1[nt][r] = mul2(ngg, fma2(z, z, mone));  // (1 - f_t) (1 - Z^2)
            hmz[nt][r] = sub2(h, z);
            R[nt][r] = fma2(r ? q1 : q0, uu[nt], C[nt][r]);  // q_t u_t^T + f_{t+1} R_{t+1}
          }
        // ---- the chain: R_t = q_t u_t^T + C_t, with C_t = f_{t+1} R_{t+1} + G_{t+1} (the part
        // without G is formed above).  G_{t+1} was committed after the dW product of step u - 2
        // was issued, and a commit completes only when every earlier product has: so it also
        // guarantees that this step's D^T slot has been read.
        if (u >= 1) {
          ok = wait_or_abort(&Bs.gready[(u - 1) & 1], (uint32_t)((u - 1) >> 1) & 1u, limit,
                             Bs.abort_flag);
          if (!ok) break;
          tc_fence_after();
          uint32_t gr[16];
          tmem_ld_16x256b_x4(t_lanes + kGCol + (uint32_t)(64 * ((u - 1) & 1) + c0), gr);
          tmem_wait_ld();
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            R[nt][0] = add2(R[nt][0], make_float2(__uint_as_float(gr[4 * nt]),
                                                  __uint_as_float(gr[4 * nt + 1])));
            R[nt][1] = add2(R[nt][1], make_float2(__uint_as_float(gr[4 * nt + 2]),
                                                  __uint_as_float(gr[4 * nt + 3])));
          }
        }
        float2 Dm[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int r = 0; r < 2; ++r) Dm[nt][r] = mul2(R[nt][r], zz1[nt][r]);  // D_t
        // ---- D_t^T (this warp's 16 rows x 32 columns) to the shared tile, then signal
        uint32_t ad[2][4];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          ad[q2][0] = pack_bf16x2(Dm[2 * q2][0].x, Dm[2 * q2][0].y);
          ad[q2][1] = pack_bf16x2(Dm[2 * q2][1].x, Dm[2 * q2][1].y);
          ad[q2][2] = pack_bf16x2(Dm[2 * q2 + 1][0].x, Dm[2 * q2 + 1][0].y);
          ad[q2][3] = pack_bf16x2(Dm[2 * q2 + 1][1].x, Dm[2 * q2 + 1][1].y);
        }
        const uint32_t dts = sbase + L.dt + (u & 1) * kTile;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int kj = 2 * ch + q2;  // D^T rows j = 16 kj .., columns i = 16 rb ..
          stsm_x4_trans(sw128_addr(dts, 16 * kj + lr + 8 * (lq >> 1), 2 * rb + (lq & 1)), ad[q2]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_if(lane == 0, &Bs.dtready[u & 1]);

        // ---- off the chain: f_t R_t (the next C without G), dL/df_t, dk_t = D_t v_t, dv partial
        float2 dfl2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            dfl2 = fma2(R[nt][r], hmz[nt][r], dfl2);
            C[nt][r] = mul2(ff, R[nt][r]);
          }
        float2 sk0 = make_float2(0.f, 0.f), sk1 = make_float2(0.f, 0.f);
        float pdv[8];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          sk0 = fma2(Dm[nt][0], vv[nt], sk0);
          sk1 = fma2(Dm[nt][1], vv[nt], sk1);
          const float2 pv = fma2(k1, Dm[nt][1], mul2(k0, Dm[nt][0]));
          pdv[2 * nt] = pv.x;
          pdv[2 * nt + 1] = pv.y;
        }
#pragma unroll
        for (int stg = 0; stg < 3; ++stg) {  // reduce-scatter over the 8 row groups
          const int mask = 16 >> stg, half = 4 >> stg;
          const bool up = (lane & mask) != 0;
#pragma unroll
          for (int i = 0; i < half; ++i) {
            const float send = up ? pdv[i] : pdv[i + half];
            const float keep = up ? pdv[i + half] : pdv[i];
            pdv[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        }
        // Lane (g, c) holds column c0 + 8 (g >> 1) + 2c + (g & 1).
        dvp[((st * kNW + rb) * kTc + s) * kV + c0 + 8 * (g >> 1) + 2 * c + (g & 1)] = pdv[0];
        // dL/df_t partial: summed over lane bits 4 and 3 only; lanes that agree in bits 0-2
        // hold the same value and store it together (the producer adds the rest).
        float dfl = dfl2.x + dfl2.y;
        dfl += __shfl_xor_sync(0xffffffffu, dfl, 16);
        dfl += __shfl_xor_sync(0xffffffffu, dfl, 8);
        dfp[((st * kCW + warp) * kTc + s) * 8 + (lane & 7)] = dfl;
        // dk (rows r0, r1): summed over the lane quad, lanes c = 0, 2 end with row r0 and
        // c = 1, 3 with row r1 (both store: same value, same address).
        {
          const float k0s = sk0.x + sk0.y, k1s = sk1.x + sk1.y;
          const bool hi1 = (c & 1) != 0;
          float ks2 = hi1 ? k1s : k0s;
          ks2 += __shfl_xor_sync(0xffffffffu, hi1 ? k0s : k1s, 1);
          ks2 += __shfl_xor_sync(0xffffffffu, ks2, 2);
          dkp[((st * 2 + ch) * kTc + s) * kK + (hi1 ? r1 : r0)] = ks2;
        }
      }
      if (!ok) break;
      mbar_arrive(&Bs.done[st]);
    }
    if (ok) {  // the last products have finished: dW (this warp's 16 x 32 block) and dH_0
      ok = wait_or_abort(&Bs.dtfree[(T - 1) & 1], (uint32_t)((T - 1) >> 1) & 1u, limit,
                         Bs.abort_flag);
      if (ok) {
        tc_fence_after();
        uint32_t wr[16], gr[16];
        tmem_ld_16x256b_x4(t_lanes + kDwCol + (uint32_t)c0, wr);
        tmem_ld_16x256b_x4(t_lanes + kGCol + (uint32_t)(64 * ((T - 1) & 1) + c0), gr);
        tmem_wait_ld();
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          *reinterpret_cast<float2*>(dWp + r0 * kV + c0 + 8 * nt + 2 * c) =
              make_float2(__uint_as_float(wr[4 * nt]), __uint_as_float(wr[4 * nt + 1]));
          *reinterpret_cast<float2*>(dWp + r1 * kV + c0 + 8 * nt + 2 * c) =
              make_float2(__uint_as_float(wr[4 * nt + 2]), __uint_as_float(wr[4 * nt + 3]));
        }
        if (dH0) {  // dL/dH_0 = f_0 R_0 + D_0 W^T
          float* hp = dH0 + (size_t)pair * kK * kV;
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            *reinterpret_cast<float2*>(hp + r0 * kV + c0 + 8 * nt + 2 * c) =
                add2(C[nt][0], make_float2(__uint_as_float(gr[4 * nt]),
                                           __uint_as_float(gr[4 * nt + 1])));
            *reinterpret_cast<float2*>(hp + r1 * kV + c0 + 8 * nt + 2 * c) =
                add2(C[nt][1], make_float2(__uint_as_float(gr[4 * nt + 2]),
                                           __uint_as_float(gr[4 * nt + 3])));
          }
        }
      }
    }
    if (!ok) {
      *Bs.abort_flag = 1;
      if (lane == 0) atomicExch(status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

bool make_map_tcc(EncodeTiledFn enc, CUtensorMap* map, CUtensorMapDataType dt, const void* base,
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

cudaError_t launch_bwd_bf16_tcc(const BackwardProblem& p, EncodeTiledFn enc, int debug,
                                int* status, cudaStream_t stream) {
  const Layout L = layout_tcc();
  const cuuint64_t B = (cuuint64_t)p.B, T = (cuuint64_t)p.T, N = (cuuint64_t)p.N;
  CUtensorMap mh, mq, mk, mv, mdy;
  const cuuint64_t dh[4] = {kV, kK, T, B * N};
  const cuuint32_t bh[4] = {kV, kK, kStageTiles, 1};
  const cuuint64_t dqk[4] = {kK, (cuuint64_t)p.Nqk, T, B};
  const cuuint32_t bqk[4] = {kK, 1, kTc, 1};
  const cuuint64_t dvv[4] = {kV, N, T, B};
  const cuuint32_t bvv[4] = {kV, 1, kTc, 1};
  if (!make_map_tcc(enc, &mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.Hs, 2, dh, bh,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_tcc(enc, &mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 2, dqk, bqk,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_tcc(enc, &mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, 2, dqk, bqk,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_tcc(enc, &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, 2, dvv, bvv,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_tcc(enc, &mdy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dy, 4, dvv, bvv,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(bwd_bf16_tcc, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  float* heads = p.ws + (size_t)p.B * p.N * backward_pair_floats(kK, kV);
  bwd_bf16_tcc<<<(unsigned)(p.B * p.N), kThreads, L.total, stream>>>(
      mh, mq, mk, mv, mdy, (const uint16_t*)p.a, p.alpha, p.beta, (const uint16_t*)p.W, p.w_r,
      p.H0, p.dH_T, p.dq, p.dk, p.dv, p.da, p.dH0, p.ws, heads, p.T, p.N, p.Nqk, debug, status);
  err = cudaGetLastError();
  return err == cudaSuccess ? launch_bwd_reduce(p, stream) : err;
}

}  // namespace m2rnn
