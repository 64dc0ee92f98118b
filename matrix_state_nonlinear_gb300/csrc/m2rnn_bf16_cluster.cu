// m2rnn_bf16_cluster.cu — bf16-operand / fp32-state forward recurrence for K = 64,
// V = 128, one 4-CTA thread-block cluster per (batch, head) pair.
//
// The recurrence is Eq. (10)-(12) and (13)/(17) of the M²RNN study notes ("M²RNN:
// 矩阵状态非线性 RNN 的容量、表达力与系统代价", Sec. 2.1-2.2).  Rows of H evolve
// independently given W and the gate (Sec. 1.2: W mixes value columns, not key rows),
// so a pair can be spread over several SMs by rows; only the readout y_t = H_t^T q_t
// sums over rows and crosses SMs.  With few pairs (e.g. B = 1, N = 16) this puts a
// pair on 4 SMs instead of 1.
//
// Mapping.  CTA rank r of the cluster owns rows 16 r .. 16 r + 15.  Its 4 compute
// warps own the column quarters 32 c .. 32 c + 31 of those rows:
//   * H (fp32) and the B fragments of W for the warp's 32 output columns (all 8
//     k-tiles, 64 registers) stay in registers; the warp-level MMA m16n8k16 runs
//     P_{t+1} = k_{t+1} v_{t+1}^T + H_t W for its 4 n-tiles;
//   * each step every warp packs the bf16 A fragments of its two k-tiles of H_t
//     (its own columns) into a double-buffered shared-memory slot, issues its own
//     two k-tiles, meets the other three warps at a named barrier, then loads and
//     issues their six k-tiles;
//   * readout: each warp reduce-scatters its q-weighted sums over its 8 row groups
//     and stores the 32 column sums of its 16 rows straight into the shared memory of
//     CTA c (the owner of column quarter c) through distributed shared memory.
//     CTA c's producer warp adds the 4 row blocks' partials and w_r ⊙ v_t and
//     stores its 32-column slice of y.
// With kCache (the training forward) every warp also stores the bf16 H_t it packs each step
// into the kept-state history Hs, so the backward reads exactly the product's operand.
// Cross-CTA handoffs are mbarriers with remote release arrives and bounded acquire
// waits: `ready` (a chunk's partials for my quarter arrived from all ranks) and
// `free` (every owner has consumed the partials I sent, so the buffer can be reused).
// A final cluster barrier keeps each CTA alive until its peers stopped writing to it.
#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 128;
constexpr int kK = 64;
constexpr int kR = 4;               // CTAs per pair (row blocks of 16)
constexpr int kQ = kV / kR;         // columns per quarter (per compute warp / owner CTA)
constexpr int kCompute = 4;         // compute warps; warp kCompute is the producer
constexpr int kThreads = 32 * (kCompute + 1);
constexpr int kBarId = 1;           // named barrier of the 4 compute warps

struct ClusterLayout {
  int qs, ks, vs, stage_bytes;  // TMA destinations: q, k [Tc][16], v [Tc][128] bf16
  int fg;                       // float2 [2][Tc]            (f, 1 - f)
  int xbuf;                     // uint4  [2][4][2][32]      A-fragment exchange
  int ypart;                    // float  [2][kR][Tc][kQ]    partials received for my quarter
  int wr;                       // float  [kV]
  int bar;                      // full[2], done[2], ready[2], free[2], never; int abort
  int total;
};

__host__ __device__ inline int al128k(int x) { return (x + 127) & ~127; }

__host__ __device__ inline ClusterLayout cluster_layout(int Tc) {
  ClusterLayout L;
  L.qs = 0;
  L.ks = al128k(Tc * 16 * 2);
  L.vs = L.ks + al128k(Tc * 16 * 2);
  L.stage_bytes = L.vs + al128k(Tc * kV * 2);
  int o = 2 * L.stage_bytes;
  L.fg = o;
  o += al128k(2 * Tc * 8);
  L.xbuf = o;
  o += 2 * kCompute * 2 * 32 * 16;
  L.ypart = o;
  o += al128k(2 * kR * Tc * kQ * 4);
  L.wr = o;
  o += al128k(kV * 4);
  L.bar = o;
  o += 128;
  L.total = o;
  return L;
}

// kCache: also keep every state H_t in Hs [B N, T, K, V] as bf16, the A fragments each warp
// packs for the next step's product (streaming stores of its 16 rows x 32 columns).
template <bool kCache>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_mma_cluster(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const uint16_t* __restrict__ a, const float* __restrict__ alpha,
                         const float* __restrict__ beta, const uint16_t* __restrict__ W,
                         const float* __restrict__ w_r, const float* H0, float* __restrict__ y,
                         float* H_T, uint16_t* __restrict__ Hs, int T, int N, int Tc, int qk_hs,
                         int debug, int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const ClusterLayout L = cluster_layout(Tc);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rb = (int)cluster_ctarank();  // row block owned by this CTA
  const int pair = (int)cluster_id_x();
  const int b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + Tc - 1) / Tc;
  const size_t row_base = (size_t)b * T;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* done = full + 2;
  uint64_t* ready = full + 4;
  uint64_t* fre = full + 6;
  uint64_t* never = full + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 9);
  float2* fgs = reinterpret_cast<float2*>(smem + L.fg);
  uint4* xbuf = reinterpret_cast<uint4*>(smem + L.xbuf);
  float* ypart = reinterpret_cast<float*>(smem + L.ypart);
  float* wrs = reinterpret_cast<float*>(smem + L.wr);
  const long long limit = kWaitLimitCycles;

  if (tid == 0) {
    mbar_init(&full[0], 32);
    mbar_init(&full[1], 32);
    mbar_init(&done[0], 32 * kCompute);
    mbar_init(&done[1], 32 * kCompute);
    mbar_init(&ready[0], 32 * kR);  // lanes of warp rb of every rank
    mbar_init(&ready[1], 32 * kR);
    mbar_init(&fre[0], 32 * kR);    // producer lanes of every owner CTA
    mbar_init(&fre[1], 32 * kR);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int j = tid; j < kV; j += kThreads) wrs[j] = w_r[(size_t)n * kV + j];
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive

  if (warp == kCompute) {
    // ======================================================= producer warp
    const float al = alpha[n], be = beta[n];
    const uint32_t stage_tx = (uint32_t)Tc * (16u + 16u + (uint32_t)kV) * 2u;
    auto arm = [&](int cc) {  // gates of chunk cc, then its TMA loads
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
        tma_load_4d(base + L.qs, &tm_q, &full[st], 16 * rb, n * qk_hs, cc * Tc, b);
        tma_load_4d(base + L.ks, &tm_k, &full[st], 16 * rb, n * qk_hs, cc * Tc, b);
        tma_load_4d(base + L.vs, &tm_v, &full[st], 0, n, cc * Tc, b);
      }
    };
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    int issued = 0;
    for (; issued < 2 && issued < nchunks; ++issued) arm(issued);
    for (int cc = 0; cc < nchunks; ++cc) {
      const int st = cc & 1;
      const uint32_t par = (uint32_t)(cc >> 1) & 1u;
      bool ok = wait_or_abort(&done[st], par, limit, abort_flag);
      ok = ok && mbar_wait_cluster(&ready[st], par, limit, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {  // one decision for the whole warp
        if (lane == 0) {
          *abort_flag = 1;
          atomicExch(status, kStatusTimeout);
          for (int ci = cc; ci < issued; ++ci)  // let copies in flight land
            mbar_wait_bounded(&full[ci & 1], (uint32_t)(ci >> 1) & 1u, kDebugWaitLimitCycles);
        }
        break;
      }
      // y_t[32 rb + j] = sum over row blocks of the partials + w_r ⊙ v_t.
      const int t0 = cc * Tc;
      const int steps = min(Tc, T - t0);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + st * L.stage_bytes + L.vs);
      const float* yp = ypart + (size_t)st * kR * Tc * kQ;
      for (int idx = lane; idx < steps * (kQ / 4); idx += 32) {
        const int s = idx / (kQ / 4), j = (idx - s * (kQ / 4)) * 4;
        const int col = kQ * rb + j;
        const uint2 vv = *reinterpret_cast<const uint2*>(vs + s * kV + col);
        const float4 w4 = *reinterpret_cast<const float4*>(wrs + col);
        float4 o = make_float4(w4.x * bf16_lo(vv.x), w4.y * bf16_hi(vv.x), w4.z * bf16_lo(vv.y),
                               w4.w * bf16_hi(vv.y));
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const float4 u = *reinterpret_cast<const float4*>(yp + ((size_t)r * Tc + s) * kQ + j);
          o.x += u.x;
          o.y += u.y;
          o.z += u.z;
          o.w += u.w;
        }
        *reinterpret_cast<float4*>(y + ((row_base + t0 + s) * N + n) * kV + col) = o;
      }
      // The partials buffer of this chunk is consumed: tell every rank.
#pragma unroll
      for (int r = 0; r < kR; ++r) mbar_arrive_cluster(mapa_shared(smem_u32(&fre[st]), (uint32_t)r));
      if (issued < nchunks) arm(issued++);
    }
  } else {
    // ======================================================= compute warps
    const int cq = warp;  // column quarter
    const int g = lane >> 2, c = lane & 3;
    const int gr0 = kK / kR * rb + g, gr1 = gr0 + 8;  // global rows of H
    const int col0 = kQ * cq;

    // W fragments for this quarter's 4 n-tiles: own k-tiles (2 cq + u) and those of
    // the other three warps in the order (cq + 1 + i) & 3, so that indices are static.
    const uint16_t* Wn = W + (size_t)n * kV * kV;
    auto wfrag = [&](int kt, int j, uint32_t (&f)[2]) {
      const int col = col0 + 8 * j + g, r = 16 * kt + 2 * c;
      f[0] = (uint32_t)Wn[r * kV + col] | ((uint32_t)Wn[(r + 1) * kV + col] << 16);
      f[1] = (uint32_t)Wn[(r + 8) * kV + col] | ((uint32_t)Wn[(r + 9) * kV + col] << 16);
    };
    uint32_t wbo[2][4][2], wbx[3][2][4][2];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wfrag(2 * cq + u, j, wbo[u][j]);
#pragma unroll
        for (int i = 0; i < 3; ++i) wfrag(2 * ((cq + 1 + i) & 3) + u, j, wbx[i][u][j]);
      }

    // H_0, this warp's 16 rows x 32 columns, in fp32 (zero when absent).
    const float* hp0 = H0 ? H0 + (size_t)pair * kK * kV : nullptr;
    auto h0_pair = [&](int row, int col) -> float2 {
      return hp0 ? *reinterpret_cast<const float2*>(hp0 + (size_t)row * kV + col)
                 : make_float2(0.f, 0.f);
    };
    float2 h[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[j][0] = h0_pair(gr0, col0 + 8 * j + 2 * c);
      h[j][1] = h0_pair(gr1, col0 + 8 * j + 2 * c);
    }

    // H W for this quarter's columns: publish the bf16 A fragments of the warp's own
    // two k-tiles (columns 32 cq .. 32 cq + 31 of H), issue them, meet the other three
    // compute warps, then issue their six k-tiles.  `slot` alternates between calls;
    // prep(u) runs just before own k-tile u is packed (it brings h up to date).
    // `hs` (kCache): the kept state of this step, or null (the initial state is not kept).
    auto hw_accumulate = [&](float2 (&nx)[4][2], int slot, uint16_t* hs, auto&& prep) {
      uint4* xslot = xbuf + (size_t)slot * kCompute * 2 * 32;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        prep(u);
        uint32_t af[4];
        af[0] = pack_bf16x2(h[2 * u][0].x, h[2 * u][0].y);
        af[1] = pack_bf16x2(h[2 * u][1].x, h[2 * u][1].y);
        af[2] = pack_bf16x2(h[2 * u + 1][0].x, h[2 * u + 1][0].y);
        af[3] = pack_bf16x2(h[2 * u + 1][1].x, h[2 * u + 1][1].y);
        xslot[(cq * 2 + u) * 32 + lane] = make_uint4(af[0], af[1], af[2], af[3]);
        if (kCache && hs) {  // (row, column pair) of each fragment register
          const int cl = col0 + 16 * u + 2 * c;
          __stcs(reinterpret_cast<unsigned int*>(hs + (size_t)gr0 * kV + cl), af[0]);
          __stcs(reinterpret_cast<unsigned int*>(hs + (size_t)gr1 * kV + cl), af[1]);
          __stcs(reinterpret_cast<unsigned int*>(hs + (size_t)gr0 * kV + cl + 8), af[2]);
          __stcs(reinterpret_cast<unsigned int*>(hs + (size_t)gr1 * kV + cl + 8), af[3]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mma2(nx[j], af, wbo[u][j][0], wbo[u][j][1]);
      }
      named_bar_sync(kBarId, 32 * kCompute);
#pragma unroll
      for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4 v4 = xslot[(((cq + 1 + i) & 3) * 2 + u) * 32 + lane];
          const uint32_t af[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) mma2(nx[j], af, wbx[i][u][j][0], wbx[i][u][j][1]);
        }
    };
    // The rank-1 term k_t v_t^T of row block rb, this quarter: initialises P_t.
    auto rank1 = [&](float2 (&nx)[4][2], const uint8_t* base, int s) {
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(base + L.ks) + s * 16;
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(base + L.vs) + s * kV + col0;
      const float kv0 = bf16_bits_to_float(ks[g]), kv1 = bf16_bits_to_float(ks[g + 8]);
      const float2 k0 = make_float2(kv0, kv0), k1 = make_float2(kv1, kv1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 vv = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vs + 8 * j + 2 * c));
        nx[j][0] = mul2(k0, vv);
        nx[j][1] = mul2(k1, vv);
      }
    };

    bool ok = wait_or_abort(&full[0], 0u, limit, abort_flag);
    if (debug & kDebugForceTimeout) ok = ok && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
    bool aborted = named_bar_or(kBarId, 32 * kCompute, !ok);

    float2 acc[4][2], nxt[4][2];
    if (!aborted) {  // P_0 = k_0 v_0^T + H_0 W (exchange slot 1; step 0 uses slot 0)
      rank1(acc, smem, 0);
      hw_accumulate(acc, 1, nullptr, [](int) {});
    }

    // One time step t.  On entry `cur` = P_t (this quarter), h = H_{t-1}; on exit
    // h = H_t and `nx` = P_{t+1}.  `px` selects the exchange slot (alternates by step).
    auto step = [&](float2 (&cur)[4][2], float2 (&nx)[4][2], int cc, int s, int steps, int px) {
      const int st = cc & 1;
      const uint8_t* sbase = smem + st * L.stage_bytes;
      const bool last = s == steps - 1;
      const uint8_t* nbase = last ? smem + (st ^ 1) * L.stage_bytes : sbase;
      const int sn = last ? 0 : s + 1;
      const float2 fg = fgs[st * Tc + s];
      const float2 ff = make_float2(fg.x, fg.x), gg = make_float2(fg.y, fg.y);
      rank1(nx, nbase, sn);  // P_{t+1} starts as k_{t+1} v_{t+1}^T
      // Z_t = tanh(P_t), H_t = f H_{t-1} + (1 - f) Z_t (Eq. (10)-(11)), one own k-tile
      // (n-tiles 2u, 2u + 1) at a time, then P_{t+1} += H_t W.
      uint16_t* hs = kCache ? Hs + ((size_t)pair * T + (size_t)cc * Tc + s) * kK * kV : nullptr;
      hw_accumulate(nx, px, hs, [&](int u) {
#pragma unroll
        for (int j = 2 * u; j < 2 * u + 2; ++j)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float2 z = make_float2(tanh_mufu(cur[j][r].x), tanh_mufu(cur[j][r].y));
            h[j][r] = fma2(gg, z, mul2(ff, h[j][r]));
          }
      });
      // Readout (Eq. (12)): column sums of this warp's 16 rows, to the quarter's owner.
      const uint16_t* qs = reinterpret_cast<const uint16_t*>(sbase + L.qs) + s * 16;
      const float qv0 = bf16_bits_to_float(qs[g]), qv1 = bf16_bits_to_float(qs[g + 8]);
      const float2 q0 = make_float2(qv0, qv0), q1 = make_float2(qv1, qv1);
      float p[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 pp = fma2(q1, h[j][1], mul2(q0, h[j][0]));
        p[2 * j] = pp.x;
        p[2 * j + 1] = pp.y;
      }
#pragma unroll
      for (int stg = 0; stg < 3; ++stg) {  // reduce-scatter over the 8 row groups
        const int mask = 16 >> stg, half = 8 >> (stg + 1);
        const bool up = (lane & mask) != 0;
#pragma unroll
        for (int i2 = 0; i2 < half; ++i2) {
          const float send = up ? p[i2] : p[i2 + half];
          const float keep = up ? p[i2 + half] : p[i2];
          p[i2] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
      // Lane (g, c) holds slot m = g: column 8 (g >> 1) + 2c + (g & 1) of the quarter.
      const int colq = 8 * (g >> 1) + 2 * c + (g & 1);
      const uint32_t dst = smem_u32(ypart + (((size_t)st * kR + rb) * Tc + s) * kQ + colq);
      st_cluster_f32(mapa_shared(dst, (uint32_t)cq), p[0]);
    };

    int px = 0;
    for (int cc = 0; cc < nchunks && !aborted; ++cc) {
      const int st = cc & 1;
      const int steps = min(Tc, T - cc * Tc);
      if (cc >= 2) {  // every owner consumed the partials this CTA sent for chunk cc-2
        const bool w_ok =
            mbar_wait_cluster(&fre[st], (uint32_t)((cc >> 1) - 1) & 1u, limit, abort_flag);
        if (named_bar_or(kBarId, 32 * kCompute, !w_ok)) {
          aborted = true;
          break;
        }
      }
      auto wait_next = [&]() {  // inputs of the next chunk, jointly decided
        if (cc + 1 < nchunks) {
          const bool w_ok = wait_or_abort(&full[(cc + 1) & 1], (uint32_t)((cc + 1) >> 1) & 1u,
                                          limit, abort_flag);
          if (named_bar_or(kBarId, 32 * kCompute, !w_ok)) aborted = true;
        }
      };
      int s = 0;
      for (; s + 1 < steps; s += 2) {
        if (s + 2 >= steps) wait_next();
        if (aborted) break;
        step(acc, nxt, cc, s, steps, px);
        step(nxt, acc, cc, s + 1, steps, px ^ 1);
      }
      if (s < steps && !aborted) {  // odd tail of the last chunk
        wait_next();
        step(acc, nxt, cc, s, steps, px);
        px ^= 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[j][0] = nxt[j][0];
          acc[j][1] = nxt[j][1];
        }
      }
      if (aborted) break;
      // This chunk's partials are sent: signal the owner of my quarter, then release the stage.
      mbar_arrive_cluster(mapa_shared(smem_u32(&ready[st]), (uint32_t)cq));
      mbar_arrive(&done[st]);
    }
    if (aborted) {
      *abort_flag = 1;
      if (lane == 0) atomicExch(status, kStatusTimeout);
    } else if (H_T) {
      float* hp = H_T + (size_t)pair * kK * kV;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        *reinterpret_cast<float2*>(hp + (size_t)gr0 * kV + col0 + 8 * j + 2 * c) = h[j][0];
        *reinterpret_cast<float2*>(hp + (size_t)gr1 * kV + col0 + 8 * j + 2 * c) = h[j][1];
      }
    }
  }
  // No CTA leaves while a peer may still write into its shared memory.
  cluster_sync_all();
}

bool make_map_cluster(EncodeTiledFn enc, CUtensorMap* map, const void* base, int inner, int box,
                      int N, int T, int B, int Tc) {
  const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)N, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * N,
                                 (cuuint64_t)inner * 2 * N * T};
  const cuuint32_t boxd[4] = {(cuuint32_t)box, 1u, (cuuint32_t)Tc, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, boxd,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mma_cluster_supports(int K, int V) { return K == kK && V == kV; }

cudaError_t launch_fwd_bf16_mma_cluster(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  const int Tc = 64;
  const ClusterLayout L = cluster_layout(Tc);
  CUtensorMap mq, mk, mv;
  if (!make_map_cluster(enc, &mq, p.q, kK, 16, p.Nqk, p.T, p.B, Tc) ||
      !make_map_cluster(enc, &mk, p.k, kK, 16, p.Nqk, p.T, p.B, Tc) ||
      !make_map_cluster(enc, &mv, p.v, kV, kV, p.N, p.T, p.B, Tc))
    return cudaErrorInvalidValue;
  auto kern = p.Hs ? fwd_bf16_mma_cluster<true> : fwd_bf16_mma_cluster<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)kR * (unsigned)p.B * (unsigned)p.N, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, (const uint16_t*)p.a, p.alpha, p.beta,
                            (const uint16_t*)p.W, p.w_r, p.H0, p.y, p.H_T,
                            static_cast<uint16_t*>(p.Hs), p.T, p.N, Tc, p.Nqk == 1 ? 0 : 1,
                            p.debug, p.status);
}

}  // namespace m2rnn
