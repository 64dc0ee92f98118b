// m2rnn_bf16_c8.cu — bf16-operand / fp32-state forward recurrence for K = 64, V = 128 on eight
// SMs per (batch, head) pair: eight state rows per CTA, the step product taken transposed on
// the warp-level tensor-core MMA (mma.sync).  Two forms: one 8-CTA thread-block cluster per
// pair (R = 8), or two independent 4-CTA clusters per pair (R = 4, rows 0..31 and 32..63),
// which fit where eight-CTA clusters do not (a GB300 runs 15 clusters of eight at once, but
// 36 of four).
//
// The recurrence is Eq. (10)-(12) with the gate of Eq. (13)/(17) of the M²RNN study notes
// (Sec. 2.1-2.2):
//   f_t = exp(-alpha softplus(a_t + beta)),  H_t = f_t H_{t-1} + (1 - f_t) tanh(H_{t-1} W + k_t v_t^T),
//   y_t = H_t^T q_t + w_r ⊙ v_t.
// Rows of H evolve independently given W and the gate (Sec. 1.2: W mixes value columns, not
// key rows), so a pair can be spread over SMs by rows; only the readout sums over rows.  With
// few pairs (B = 1, N = 16 on 152 SMs) eight SMs per pair put 128 SMs to work.
//
// Mapping.  CTA r of the cluster owns rows 8r .. 8r + 7.  Its four compute warps own value
// columns 32w .. 32w + 31 (column tiles 2w, 2w + 1) and compute, for those columns,
//   P_{t+1}^T (32 x 8) = W^T (32 x 128) H_t^T (128 x 8) + v_{t+1} k_{t+1}^T
// as m16n8k16 MMAs: the W^T rows of their columns sit in register-resident A fragments (two
// m-tiles x eight k-tiles) and the CTA's eight rows are the N = 8 operand.  A lane holds
// rows (8r + 2c, 8r + 2c + 1) of columns 16m + g and 16m + 8 + g (m its two column tiles);
// the bf16 pack of such a pair, transposed by movmatrix, is the B fragment of k-tile m.
// Each step a warp finishes its own two column tiles (tanh, lerp, pack, transpose), writes
// their B fragments into a double-buffered shared-memory slot and issues their MMAs, meets
// the other compute warps at a named barrier, then issues the other six k-tiles.
//
// With R = 4, CTA r of cluster h owns rows 8 (4h + r) .. and y columns 32r .. 32r + 31 of its
// half; each cluster sums its four row blocks and adds the sum into y (red.global.add) after
// the launcher has zeroed y.  With two addends onto an exact zero the bits do not depend on
// which cluster adds first (0 + a = a, a + b = b + a), so y stays deterministic; the two
// clusters never wait for each other.
//
// Readout, two steps per MMA.  The untransposed bf16 pack of a column tile is half of an
// m16n8k16 A fragment over the CTA's eight rows; with A = [H_t^T | H_{t+1}^T] (16 columns x
// the eight rows at t, then at t+1) and B holding q_t in rows 0..7 of column 2m and q_{t+1}
// in rows 8..15 of column 2m + 1 (m = 0, 1 the warp's tiles), lanes c = 0, 1 receive the
// q-weighted row sums of tile 2w + c for both steps.  They store them straight into the
// shared memory of CTA 2w + c, the owner of those 16 y columns, through distributed shared
// memory (mapa + st.shared::cluster).  The readout reads the bf16 rounding of H_t, the
// operand the next step multiplies by W (a 2^-9 relative rounding per term).
//
// Producer warp.  A fifth warp, per chunk of Tc steps: computes the gates (f, 1 - f), starts
// the TMA loads of q, k (the CTA's eight rows) and v (all columns) two chunks ahead, converts
// v into fp32 pairs (v_j, v_j, v_j', v_j') and k into fp32 in the order lanes read them, and,
// once every CTA's partials of a chunk have arrived, sums the eight row blocks' partials in
// CTA order plus w_r ⊙ v into its 16 y columns (deterministic).
// Handoffs are mbarriers: `full` (TMA landed), `conv` (operands converted), `done` (the
// compute warps finished a chunk), `ready` (a chunk's partials for my columns arrived from
// all eight CTAs; remote release arrives) and `fre` (every owner consumed the partials this
// CTA sent).  Every wait is bounded; a timeout raises the CTA's abort flag, which the other
// waits watch, and a final cluster barrier keeps each CTA resident while peers may still
// write to it.
//
// kCache (the training forward) also stores every state H_t as bf16 into Hs [B N, T, K, V]:
// the B fragments a warp publishes for its own k-tiles, i.e. exactly the next product's
// operand.
#include <cuda_bf16.h>

#include <mutex>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 128;
constexpr int kK = 64;
constexpr int kCW = 4;            // compute warps: warp w owns columns 32w .. 32w + 31
constexpr int kThreads = 32 * (kCW + 1);
constexpr int kBar = 1;           // named barrier of the compute warps
constexpr int kTc = 32;           // steps per chunk
constexpr int kMinSmem = 120 * 1024;  // one CTA per SM

struct C8Layout {
  int qs, ks, vs, stage;  // TMA destinations q, k [Tc][8], v [Tc][128] bf16; two stages
  int vd;                 // float4 [2][Tc][8 tiles][8 g] (v_j, v_j, v_j', v_j'), j = 16m + g
  int kf;                 // float  [2][Tc][8]
  int fg;                 // float2 [2][Tc] (f, 1 - f)
  int xbuf;               // uint4  [2][kCW][32] B fragments of each warp's two k-tiles
  int ypart;              // float2 [2][R][Tc / 2][V / R] partials for my columns, (t, t+1)
  int wr;                 // float  [V / R]
  int bar;                // full[2], conv[2], done[2], ready[2], fre[2], never; int abort
  int total;
};

__host__ __device__ inline int c8_al128(int x) { return (x + 127) & ~127; }

// D = A * B (zero accumulator in), m16n8k16, bf16 operands, fp32 result, in the fragment
// layout of mma2 (two float2 rows of the accumulator).
__device__ __forceinline__ void c8_mma2_z(float2 (&d)[2], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0].x), "=f"(d[0].y), "=f"(d[1].x), "=f"(d[1].y)
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}
// Store of two floats into the shared memory of a CTA of the cluster (address from mapa).
__device__ __forceinline__ void c8_st_cluster_v2(uint32_t cluster_addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(cluster_addr), "f"(v.x), "f"(v.y)
               : "memory");
}

__host__ __device__ inline C8Layout c8_layout() {
  C8Layout L;
  L.qs = 0;
  L.ks = c8_al128(kTc * 8 * 2);
  L.vs = L.ks + c8_al128(kTc * 8 * 2);
  L.stage = L.vs + c8_al128(kTc * kV * 2);
  int o = 2 * L.stage;
  L.vd = o;
  o += 2 * kTc * 64 * 16;
  L.kf = o;
  o += c8_al128(2 * kTc * 8 * 4);
  L.fg = o;
  o += c8_al128(2 * kTc * 8);
  L.xbuf = o;
  o += 2 * kCW * 32 * 16;
  L.ypart = o;
  o += 2 * (kTc / 2) * kV * 8;
  L.wr = o;
  o += c8_al128(kV * 4);
  L.bar = o;
  o += 128;
  L.total = o < kMinSmem ? kMinSmem : o;
  return L;
}

template <bool kCache, int R>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_c8(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ a,
                const float* __restrict__ alpha, const float* __restrict__ beta,
                const uint16_t* __restrict__ W, const float* __restrict__ w_r, const float* H0,
                float* __restrict__ y, float* H_T, uint16_t* __restrict__ Hs, int T, int N,
                int qk_hs, int debug, int* status) {
  constexpr int Tc = kTc;
  constexpr int kOwn = kV / R;          // y columns a CTA owns: kOwn rank .. kOwn (rank + 1) - 1
  constexpr int kHalves = 8 / R;        // clusters per pair (rows 8 R h .. of cluster h)
  constexpr int kTilesPerOwner = kOwn / 16;
  extern __shared__ __align__(128) uint8_t smem[];
  const C8Layout L = c8_layout();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster_ctarank();  // y column block of this CTA within its cluster
  const int cid = (int)cluster_id_x();
  const int pair = cid / kHalves, half = cid - (cid / kHalves) * kHalves;
  const int rb = half * R + rank;           // row block: rows 8 rb .. 8 rb + 7
  const int b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + Tc - 1) / Tc;
  const size_t row_base = (size_t)b * T;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* conv = full + 2;
  uint64_t* done = full + 4;
  uint64_t* ready = full + 6;
  uint64_t* fre = full + 8;
  uint64_t* never = full + 10;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 11);
  float4* vd = reinterpret_cast<float4*>(smem + L.vd);
  float* kf = reinterpret_cast<float*>(smem + L.kf);
  float2* fgs = reinterpret_cast<float2*>(smem + L.fg);
  uint4* xbuf = reinterpret_cast<uint4*>(smem + L.xbuf);
  float2* ypart = reinterpret_cast<float2*>(smem + L.ypart);
  float* wrs = reinterpret_cast<float*>(smem + L.wr);
  const long long limit = kWaitLimitCycles;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&conv[i], 32);
      mbar_init(&done[i], 32 * kCW);
      mbar_init(&ready[i], 32 * R);  // lanes of the warp(s) of every CTA whose tiles I own
      mbar_init(&fre[i], 32 * R);    // producer lanes of every owner
    }
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kOwn) wrs[tid] = w_r[(size_t)n * kV + kOwn * rank + tid];
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive

  if (warp == kCW) {
    // ======================================================= producer warp
    const float al = alpha[n], be = beta[n];
    const uint32_t stage_tx = (uint32_t)Tc * (8u + 8u + (uint32_t)kV) * 2u;
    auto arm = [&](int cc) {  // gates of chunk cc, then its TMA loads, into stage cc & 1
      const int st = cc & 1;
      for (int s = lane; s < Tc; s += 32) {
        const int t = cc * Tc + s;
        const float av = t < T ? bf16_bits_to_float(a[(row_base + t) * N + n]) : 0.f;
        fgs[st * Tc + s] = gate_fg(av, al, be);
      }
      if (lane == 0) {
        uint8_t* base = smem + st * L.stage;
        mbar_arrive_expect_tx(&full[st], stage_tx);
        tma_load_4d(base + L.qs, &tm_q, &full[st], 8 * rb, n * qk_hs, cc * Tc, b);
        tma_load_4d(base + L.ks, &tm_k, &full[st], 8 * rb, n * qk_hs, cc * Tc, b);
        tma_load_4d(base + L.vs, &tm_v, &full[st], 0, n, cc * Tc, b);
      }
    };
    // Chunk cc's v and k (stage cc & 1 has landed) into the fp32 operand buffers.
    auto convert = [&](int cc) {
      const int st = cc & 1;
      const uint8_t* raw = smem + st * L.stage;
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(raw + L.vs);
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(raw + L.ks);
      float4* vdst = vd + (size_t)st * Tc * 64;
      for (int e = lane; e < Tc * 64; e += 32) {  // e = (s, tile m, g)
        const int s = e >> 6, m = (e >> 3) & 7, gg = e & 7;
        const float v0 = bf16_bits_to_float(vs[s * kV + 16 * m + gg]);
        const float v1 = bf16_bits_to_float(vs[s * kV + 16 * m + 8 + gg]);
        vdst[e] = make_float4(v0, v0, v1, v1);
      }
      for (int e = lane; e < Tc * 8; e += 32) kf[st * Tc * 8 + e] = bf16_bits_to_float(ks[e]);
    };
    auto land_and_convert = [&](int cc) -> bool {
      const bool ok = wait_or_abort(&full[cc & 1], (uint32_t)(cc >> 1) & 1u, limit, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) return false;
      convert(cc);
      mbar_arrive(&conv[cc & 1]);
      return true;
    };
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    int issued = 0;
    for (; issued < 2 && issued < nchunks; ++issued) arm(issued);
    bool ok = true;
    for (int cc = 0; cc < 2 && cc < nchunks && ok; ++cc) ok = land_and_convert(cc);
    for (int cc = 0; cc < nchunks && ok; ++cc) {
      const int st = cc & 1;
      const uint32_t par = (uint32_t)(cc >> 1) & 1u;
      bool w = wait_or_abort(&done[st], par, limit, abort_flag);
      w = w && mbar_wait_cluster(&ready[st], par, limit, abort_flag);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      // y_t[kOwn rank + jj]: the cluster's R row blocks' partials in CTA order, plus w_r ⊙ v_t
      // (cluster 0 of the pair).  One cluster per pair stores y; with two (R = 4) each adds
      // its sum into y, which the host zeroed: two addends onto an exact zero give the same
      // bits in either order (0 + a = a, a + b = b + a).
      const int steps = min(Tc, T - cc * Tc);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + st * L.stage + L.vs);
      const float2* yp = ypart + (size_t)st * R * (Tc / 2) * kOwn;
      for (int idx = lane; idx < ((steps + 1) >> 1) * kOwn; idx += 32) {
        const int s2 = idx / kOwn, jj = idx - s2 * kOwn, s = 2 * s2;
        const int col = kOwn * rank + jj;
        float2 u[R];
#pragma unroll
        for (int r = 0; r < R; ++r) u[r] = yp[((size_t)r * (Tc / 2) + s2) * kOwn + jj];
        float* y0 = y + ((row_base + (size_t)cc * Tc + s) * N + n) * kV + col;
        float o0 = half == 0 ? wrs[jj] * bf16_bits_to_float(vs[s * kV + col]) : 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) o0 += u[r].x;
        if (kHalves == 1)
          *y0 = o0;
        else
          atomicAdd(y0, o0);
        if (s + 1 < steps) {
          float* y1 = y0 + (size_t)N * kV;
          float o1 = half == 0 ? wrs[jj] * bf16_bits_to_float(vs[(s + 1) * kV + col]) : 0.f;
#pragma unroll
          for (int r = 0; r < R; ++r) o1 += u[r].y;
          if (kHalves == 1)
            *y1 = o1;
          else
            atomicAdd(y1, o1);
        }
      }
      // This chunk's partials are consumed: tell every CTA (each lane's own reads are done).
#pragma unroll
      for (int r = 0; r < R; ++r) mbar_arrive_cluster(mapa_shared(smem_u32(&fre[st]), (uint32_t)r));
      if (issued < nchunks) {
        arm(issued);
        ok = land_and_convert(issued);
        ++issued;
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicExch(status, kStatusTimeout);
      // Let the loads in flight land before the CTA can leave.
      for (int ci = issued > 2 ? issued - 2 : 0; ci < issued; ++ci)
        mbar_wait_bounded(&full[ci & 1], (uint32_t)(ci >> 1) & 1u, kDebugWaitLimitCycles);
    }
  } else {
    // ======================================================= compute warps
    const int w = warp;
    const int g = lane >> 2, c = lane & 3;
    const int i0 = 8 * rb + 2 * c;  // the lane's accumulator rows i0, i0 + 1

    // W^T A fragments of the warp's column tiles ct = 2w + mm: rows j = 16 ct + g (+8) of W^T,
    // columns l = 16 kt + 2c (+1, +8, +9), i.e. W[l][j].  Own k-tiles (2w + u) in wo, those of
    // warp (w + 1 + i) & 3 in wx[i], so that every register index is static.
    const uint16_t* Wn = W + (size_t)n * kV * kV;
    auto wfrag = [&](int ct, int kt, uint32_t (&f)[4]) {
      const int l = 16 * kt + 2 * c, j = 16 * ct + g;
      f[0] = (uint32_t)Wn[l * kV + j] | ((uint32_t)Wn[(l + 1) * kV + j] << 16);
      f[1] = (uint32_t)Wn[l * kV + j + 8] | ((uint32_t)Wn[(l + 1) * kV + j + 8] << 16);
      f[2] = (uint32_t)Wn[(l + 8) * kV + j] | ((uint32_t)Wn[(l + 9) * kV + j] << 16);
      f[3] = (uint32_t)Wn[(l + 8) * kV + j + 8] | ((uint32_t)Wn[(l + 9) * kV + j + 8] << 16);
    };
    uint32_t wo[2][2][4], wx[3][2][2][4];
#pragma unroll
    for (int mm = 0; mm < 2; ++mm)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        wfrag(2 * w + mm, 2 * w + u, wo[mm][u]);
#pragma unroll
        for (int i = 0; i < 3; ++i) wfrag(2 * w + mm, 2 * ((w + 1 + i) & 3) + u, wx[i][mm][u]);
      }

    // State (fp32) in the accumulator layout: h[mm][hh] = (H[i0][j], H[i0 + 1][j]),
    // j = 16 (2w + mm) + 8 hh + g.
    float2 h[2][2];
    {
      const float* hp = H0 ? H0 + (size_t)pair * kK * kV : nullptr;
#pragma unroll
      for (int mm = 0; mm < 2; ++mm)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int j = 16 * (2 * w + mm) + 8 * hh + g;
          h[mm][hh] = hp ? make_float2(hp[(size_t)i0 * kV + j], hp[(size_t)(i0 + 1) * kV + j])
                         : make_float2(0.f, 0.f);
        }
    }
    // Lanes c < 2 send the readout of tile 2w + c: its owner within the cluster, the remote
    // base address of the owner's partial buffers, and the tile's first local column there.
    const int my_tile = 2 * w + (c & 1);
    const int owner = my_tile / kTilesPerOwner;
    const uint32_t yremote = mapa_shared(smem_u32(ypart), (uint32_t)owner);
    const int ycol0 = 16 * (my_tile - owner * kTilesPerOwner);

    // A step's shared-memory operands, loaded during the step before: the gate and q of step
    // t, v and k of step t + 1 (its rank-1 term).
    struct StepIn {
      float2 fg, kk;
      float4 v[2];
      uint32_t qp;
    };
    struct ChunkPtrs {
      const float4 *vd0, *vd1;
      const float *kf0, *kf1;
      const uint16_t *q0, *q1;
      const float2 *fg0, *fg1;
    };
    auto chunk_ptrs = [&](int cc) {
      ChunkPtrs P;
      const int s0 = cc & 1, s1 = s0 ^ 1;
      P.vd0 = vd + (size_t)s0 * Tc * 64;
      P.vd1 = vd + (size_t)s1 * Tc * 64;
      P.kf0 = kf + s0 * Tc * 8;
      P.kf1 = kf + s1 * Tc * 8;
      P.q0 = reinterpret_cast<const uint16_t*>(smem + s0 * L.stage + L.qs);
      P.q1 = reinterpret_cast<const uint16_t*>(smem + s1 * L.stage + L.qs);
      P.fg0 = fgs + s0 * Tc;
      P.fg1 = fgs + s1 * Tc;
      return P;
    };
    // Operands of the step after step s: gate and q of step s + 1, v and k of step s + 2 (either
    // may fall in the next chunk, converted before they are read; past the end of the sequence
    // they are stale and never used).
    auto fetch = [&](StepIn& in, const ChunkPtrs& P, int s, int steps) {
      const bool n1 = s + 1 >= steps, n2 = s + 2 >= steps;
      const int s1 = n1 ? s + 1 - steps : s + 1, s2 = n2 ? s + 2 - steps : s + 2;
      in.fg = (n1 ? P.fg1 : P.fg0)[s1];
      in.qp = *reinterpret_cast<const uint32_t*>((n1 ? P.q1 : P.q0) + s1 * 8 + 2 * c);
      in.kk = *reinterpret_cast<const float2*>((n2 ? P.kf1 : P.kf0) + s2 * 8 + 2 * c);
      const float4* vp = (n2 ? P.vd1 : P.vd0) + (size_t)s2 * 64 + 2 * w * 8 + g;
      in.v[0] = vp[0];
      in.v[1] = vp[8];
    };
    auto rank1 = [&](float2 (&nx)[2][2], const StepIn& si) {
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        nx[mm][0] = mul2(si.kk, make_float2(si.v[mm].x, si.v[mm].y));
        nx[mm][1] = mul2(si.kk, make_float2(si.v[mm].z, si.v[mm].w));
      }
    };
    // Own k-tile u of H_t (B fragment bo) into slot px and its MMAs.
    auto own_tile = [&](float2 (&nx)[2][2], uint4* xs, int u, uint32_t b0, uint32_t b1) {
      reinterpret_cast<uint2*>(xs + w * 32 + lane)[u] = make_uint2(b0, b1);
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) mma2(nx[mm], wo[mm][u], b0, b1);
    };
    // After the barrier: the other warps' six k-tiles, the first of each pair into a second
    // accumulator (two dependent chains of three per column tile instead of one of six, so the
    // MMA latency overlaps), added in at the end.
    auto other_tiles = [&](float2 (&nx)[2][2], const uint4* xs) {
      float2 nx2[2][2];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const uint4 x = xs[((w + 1 + i) & 3) * 32 + lane];
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          if (i == 0)
            c8_mma2_z(nx2[mm], wx[i][mm][0], x.x, x.y);
          else
            mma2(nx2[mm], wx[i][mm][0], x.x, x.y);
          mma2(nx[mm], wx[i][mm][1], x.z, x.w);
        }
      }
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        nx[mm][0] = add2(nx[mm][0], nx2[mm][0]);
        nx[mm][1] = add2(nx[mm][1], nx2[mm][1]);
      }
    };

    bool ok = wait_or_abort(&conv[0], 0u, limit, abort_flag);
    if (debug & kDebugForceTimeout) ok = ok && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
    if (nchunks > 1) ok = ok && wait_or_abort(&conv[1], 0u, limit, abort_flag);
    bool aborted = named_bar_or(kBar, 32 * kCW, !ok);

    // P_0 = v_0 k_0^T + W^T H_0^T (exchange slot 1; step 0 uses slot 0).
    float2 acc[2][2], nxt[2][2];
    StepIn in;
    if (!aborted) {
      const ChunkPtrs P0 = chunk_ptrs(0);
      StepIn s0;
      s0.kk = *reinterpret_cast<const float2*>(P0.kf0 + 2 * c);
      s0.v[0] = P0.vd0[2 * w * 8 + g];
      s0.v[1] = P0.vd0[2 * w * 8 + 8 + g];
      rank1(acc, s0);
      fetch(in, P0, -1, min(Tc, T));  // step 0's operands
      uint4* xs = xbuf + 1 * kCW * 32;
#pragma unroll
      for (int u = 0; u < 2; ++u)
        own_tile(acc, xs, u, movmatrix_trans(pack_bf16x2(h[u][0].x, h[u][0].y)),
                 movmatrix_trans(pack_bf16x2(h[u][1].x, h[u][1].y)));
      named_bar_sync(kBar, 32 * kCW);
      other_tiles(acc, xs);
    }

    // One time step (step s of the chunk, exchange slot px).  On entry `cur` holds P_t, h holds
    // H_{t-1} and `in` this step's operands; on exit h holds H_t, `nx` holds P_{t+1}, `in` the
    // next step's operands, and ap, qp the bf16 pack of H_t and q_t.
    auto step = [&](float2 (&cur)[2][2], float2 (&nx)[2][2], const ChunkPtrs& P, int s,
                    int steps, int px, uint16_t* hs, uint32_t (&ap)[2][2], uint32_t& qp) {
      const StepIn cin = in;
      fetch(in, P, s, steps);
      qp = cin.qp;
      rank1(nx, cin);
      const float2 ff = make_float2(cin.fg.x, cin.fg.x), gg = make_float2(cin.fg.y, cin.fg.y);
      uint4* xs = xbuf + px * kCW * 32;
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        // Eq. (10)-(11): Z = tanh(P), H = f H + (1 - f) Z, for column tile 2w + mm.
        const float z0 = tanh_mufu(cur[mm][0].x), z1 = tanh_mufu(cur[mm][0].y);
        const float z2 = tanh_mufu(cur[mm][1].x), z3 = tanh_mufu(cur[mm][1].y);
        h[mm][0] = fma2(gg, make_float2(z0, z1), mul2(ff, h[mm][0]));
        h[mm][1] = fma2(gg, make_float2(z2, z3), mul2(ff, h[mm][1]));
        ap[mm][0] = pack_bf16x2(h[mm][0].x, h[mm][0].y);
        ap[mm][1] = pack_bf16x2(h[mm][1].x, h[mm][1].y);
        const uint32_t b0 = movmatrix_trans(ap[mm][0]), b1 = movmatrix_trans(ap[mm][1]);
        if (kCache) {  // row 8 rb + g, columns 16 (2w + mm) + 2c (+1) and + 8
          uint32_t* hr = reinterpret_cast<uint32_t*>(hs + (size_t)(8 * rb + g) * kV +
                                                     16 * (2 * w + mm) + 2 * c);
          __stcs(hr, b0);
          __stcs(hr + 4, b1);
        }
        own_tile(nx, xs, mm, b0, b1);
      }
      named_bar_sync(kBar, 32 * kCW);
      other_tiles(nx, xs);
    };
    // Eq. (12) readout of steps s and s + 1 (s even) over this CTA's rows for tiles 2w, 2w + 1,
    // into the owners' partial buffer `buf`.  A lone last step passes q_{s+1} = 0.
    auto readout2 = [&](int buf, const uint32_t (&apA)[2][2], const uint32_t (&apB)[2][2],
                        uint32_t qA, uint32_t qB, int s) {
      float d[2][4];
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const uint32_t af[4] = {apA[mm][0], apA[mm][1], apB[mm][0], apB[mm][1]};
        mma_bf16_16816_z(d[mm], af, g == 2 * mm ? qA : 0u, g == 2 * mm + 1 ? qB : 0u);
      }
      if (c < 2) {  // tile 2w + c: (y_s, y_{s+1}) of local columns g and g + 8
        const float2 lo = add2(make_float2(d[0][0], d[0][1]), make_float2(d[1][0], d[1][1]));
        const float2 hi = add2(make_float2(d[0][2], d[0][3]), make_float2(d[1][2], d[1][3]));
        const uint32_t off =
            (uint32_t)((((size_t)buf * R + rank) * (Tc / 2) + (s >> 1)) * kOwn + ycol0 + g) * 8u;
        c8_st_cluster_v2(yremote + off, lo);
        c8_st_cluster_v2(yremote + off + 64u, hi);
      }
    };

    for (int cc = 0; cc < nchunks && !aborted; ++cc) {
      const int st = cc & 1;
      const int steps = min(Tc, T - cc * Tc);
      const ChunkPtrs P = chunk_ptrs(cc);
      if (cc >= 2) {  // every owner consumed the partials this CTA sent for chunk cc - 2
        const bool w_ok =
            mbar_wait_cluster(&fre[st], (uint32_t)((cc >> 1) - 1) & 1u, limit, abort_flag);
        if (named_bar_or(kBar, 32 * kCW, !w_ok)) {
          aborted = true;
          break;
        }
      }
      // A chunk with a successor is whole; its last trip reads the successor's operands,
      // converted by the producer (chunk 1's before the loop).
      const int s_wait = (cc >= 1 && cc + 1 < nchunks) ? Tc - 2 : -1;
      uint16_t* hs_chunk = kCache ? Hs + ((size_t)pair * T + (size_t)cc * Tc) * kK * kV : nullptr;
      auto trip = [&](int s) {
        uint32_t apA[2][2], apB[2][2], qA, qB;
        step(acc, nxt, P, s, steps, 0, kCache ? hs_chunk + (size_t)s * kK * kV : nullptr, apA,
             qA);
        step(nxt, acc, P, s + 1, steps, 1,
             kCache ? hs_chunk + (size_t)(s + 1) * kK * kV : nullptr, apB, qB);
        readout2(st, apA, apB, qA, qB, s);
      };
      int s = 0;
      for (; s + 1 < steps && s != s_wait; s += 2) trip(s);
      if (s == s_wait) {
        const bool w_ok =
            wait_or_abort(&conv[(cc + 1) & 1], (uint32_t)((cc + 1) >> 1) & 1u, limit, abort_flag);
        if (named_bar_or(kBar, 32 * kCW, !w_ok)) {
          aborted = true;
          break;
        }
        trip(s);
        s += 2;
      }
      if (s < steps) {  // odd tail of the last chunk
        uint32_t apA[2][2], apB[2][2], qA;
        step(acc, nxt, P, s, steps, 0, kCache ? hs_chunk + (size_t)s * kK * kV : nullptr, apA,
             qA);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          apB[mm][0] = apB[mm][1] = 0u;
          acc[mm][0] = nxt[mm][0];
          acc[mm][1] = nxt[mm][1];
        }
        readout2(st, apA, apB, qA, 0u, s);
      }
      // This chunk's partials are sent: signal the owner(s) of my two tiles, release the stage.
      if (kTilesPerOwner == 1) {
        mbar_arrive_cluster(mapa_shared(smem_u32(&ready[st]), (uint32_t)(2 * w)));
        mbar_arrive_cluster(mapa_shared(smem_u32(&ready[st]), (uint32_t)(2 * w + 1)));
      } else {
        mbar_arrive_cluster(mapa_shared(smem_u32(&ready[st]), (uint32_t)(2 * w / kTilesPerOwner)));
      }
      mbar_arrive(&done[st]);
    }
    if (aborted) {
      *abort_flag = 1;
      if (lane == 0) atomicExch(status, kStatusTimeout);
    } else if (H_T) {
      float* hp = H_T + (size_t)pair * kK * kV;
#pragma unroll
      for (int mm = 0; mm < 2; ++mm)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int j = 16 * (2 * w + mm) + 8 * hh + g;
          hp[(size_t)i0 * kV + j] = h[mm][hh].x;
          hp[(size_t)(i0 + 1) * kV + j] = h[mm][hh].y;
        }
    }
  }
  // No CTA leaves while a peer may still write into its shared memory or arrive on its
  // barriers.
  cluster_sync_all();
}

bool make_map_c8(EncodeTiledFn enc, CUtensorMap* map, const void* base, int inner, int box, int N,
                 int T, int B) {
  const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)N, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * N,
                                 (cuuint64_t)inner * 2 * N * T};
  const cuuint32_t boxd[4] = {(cuuint32_t)box, 1u, (cuuint32_t)kTc, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, boxd,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Grid of 8 CTAs per pair (8 / R clusters of R), one CTA per SM (dynamic shared memory above
// half an SM).
template <int R>
cudaLaunchConfig_t c8_config(int pairs, cudaStream_t stream, cudaLaunchAttribute* attr) {
  const C8Layout L = c8_layout();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(8u * (unsigned)pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool kCache, int R>
cudaError_t c8_prepare() {
  return cudaFuncSetAttribute(fwd_bf16_c8<kCache, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              c8_layout().total);
}

template <int R>
int c8_max_clusters() {
  static int cache[64];
  static bool known[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (known[dev]) return cache[dev];
  int n = 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = c8_config<R>(1, nullptr, attr);
  if (c8_prepare<false, R>() != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, fwd_bf16_c8<false, R>, &cfg) != cudaSuccess)
    n = 0;
  cache[dev] = n;
  known[dev] = true;
  return n;
}

template <int R>
cudaError_t launch_c8(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map_c8(enc, &mq, p.q, kK, 8, p.Nqk, p.T, p.B) ||
      !make_map_c8(enc, &mk, p.k, kK, 8, p.Nqk, p.T, p.B) ||
      !make_map_c8(enc, &mv, p.v, kV, kV, p.N, p.T, p.B))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  const int pairs = p.B * p.N;
  const int qk_hs = p.Nqk == 1 ? 0 : 1;
  if (R < 8) {  // two clusters per pair add their sums into y
    cudaError_t err =
        cudaMemsetAsync(p.y, 0, sizeof(float) * (size_t)p.B * p.T * p.N * kV, stream);
    if (err != cudaSuccess) return err;
  }
  if (p.Hs) {
    cudaError_t err = c8_prepare<true, R>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = c8_config<R>(pairs, stream, attr);
    return cudaLaunchKernelEx(&cfg, fwd_bf16_c8<true, R>, mq, mk, mv, (const uint16_t*)p.a,
                              p.alpha, p.beta, (const uint16_t*)p.W, p.w_r, p.H0, p.y, p.H_T,
                              static_cast<uint16_t*>(p.Hs), p.T, p.N, qk_hs, p.debug, p.status);
  }
  cudaError_t err = c8_prepare<false, R>();
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = c8_config<R>(pairs, stream, attr);
  return cudaLaunchKernelEx(&cfg, fwd_bf16_c8<false, R>, mq, mk, mv, (const uint16_t*)p.a,
                            p.alpha, p.beta, (const uint16_t*)p.W, p.w_r, p.H0, p.y, p.H_T,
                            static_cast<uint16_t*>(nullptr), p.T, p.N, qk_hs, p.debug, p.status);
}

}  // namespace

bool mma_c8_supports(int K, int V) { return K == kK && V == kV; }

// Clusters of the R-CTA form the current device runs at once (0 when it cannot say), cached
// per device (under a mutex): a form pays only when all its clusters are resident at once.
int mma_c8_max_clusters(int R) { return R == 8 ? c8_max_clusters<8>() : c8_max_clusters<4>(); }

cudaError_t launch_fwd_bf16_mma_c8(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                                   int R) {
  return R == 8 ? launch_c8<8>(p, enc, stream) : launch_c8<4>(p, enc, stream);
}

}  // namespace m2rnn
