// m2rnn_bf16_r8.cu — bf16-operand / fp32-state forward recurrence with eight state rows per
// warp and each step's product taken transposed, on the warp-level tensor-core MMA
// (mma.sync), for K in {32, 64} and V in {16, 32, 48, 64}; one thread block per (batch, head)
// pair, or (K = 64, few pairs) a two-block cluster per pair.
//
// The recurrence is the M²RNN study notes' Sec. 2.1 Eq. (10)-(12) with the gate of Sec. 2.2
// Eq. (13)/(17):
//   f_t = exp(-alpha softplus(a_t + beta)),  H_t = f_t H_{t-1} + (1 - f_t) tanh(H_{t-1} W + k_t v_t^T),
//   y_t = H_t^T q_t + w_r ⊙ v_t,
// one thread block per (batch, head) pair (Sec. 2.6: pairs are independent units).
//
// Mapping.  W mixes value columns, not key rows (Sec. 1.2), so row i of H_t depends only on
// row i of H_{t-1}, on W, and on the step's scalars: the K rows are K independent chains that
// meet only in the readout.  Compute warp w owns rows 8w .. 8w + 7 (at K = 64 two compute
// warps share each sub-partition, so one warp's MMAs overlap the other's tanh) and computes
//   P_t^T (V x 8) = W^T (V x V) H_{t-1}^T (V x 8)  +  v_t k_t^T
// as m16n8k16 MMAs with W^T in register-resident A fragments and its eight state rows as the
// B operand.  Its accumulator holds rows (8w + 2c, 8w + 2c + 1) of columns 16m + g and
// 16m + 8 + g; the bf16 pack of such a pair, transposed by movmatrix, is the B fragment of
// k-tile m of the next step, so the state stays in fp32 registers for the whole sequence.
// Column tile m of H_t is finished (tanh, lerp, pack, transpose) and immediately used as
// k-tile m of step t+1's MMAs, so the MMAs of one tile overlap the tanh of the next.  A step's
// shared-memory operands are loaded during the step before.
//
// Readout on the tensor core, two steps per MMA.  The untransposed bf16 pack of a column
// tile is exactly an A-fragment half of an m16n8k16 MMA over the warp's eight rows, so with
// A = [H_t^T | H_{t+1}^T] (16 columns j x 16: the warp's rows at step t, then at step t+1)
// and B holding q_t in rows 0..7 of column 2m and q_{t+1} in rows 8..15 of column 2m + 1,
//   D[j][2m] = y_part_t[16m + j],  D[j][2m + 1] = y_part_{t+1}[16m + j]
// for column tile m (y_part: the sum over this warp's rows r of H[r][.] q[r]).  Each tile has
// its own accumulator (no MMA waits on another); lane (g, c) takes its values from tile c,
// the other tiles giving it exact zeros: both steps' y_part[16c + g] and y_part[16c + 8 + g],
// four stores per two steps, no shuffles.  The readout thus reads the bf16 rounding of H_t
// (the operand the next step's H W uses); its error, a 2^-9 relative rounding of each term,
// stays far inside the bf16 path's bar.
//
// Helper warps.  Four more warps, one per sub-partition, do everything that is not the step
// chain, concurrently with it and chunk by chunk (Tc steps), ordered by mbarriers:
//   * once the compute warps have finished chunk c (`pdone`): sum chunk c's per-warp readout
//     partials plus w_r ⊙ v into y (warps in order, so y is deterministic; `ydone`; the
//     partial buffers are double-buffered), start the TMA load of chunk c+3 into the stage
//     chunk c used (three stages, mbarrier completion), and convert chunk c+2 (its load has
//     landed) into the operand buffer chunk c used: v as fp32 pairs (v_j, v_j) in the order a
//     lane reads them, k in fp32, and, every G chunks, the next batch of gates (f, 1 - f),
//     one per helper thread, from logits loaded a batch earlier (`cready`);
//   * the compute warps wait only for chunk c+1's operands before the last trip (two steps)
//     of chunk c, whose prefetch reads them, and for a free partial buffer at a chunk's
//     start; both are normally complete long before.
// Two-block clusters (CS = 2).  When the pairs fill at most half the GPU, a pair's rows are
// split over the two blocks of a cluster (block r owns rows 32r .. 32r + 31, four compute
// warps, one per sub-partition), which halves each sub-partition's share of the step chain.
// Only the readout couples the blocks, and only through the helpers: the compute warps run
// exactly as in a one-block pair (local partials, local barriers).  Block r owns y columns
// [rV/2, (r+1)V/2).  Each block's helpers sum their own warps' partials of chunk c and store
// the sums of each column into the owning block's exchange buffer through distributed shared
// memory (mapa + st.shared::cluster; `xready`, arrived on at cluster scope); the owner adds
// the two blocks' sums in block order (deterministic) plus w_r ⊙ v into y and releases the
// buffers (`xfree`).  Each block loads and converts its own copy of the operands.  Both
// blocks stay resident until a final cluster barrier that every thread reaches, also after
// a timeout.
//
// With that work off the compute warps, their step machinery fits the 168 registers per
// thread a 384-thread block allows.  Every wait is bounded; a timeout raises a block-wide
// abort flag that every other wait also watches.  Every thread arrives on the mbarriers that
// order its shared-memory writes (or reads) before another warp's, so that its own arrive
// releases them.
#include <cuda_bf16.h>

#include <cstring>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kR8Tc = 32;      // steps per chunk
constexpr int kR8Helpers = 4;  // helper warps (one warpgroup, one warp per sub-partition)
constexpr int kR8GateChunks = 32 * kR8Helpers / kR8Tc;  // chunks per gate batch (G)

struct R8Layout {
  int qs, ks, vs, stage;  // raw bf16 TMA destinations; three stages `stage` bytes apart
  int cb;                 // operand buffers (two, `cbuf` bytes apart) start here:
  int vd, kf, cbuf;       //   float4 [Tc][8][MT] (v_j, v_j, v_j', v_j'); float [Tc][K]
  int ypart, ybuf;        // float [2][K / 8 / CS][Tc][V] this block's warps' readout partials
  int xpart, xbuf;        // CS > 1: float [2][CS][Tc][V / CS] per-block sums for this block's
                          //   columns, `xbuf` apart
  int fgr;                // float2 [2][G Tc] gates of two batches of G chunks
  int wr;                 // float [V]
  int cw;                 // fused prologue: float [2K + V][4] conv taps, then [2K + V] biases
  int halo;               //   bf16 [2][3][2K + V] last three raw rows of a chunk, by parity
  int mid;                //   bf16 [3][2K + V] raw rows Tc/2 - 3 .. Tc/2 - 1 of the chunk
  int bar;                // uint64 full[3], pdone[2], ydone[2], cready, never, xready[2],
                          //   xfree[2]; int abort
  int total;
};

__host__ __device__ inline int r8_al128(int x) { return (x + 127) & ~127; }

__host__ __device__ inline R8Layout r8_layout(int K, int V, int CS, bool conv = false) {
  constexpr int Tc = kR8Tc;
  R8Layout L;
  const int MT = V / 16;
  L.qs = 0;
  L.ks = r8_al128(Tc * K * 2);
  L.vs = L.ks + r8_al128(Tc * K * 2);
  L.stage = L.vs + r8_al128(Tc * V * 2);
  L.cb = 3 * L.stage;
  L.vd = 0;
  L.kf = r8_al128(Tc * 8 * 2 * MT * 8);
  L.cbuf = L.kf + r8_al128(Tc * K * 4);
  L.ypart = L.cb + 2 * L.cbuf;
  L.ybuf = r8_al128((K / 8 / CS) * Tc * V * 4);
  L.xpart = L.ypart + 2 * L.ybuf;
  L.xbuf = CS > 1 ? r8_al128(CS * Tc * (V / CS) * 4) : 0;
  L.fgr = L.xpart + 2 * L.xbuf;
  L.wr = L.fgr + r8_al128(2 * kR8GateChunks * Tc * 8);
  const int C = 2 * K + V;
  L.cw = L.wr + r8_al128(V * 4);
  L.halo = L.cw + (conv ? r8_al128(C * 5 * 4) : 0);
  L.mid = L.halo + (conv ? r8_al128(2 * 3 * C * 2) : 0);
  L.bar = L.mid + (conv ? r8_al128(3 * C * 2) : 0);
  L.total = L.bar + 160;
  return L;
}

// The block prologue's causal depthwise conv (kernel 4) and SiLU, for one channel: the same
// fp32 operations in the same order as the separate prologue kernel (m2rnn_block.cu), so the
// fused forward's operands are those bits.
__device__ __forceinline__ float r8_conv_silu(const float* tap, float bias, float x3, float x2,
                                              float x1, float x0) {
  float acc = bias;
  acc = fmaf(tap[0], x3, acc);
  acc = fmaf(tap[1], x2, acc);
  acc = fmaf(tap[2], x1, acc);
  acc = fmaf(tap[3], x0, acc);
  return __fdividef(acc, 1.f + __expf(-acc));
}
__device__ __forceinline__ uint16_t r8_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// kConv: the block prologue is fused in.  The TMA stages then hold the raw projections x_q,
// x_k, x_v; the helpers put each chunk through the conv and SiLU (bf16 results: q and v back
// into the stage in place, k and v also into the fp32 operand buffers) before the compute warps
// read it.  Conv taps and biases come as [C][4] and [C] per tensor (C = heads x width).
template <int MT, int CS, bool kConv>
__global__ void __launch_bounds__(384, 1)
    fwd_bf16_r8(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ a,
                const float* __restrict__ alpha, const float* __restrict__ beta,
                const uint16_t* __restrict__ W, const float* __restrict__ w_r, const float* H0,
                float* __restrict__ y, float* H_T, int T, int N, int K, int qk_hs, int debug,
                int* status, const float* __restrict__ cw_q, const float* __restrict__ cb_q,
                const float* __restrict__ cw_k, const float* __restrict__ cb_k,
                const float* __restrict__ cw_v, const float* __restrict__ cb_v) {
  constexpr int V = 16 * MT;
  constexpr int VL = V / CS;  // y columns this block owns: rank VL .. rank VL + VL - 1
  constexpr int Tc = kR8Tc;
  constexpr int G = kR8GateChunks, GB = G * Tc;  // chunks and steps per gate batch
  extern __shared__ __align__(128) uint8_t smem[];
  const R8Layout L = r8_layout(K, V, CS, kConv);
  const int wt = K / 8;       // compute warps of the pair
  const int nw = wt / CS;     // compute warps of this block; warps nw .. nw + 3 are the helpers
  const int rank = CS > 1 ? (int)cluster_ctarank() : 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
  const int pair = blockIdx.x / CS, b = pair / N, n = pair - (pair / N) * N;
  const int nchunks = (T + Tc - 1) / Tc;
  const size_t row_base = (size_t)b * T;  // (b, t) row index base
  const int tma_tid = 32 * nw;            // helper thread 0 issues every TMA load

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* pdone = full + 3;   // [2]: compute warps finished chunk c, on pdone[c & 1]
  uint64_t* ydone = full + 5;   // [2]: chunk c's y summed, on ydone[c & 1]
  uint64_t* cready = full + 7;  // chunk c's operands converted (c >= 2)
  uint64_t* never = full + 8;   // never armed: the forced-timeout test hook waits on it
  uint64_t* xready = full + 9;  // [2]: both blocks' sums of chunk c stored here (CS > 1)
  uint64_t* xfree = full + 11;  // [2]: both owners have read this block's sums of chunk c
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 13);
  float* xpart = reinterpret_cast<float*>(smem + L.xpart);
  float2* fgr = reinterpret_cast<float2*>(smem + L.fgr);
  float* ypart = reinterpret_cast<float*>(smem + L.ypart);
  float* wrs = reinterpret_cast<float*>(smem + L.wr);
  const float al = alpha[n], be = beta[n];
  const uint32_t stage_tx = (uint32_t)(2 * K + V) * (uint32_t)Tc * 2u;
  const long long limit = kWaitLimitCycles;

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&full[i], 1);
    mbar_init(&pdone[0], 32 * nw);  // every compute lane of the block
    mbar_init(&pdone[1], 32 * nw);
    mbar_init(&ydone[0], 32 * kR8Helpers);  // every helper lane of the block
    mbar_init(&ydone[1], 32 * kR8Helpers);
    mbar_init(cready, 32 * kR8Helpers);
    mbar_init(never, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xready[i], 32 * kR8Helpers * CS);  // every helper lane of the pair
      mbar_init(&xfree[i], 32 * kR8Helpers * CS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int j = tid; j < V; j += nthreads) wrs[j] = w_r[(size_t)n * V + j];
  // Fused prologue: this pair's conv taps and biases (q, k channels of head n * qk_hs, v of
  // head n) in channel order q, k, v; the halo of chunk 0 (steps -3 .. -1) is zero.
  float* cws = reinterpret_cast<float*>(smem + L.cw);
  uint16_t* halo = reinterpret_cast<uint16_t*>(smem + L.halo);
  uint16_t* mid = reinterpret_cast<uint16_t*>(smem + L.mid);
  const int CC = 2 * K + V;  // conv channels of the pair
  if constexpr (kConv) {
    for (int c = tid; c < CC; c += nthreads) {
      const float* wsrc;
      const float* bsrc;
      int gc;
      if (c < K) {
        wsrc = cw_q, bsrc = cb_q, gc = n * qk_hs * K + c;
      } else if (c < 2 * K) {
        wsrc = cw_k, bsrc = cb_k, gc = n * qk_hs * K + c - K;
      } else {
        wsrc = cw_v, bsrc = cb_v, gc = n * V + c - 2 * K;
      }
      *reinterpret_cast<float4*>(cws + 4 * c) = *reinterpret_cast<const float4*>(wsrc + 4 * gc);
      cws[4 * CC + c] = bsrc ? bsrc[gc] : 0.f;
      for (int r = 0; r < 3; ++r) halo[r * CC + c] = 0;
    }
  }
  __syncthreads();
  if constexpr (CS > 1) cluster_sync_all();  // every block's barriers exist before remote arrives

  int issued = 0;  // chunks whose TMA load this thread has started (the TMA thread only)
  auto issue = [&](int cc) {
    const int st = cc % 3;
    uint8_t* base = smem + st * L.stage;
    mbar_arrive_expect_tx(&full[st], stage_tx);
    tma_load_4d(base + L.qs, &tm_q, &full[st], 0, n * qk_hs, cc * Tc, b);
    tma_load_4d(base + L.ks, &tm_k, &full[st], 0, n * qk_hs, cc * Tc, b);
    tma_load_4d(base + L.vs, &tm_v, &full[st], 0, n, cc * Tc, b);
    issued = cc + 1;
  };
  // Before leaving after a timeout the TMA thread lets the loads it started land (the last
  // three issued hold the three stages; earlier ones were consumed).
  auto drain = [&]() {
    for (int ci = issued > 3 ? issued - 3 : 0; ci < issued; ++ci)
      mbar_wait_bounded(&full[ci % 3], (uint32_t)(ci / 3) & 1u, kDebugWaitLimitCycles);
  };
  // Bounded wait that also gives up once another warp of the block has given up; on failure
  // this thread raises the block's abort flag and records the timeout.  `remote`: arrivals
  // may come from the other block of the cluster (acquire at cluster scope).
  // `sleep` (two-block clusters only): a warp that waits long (a helper waiting for the
  // compute warps) sleeps on the barrier instead of polling it, so it takes no issue slots
  // from its sub-partition.  One-block pairs keep polling helpers: the hot loop's schedule
  // depends on the code around it, and theirs is the one measured fastest.
  auto wait = [&](uint64_t* bar, uint32_t parity, bool remote = false,
                  bool sleep = false) -> bool {
    const bool ok =
        (CS > 1 && remote)
            ? (sleep ? mbar_wait_cluster_sleep(bar, parity, limit, abort_flag)
                     : mbar_wait_cluster(bar, parity, limit, abort_flag))
            : ((sleep && CS > 1) ? wait_or_abort_sleep(bar, parity, limit, abort_flag)
                     : wait_or_abort(bar, parity, limit, abort_flag));
    if (ok) return true;
    *abort_flag = 1;
    if (lane == 0) atomicExch(status, kStatusTimeout);
    return false;
  };
  // Arrive on a barrier of every block of the pair (release at cluster scope when CS > 1).
  auto arrive_all = [&](uint64_t* bar) {
    if constexpr (CS == 1) {
      mbar_arrive(bar);
    } else {
#pragma unroll
      for (int r = 0; r < CS; ++r) mbar_arrive_cluster(mapa_shared(smem_u32(bar), (uint32_t)r));
    }
  };

  // ---------------------------------------------------------------- staging helpers
  // Gate batch bt covers steps bt GB .. (bt + 1) GB - 1 (chunks bt G ..); participant i
  // computes batch step i into ring slot bt & 1.
  auto load_a = [&](int bt, int i) -> float {
    const int t = bt * GB + i;
    return (i < GB && t < T) ? bf16_bits_to_float(a[(row_base + t) * N + n]) : 0.f;
  };
  auto gate = [&](int bt, int i, float av) {
    if (i < GB) fgr[(bt & 1) * GB + i] = gate_fg(av, al, be);
  };
  // Chunk cc's v pairs and k (its TMA stage has landed) into operand buffer cc & 1; rows
  // i0, i0 + count, ... (participant i0 of `count`).
  auto convert = [&](int cc, int i0, int count) {
    const uint8_t* raw = smem + (cc % 3) * L.stage;
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(raw + L.vs);
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(raw + L.ks);
    uint8_t* cbase = smem + L.cb + (cc & 1) * L.cbuf;
    float4* vd = reinterpret_cast<float4*>(cbase + L.vd);
    float4* kf = reinterpret_cast<float4*>(cbase + L.kf);
    // One (step, g) row per pass: (v_j, v_j, v_j', v_j'), j = 16m + g, j' = j + 8.
    for (int e = i0; e < Tc * 8; e += count) {
      const uint16_t* vr = vs + (e >> 3) * V + (e & 7);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float v0 = bf16_bits_to_float(vr[16 * m]), v1 = bf16_bits_to_float(vr[16 * m + 8]);
        vd[(size_t)e * MT + m] = make_float4(v0, v0, v1, v1);
      }
    }
    for (int e = i0; e < Tc * K / 8; e += count) {  // eight k values per pass
      const uint4 u = reinterpret_cast<const uint4*>(ks)[e];
      kf[2 * e] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
      kf[2 * e + 1] = make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
    }
  };
  // Fused prologue for chunk cc (its TMA stage has landed): units (channel c of the 2K + V,
  // half hf of the chunk's steps), participants i0, i0 + count, ...; `sync` is a barrier over
  // the participants.  Phase A saves the raw rows other units still need (the first half's
  // last three, for the second half; the chunk's last three, for the next chunk), phase B
  // runs each unit's 16 steps in order with a three-step window, writing q and v back in
  // place and k, v into the operand buffer cc & 1 as fp32.
  auto convert_conv = [&](int cc, int i0, int count, auto sync) {
    constexpr int kHalf = Tc / 2;
    uint8_t* raw = smem + (cc % 3) * L.stage;
    uint16_t* qs = reinterpret_cast<uint16_t*>(raw + L.qs);
    uint16_t* ks = reinterpret_cast<uint16_t*>(raw + L.ks);
    uint16_t* vs = reinterpret_cast<uint16_t*>(raw + L.vs);
    const uint16_t* hal_in = halo + (cc & 1) * 3 * CC;
    uint16_t* hal_out = halo + ((cc + 1) & 1) * 3 * CC;
    uint8_t* cbase = smem + L.cb + (cc & 1) * L.cbuf;
    float4* vd = reinterpret_cast<float4*>(cbase + L.vd);
    float* kf = reinterpret_cast<float*>(cbase + L.kf);
    auto xat = [&](int c, int r) -> uint16_t {  // raw row r of channel c in the stage
      return c < K ? qs[r * K + c] : c < 2 * K ? ks[r * K + c - K] : vs[r * V + c - 2 * K];
    };
    for (int e = i0; e < 3 * CC; e += count) {
      const int r = e / CC, c = e - r * CC;
      mid[r * CC + c] = xat(c, kHalf - 3 + r);
      hal_out[r * CC + c] = xat(c, Tc - 3 + r);
    }
    sync();
    for (int e = i0; e < 2 * CC; e += count) {
      const int hf = e / CC, c = e - hf * CC;
      const uint16_t* win = hf == 0 ? hal_in : mid;
      float x3 = bf16_bits_to_float(win[c]), x2 = bf16_bits_to_float(win[CC + c]),
            x1 = bf16_bits_to_float(win[2 * CC + c]);
      const float* tap = cws + 4 * c;
      const float bias = cws[4 * CC + c];
      for (int r = hf * kHalf; r < (hf + 1) * kHalf; ++r) {
        const float x0 = bf16_bits_to_float(xat(c, r));
        const uint16_t o = r8_bf16_bits(r8_conv_silu(tap, bias, x3, x2, x1, x0));
        const float of = bf16_bits_to_float(o);
        if (c < K) {
          qs[r * K + c] = o;
        } else if (c < 2 * K) {
          kf[r * K + c - K] = of;
        } else {
          const int j = c - 2 * K;
          vs[r * V + j] = o;
          reinterpret_cast<float2*>(vd + (size_t)(r * 8 + (j & 7)) * MT + (j >> 4))[(j >> 3) & 1] =
              make_float2(of, of);
        }
        x3 = x2;
        x2 = x1;
        x1 = x0;
      }
    }
    sync();
  };
  // y of chunk cc (CS == 1): w_r ⊙ v plus the compute warps' partials in warp order, float4
  // rows; outputs i0, i0 + count, ...  The loop over warps is unrolled so that an output's
  // partial loads are in flight together.
  auto ysum = [&](int cc, int i0, int count) {
    const int steps = min(Tc, T - cc * Tc);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + (cc % 3) * L.stage + L.vs);
    const float* yp = ypart + (size_t)(cc & 1) * (L.ybuf / 4);
    constexpr int V4 = V / 4;
    for (int idx = i0; idx < steps * V4; idx += count) {
      const int s = idx / V4, j = (idx - s * V4) * 4;
      float4 u[8];
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (w < nw) u[w] = *reinterpret_cast<const float4*>(yp + ((size_t)w * Tc + s) * V + j);
      const uint2 vv = *reinterpret_cast<const uint2*>(vs + s * V + j);
      const float4 w4 = *reinterpret_cast<const float4*>(wrs + j);
      float4 o = make_float4(w4.x * bf16_lo(vv.x), w4.y * bf16_hi(vv.x), w4.z * bf16_lo(vv.y),
                             w4.w * bf16_hi(vv.y));
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (w < nw) {
          o.x += u[w].x;
          o.y += u[w].y;
          o.z += u[w].z;
          o.w += u[w].w;
        }
      *reinterpret_cast<float4*>(y + ((row_base + (size_t)cc * Tc + s) * N + n) * V + j) = o;
    }
  };
  // CS > 1, first half: this block's warps' partials of chunk cc summed in warp order, each
  // float4 of columns stored into its owner's exchange buffer (slot `rank`).
  auto xsum = [&](int cc, int i0, int count) {
    const int steps = min(Tc, T - cc * Tc);
    const float* yp = ypart + (size_t)(cc & 1) * (L.ybuf / 4);
    constexpr int V4 = V / 4;
    for (int idx = i0; idx < steps * V4; idx += count) {
      const int s = idx / V4, j = (idx - s * V4) * 4;
      float4 u[8];
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (w < nw) u[w] = *reinterpret_cast<const float4*>(yp + ((size_t)w * Tc + s) * V + j);
      float4 o = u[0];
#pragma unroll
      for (int w = 1; w < 8; ++w)
        if (w < nw) {
          o.x += u[w].x;
          o.y += u[w].y;
          o.z += u[w].z;
          o.w += u[w].w;
        }
      const int owner = j / VL;
      const uint32_t a = smem_u32(xpart + (size_t)(cc & 1) * (L.xbuf / 4) +
                                  ((size_t)rank * Tc + s) * VL + (j - owner * VL));
      st_cluster_v4_f32(mapa_shared(a, (uint32_t)owner), o);
    }
  };
  // CS > 1, second half: y of chunk cc for this block's columns: w_r ⊙ v plus the blocks' sums
  // in block order.
  auto ysum_x = [&](int cc, int i0, int count) {
    const int steps = min(Tc, T - cc * Tc);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + (cc % 3) * L.stage + L.vs);
    const float* xp = xpart + (size_t)(cc & 1) * (L.xbuf / 4);
    constexpr int V4 = VL / 4;
    for (int idx = i0; idx < steps * V4; idx += count) {
      const int s = idx / V4, jl = (idx - s * V4) * 4, j = rank * VL + jl;
      float4 u[CS];
#pragma unroll
      for (int r = 0; r < CS; ++r)
        u[r] = *reinterpret_cast<const float4*>(xp + ((size_t)r * Tc + s) * VL + jl);
      const uint2 vv = *reinterpret_cast<const uint2*>(vs + s * V + j);
      const float4 w4 = *reinterpret_cast<const float4*>(wrs + j);
      float4 o = make_float4(w4.x * bf16_lo(vv.x), w4.y * bf16_hi(vv.x), w4.z * bf16_lo(vv.y),
                             w4.w * bf16_hi(vv.y));
#pragma unroll
      for (int r = 0; r < CS; ++r) {
        o.x += u[r].x;
        o.y += u[r].y;
        o.z += u[r].z;
        o.w += u[r].w;
      }
      *reinterpret_cast<float4*>(y + ((row_base + (size_t)cc * Tc + s) * N + n) * V + j) = o;
    }
  };

  // ---------------------------------------------------------------- prologue (all threads)
  // Chunks 0, 1, 2 start loading; chunks 0 and 1 are converted and gate batch 0 computed by
  // every thread before the roles split.
  if (tid == tma_tid)
    for (int cc = 0; cc < 3 && cc < nchunks; ++cc) issue(cc);
  bool started;
  {
    const float a0 = load_a(0, tid);
    bool ok = mbar_wait_bounded(&full[0], 0u, limit);
    if (debug & kDebugForceTimeout) ok = ok && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
    if (nchunks > 1) ok = ok && mbar_wait_bounded(&full[1], 0u, limit);
    started = !__syncthreads_or(!ok);
    if (!started) {
      if (tid == 0) atomicExch(status, kStatusTimeout);
      if (tid == tma_tid) drain();
      if constexpr (CS == 1) return;  // (a cluster's blocks leave together, below)
    } else {
      if constexpr (kConv) {
        auto block_sync = [] { __syncthreads(); };
        convert_conv(0, tid, nthreads, block_sync);
        if (nchunks > 1) convert_conv(1, tid, nthreads, block_sync);
      } else {
        convert(0, tid, nthreads);
        if (nchunks > 1) convert(1, tid, nthreads);
      }
      gate(0, tid, a0);
    }
  }
  __syncthreads();

  // ================================================================ helper warps
  if ((CS == 1 || started) && warp >= nw) {
    const int hid = tid - tma_tid;  // 0 .. 127
    float a_nx = load_a(1, hid);    // logits of gate batch 1
    for (int cc = 0; cc < nchunks; ++cc) {
      bool ok = wait(&pdone[cc & 1], (uint32_t)(cc >> 1) & 1u, false, true);
      if constexpr (CS > 1)  // both owners have read what this block stored for chunk cc-2
        if (ok && cc >= 2) ok = wait(&xfree[cc & 1], (uint32_t)((cc - 2) >> 1) & 1u, true, true);
      if (named_bar_or(1, 32 * kR8Helpers, !ok)) break;
      if constexpr (CS == 1) {
        ysum(cc, hid, 32 * kR8Helpers);
        mbar_arrive(&ydone[cc & 1]);
      } else {
        xsum(cc, hid, 32 * kR8Helpers);
        mbar_arrive(&ydone[cc & 1]);
        arrive_all(&xready[cc & 1]);
        ok = wait(&xready[cc & 1], (uint32_t)(cc >> 1) & 1u, true, true);
        if (named_bar_or(4, 32 * kR8Helpers, !ok)) break;
        ysum_x(cc, hid, 32 * kR8Helpers);
        arrive_all(&xfree[cc & 1]);
      }
      if (cc + 3 < nchunks) {
        // Stage cc % 3 is free: every helper has read chunk cc's v, the compute warps its q.
        named_bar_sync(2, 32 * kR8Helpers);
        if (hid == 0) issue(cc + 3);
      }
      if (cc + 2 < nchunks) {
        const int nc = cc + 2;  // into operand buffer cc & 1, which chunk cc has released
        ok = wait(&full[nc % 3], (uint32_t)(nc / 3) & 1u, false, true);
        if (named_bar_or(3, 32 * kR8Helpers, !ok)) break;
        if constexpr (kConv)
          convert_conv(nc, hid, 32 * kR8Helpers, [] { named_bar_sync(5, 32 * kR8Helpers); });
        else
          convert(nc, hid, 32 * kR8Helpers);
        if (nc % G == 0) {  // the gate batch that starts with chunk nc
          gate(nc / G, hid, a_nx);
          a_nx = load_a(nc / G + 1, hid);
        }
        mbar_arrive(cready);
      }
    }
    if (hid == 0) drain();  // nothing is in flight unless the loop was left on a timeout
    if constexpr (CS == 1) return;
  }

  // ================================================================ compute warps
  if ((CS == 1 || started) && warp < nw) {
  const int g = lane >> 2, c = lane & 3;

  // W^T as m16n8k16 A fragments: wa[m][kt] covers rows j = 16m + g (+8) of W^T and columns
  // l = 16kt + 2c (+1, +8, +9), i.e. W[l][j].
  const uint16_t* Wn = W + (size_t)n * V * V;
  uint32_t wa[MT][MT][4];
#pragma unroll
  for (int kt = 0; kt < MT; ++kt)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const int l = 16 * kt + 2 * c, j = 16 * m + g;
      wa[m][kt][0] = (uint32_t)Wn[l * V + j] | ((uint32_t)Wn[(l + 1) * V + j] << 16);
      wa[m][kt][1] = (uint32_t)Wn[l * V + j + 8] | ((uint32_t)Wn[(l + 1) * V + j + 8] << 16);
      wa[m][kt][2] = (uint32_t)Wn[(l + 8) * V + j] | ((uint32_t)Wn[(l + 9) * V + j] << 16);
      wa[m][kt][3] = (uint32_t)Wn[(l + 8) * V + j + 8] | ((uint32_t)Wn[(l + 9) * V + j + 8] << 16);
    }

  // State (fp32) in the accumulator layout: h[m][hh] = (H[i0][j], H[i0 + 1][j]), j = 16m + 8hh + g.
  const int wg = nw * rank + warp;  // this warp's index among the pair's compute warps
  const int i0 = 8 * wg + 2 * c;
  float2 h[MT][2];
  if (H0) {
    const float* hp = H0 + (size_t)pair * K * V;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int j = 16 * m + 8 * hh + g;
        h[m][hh] = make_float2(hp[(size_t)i0 * V + j], hp[(size_t)(i0 + 1) * V + j]);
      }
  } else {
#pragma unroll
    for (int m = 0; m < MT; ++m) h[m][0] = h[m][1] = make_float2(0.f, 0.f);
  }

  // A step's shared-memory operands, loaded during the step before so that their latency
  // overlaps it: the gate and q of step t, and v, k of step t+1 (its rank-1 term).
  struct StepIn {
    float2 fg, kk;
    float4 v[MT];
    uint32_t qp;
  };
  // Shared-memory bases of chunk cc and of the chunk after it.
  struct ChunkPtrs {
    const uint8_t *cb0, *cb1;  // operand buffers
    const uint16_t *q0, *q1;   // raw q stages
    const float2 *fg0, *fg1;   // gates
  };
  auto chunk_ptrs = [&](int cc) {
    ChunkPtrs P;
    P.cb0 = smem + L.cb + (cc & 1) * L.cbuf;
    P.cb1 = smem + L.cb + ((cc + 1) & 1) * L.cbuf;
    P.q0 = reinterpret_cast<const uint16_t*>(smem + (cc % 3) * L.stage + L.qs);
    P.q1 = reinterpret_cast<const uint16_t*>(smem + ((cc + 1) % 3) * L.stage + L.qs);
    P.fg0 = fgr + ((cc / G) & 1) * GB + (cc % G) * Tc;
    P.fg1 = fgr + (((cc + 1) / G) & 1) * GB + ((cc + 1) % G) * Tc;
    return P;
  };
  // The operands of the step after step s: gate and q of step s + 1, v and k of step s + 2
  // (either may fall in the next chunk, whose operands are ready before they are read; past
  // the end of the sequence they are stale and never used).  Selects, not branches.
  auto fetch = [&](StepIn& in, const ChunkPtrs& P, int s, int steps) {
    const bool n1 = s + 1 >= steps, n2 = s + 2 >= steps;
    const int s1 = n1 ? s + 1 - steps : s + 1, s2 = n2 ? s + 2 - steps : s + 2;
    const uint8_t* c2 = n2 ? P.cb1 : P.cb0;
    in.fg = (n1 ? P.fg1 : P.fg0)[s1];
    in.qp = *reinterpret_cast<const uint32_t*>((n1 ? P.q1 : P.q0) + s1 * K + i0);
    in.kk = *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(c2 + L.kf) + s2 * K + i0);
    const float4* vp = reinterpret_cast<const float4*>(c2 + L.vd) + (size_t)(s2 * 8 + g) * MT;
#pragma unroll
    for (int m = 0; m < MT; ++m) in.v[m] = vp[m];
  };

  // P_0 = v_0 k_0^T + W^T H_0^T.
  float2 acc[MT][2], nxt[MT][2];
  StepIn in;
  {
    const ChunkPtrs P0 = chunk_ptrs(0);
    const float2 kk0 = *reinterpret_cast<const float2*>(
        reinterpret_cast<const float*>(P0.cb0 + L.kf) + i0);
    const float4* vp0 = reinterpret_cast<const float4*>(P0.cb0 + L.vd) + (size_t)g * MT;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float4 v4 = vp0[m];
      acc[m][0] = mul2(kk0, make_float2(v4.x, v4.y));
      acc[m][1] = mul2(kk0, make_float2(v4.z, v4.w));
    }
    fetch(in, P0, -1, min(Tc, T));  // step 0's operands
  }
#pragma unroll
  for (int kt = 0; kt < MT; ++kt) {
    const uint32_t b0 = movmatrix_trans(pack_bf16x2(h[kt][0].x, h[kt][0].y));
    const uint32_t b1 = movmatrix_trans(pack_bf16x2(h[kt][1].x, h[kt][1].y));
#pragma unroll
    for (int m = 0; m < MT; ++m) mma2(acc[m], wa[m][kt], b0, b1);
  }

  // One time step (step s).  On entry `cur` holds P_t (complete), h holds H_{t-1} and `in`
  // this step's operands; on exit h holds H_t, `nx` holds P_{t+1} (its last MMAs may be in
  // flight), `in` the next step's operands, and ap, qp the bf16 pack of H_t and q_t.
  auto step = [&](float2 (&cur)[MT][2], float2 (&nx)[MT][2], const ChunkPtrs& P, int s,
                  int steps, uint32_t (&ap)[MT][2], uint32_t& qp) {
    const StepIn cin = in;
    fetch(in, P, s, steps);
    qp = cin.qp;
    // Rank-1 term v_{t+1} k_{t+1}^T initialises P_{t+1}^T.
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      nx[m][0] = mul2(cin.kk, make_float2(cin.v[m].x, cin.v[m].y));
      nx[m][1] = mul2(cin.kk, make_float2(cin.v[m].z, cin.v[m].w));
    }
    const float2 ff = make_float2(cin.fg.x, cin.fg.x), gg = make_float2(cin.fg.y, cin.fg.y);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      // Eq. (10)-(11): Z = tanh(P), H = f H + (1 - f) Z, for column tile m.
      const float z0 = tanh_mufu(cur[m][0].x), z1 = tanh_mufu(cur[m][0].y);
      const float z2 = tanh_mufu(cur[m][1].x), z3 = tanh_mufu(cur[m][1].y);
      h[m][0] = fma2(gg, make_float2(z0, z1), mul2(ff, h[m][0]));
      h[m][1] = fma2(gg, make_float2(z2, z3), mul2(ff, h[m][1]));
      ap[m][0] = pack_bf16x2(h[m][0].x, h[m][0].y);
      ap[m][1] = pack_bf16x2(h[m][1].x, h[m][1].y);
      const uint32_t b0 = movmatrix_trans(ap[m][0]), b1 = movmatrix_trans(ap[m][1]);
#pragma unroll
      for (int m2 = 0; m2 < MT; ++m2) mma2(nx[m2], wa[m2][m], b0, b1);
    }
  };
  auto store_part = [&](float* yp, int s, int j, float val) {
    yp[((size_t)warp * Tc + s) * V + j] = val;
  };
  // Eq. (12) readout of steps s and s + 1 over this warp's rows, one m16n8k16 MMA per column
  // tile (see the header), into partial buffer yp; `two` is false for a lone last step.
  auto readout2 = [&](float* yp, const uint32_t (&apA)[MT][2], const uint32_t (&apB)[MT][2],
                      uint32_t qA, uint32_t qB, int s, bool two) {
    float d[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const uint32_t af[4] = {apA[m][0], apA[m][1], apB[m][0], apB[m][1]};
      mma_bf16_16816_z(d[m], af, g == 2 * m ? qA : 0u, g == 2 * m + 1 ? qB : 0u);
    }
    float2 lo = make_float2(d[0][0], d[0][1]), hi = make_float2(d[0][2], d[0][3]);
#pragma unroll
    for (int m = 1; m < MT; ++m) {
      lo = add2(lo, make_float2(d[m][0], d[m][1]));
      hi = add2(hi, make_float2(d[m][2], d[m][3]));
    }
    if (c < MT) {
      store_part(yp, s, 16 * c + g, lo.x);
      store_part(yp, s, 16 * c + 8 + g, hi.x);
      if (two) {
        store_part(yp, s + 1, 16 * c + g, lo.y);
        store_part(yp, s + 1, 16 * c + 8 + g, hi.y);
      }
    }
  };

  bool ok = true;
  for (int cc = 0; cc < nchunks && ok; ++cc) {
    const int steps = min(Tc, T - cc * Tc);
    const ChunkPtrs P = chunk_ptrs(cc);
    float* yp = ypart + (size_t)(cc & 1) * (L.ybuf / 4);
    // The partial buffer was last read by the helpers' sums of chunk cc-2.
    if (cc >= 2 && !wait(&ydone[cc & 1], (uint32_t)((cc - 2) >> 1) & 1u)) {
      ok = false;
      break;
    }
    // A chunk with a successor is whole; its last trip prefetches the successor's operands,
    // converted by the helpers (chunk 1's before the loop).  No wait otherwise.
    const int s_wait = (cc >= 1 && cc + 1 < nchunks) ? Tc - 2 : -1;
    auto trip = [&](int s) {
      uint32_t apA[MT][2], apB[MT][2], qA, qB;
      step(acc, nxt, P, s, steps, apA, qA);
      step(nxt, acc, P, s + 1, steps, apB, qB);
      readout2(yp, apA, apB, qA, qB, s, true);
    };
    int s = 0;
    for (; s + 1 < steps && s != s_wait; s += 2) trip(s);
    if (s == s_wait) {
      if (!wait(cready, (uint32_t)(cc - 1) & 1u)) {
        ok = false;
        break;
      }
      trip(s);
      s += 2;
    }
    if (s < steps) {  // odd tail of the last chunk
      uint32_t apA[MT][2], apB[MT][2], qA;
      step(acc, nxt, P, s, steps, apA, qA);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        apB[m][0] = apB[m][1] = 0u;
        acc[m][0] = nxt[m][0];
        acc[m][1] = nxt[m][1];
      }
      readout2(yp, apA, apB, qA, 0u, s, false);
    }
    mbar_arrive(&pdone[cc & 1]);
  }
  if constexpr (CS == 1)
    if (!ok) return;

  if (ok && H_T) {
    float* hp = H_T + (size_t)pair * K * V;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int j = 16 * m + 8 * hh + g;
        hp[(size_t)i0 * V + j] = h[m][hh].x;
        hp[(size_t)(i0 + 1) * V + j] = h[m][hh].y;
      }
  }
  }
  // Neither block of a cluster leaves while the other may still store to its shared memory
  // or arrive on its barriers.
  if constexpr (CS > 1) cluster_sync_all();
}

bool make_map_r8(EncodeTiledFn enc, CUtensorMap* map, const void* base, int inner, int N, int T,
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

template <int MT, int CS, bool kConv>
cudaError_t launch_r8(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  constexpr int V = 16 * MT;
  const R8Layout L = r8_layout(p.K, V, CS, kConv);
  CUtensorMap mq, mk, mv;
  if (!make_map_r8(enc, &mq, p.q, p.K, p.Nqk, p.T, p.B, kR8Tc) ||
      !make_map_r8(enc, &mk, p.k, p.K, p.Nqk, p.T, p.B, kR8Tc) ||
      !make_map_r8(enc, &mv, p.v, V, p.N, p.T, p.B, kR8Tc))
    return cudaErrorInvalidValue;
  auto kern = fwd_bf16_r8<MT, CS, kConv>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)CS * (unsigned)p.B * (unsigned)p.N, 1, 1);
  cfg.blockDim = dim3(32u * (unsigned)(p.K / 8 / CS + kR8Helpers), 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CS > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, (const uint16_t*)p.a, p.alpha, p.beta,
                            (const uint16_t*)p.W, p.w_r, p.H0, p.y, p.H_T, p.T, p.N, p.K,
                            p.Nqk == 1 ? 0 : 1, p.debug, p.status, p.conv.wq, p.conv.bq,
                            p.conv.wk, p.conv.bk, p.conv.wv, p.conv.bv);
}

template <int CS, bool kConv>
cudaError_t launch_r8_cs(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  switch (p.V) {
    case 16: return launch_r8<1, CS, kConv>(p, enc, stream);
    case 32: return launch_r8<2, CS, kConv>(p, enc, stream);
    case 48: return launch_r8<3, CS, kConv>(p, enc, stream);
    case 64: return launch_r8<4, CS, kConv>(p, enc, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool mma_r8_supports(int K, int V) {
  return (K == 32 || K == 64) && (V == 16 || V == 32 || V == 48 || V == 64);
}

bool mma_r8_cluster_supports(int K, int V) { return K == 64 && mma_r8_supports(K, V); }

cudaError_t launch_fwd_bf16_mma_r8(const Problem& p, EncodeTiledFn enc, cudaStream_t stream) {
  return p.conv.wq ? launch_r8_cs<1, true>(p, enc, stream) : launch_r8_cs<1, false>(p, enc, stream);
}

cudaError_t launch_fwd_bf16_mma_r8_cluster(const Problem& p, EncodeTiledFn enc,
                                           cudaStream_t stream) {
  return p.conv.wq ? launch_r8_cs<2, true>(p, enc, stream) : launch_r8_cs<2, false>(p, enc, stream);
}

}  // namespace m2rnn
