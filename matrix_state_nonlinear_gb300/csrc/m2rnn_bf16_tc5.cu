// m2rnn_bf16_tc5.cu — bf16-operand / fp32-state forward recurrence on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), for K = V = 128.
//
// The recurrence is Eq. (10)-(12) and (13)/(17) of the M²RNN study notes ("M²RNN:
// 矩阵状态非线性 RNN 的容量、表达力与系统代价", Sec. 2.1-2.2); the (batch, head) pair is
// the work unit (the notes' Sec. 2.6).  A thread block of 256 threads runs one pair at a
// time; two blocks share an SM.
//
// Per step t, with H_{t-1} in fp32 registers (thread = row i, half the columns):
//   * tensor memory holds D = H_{t-1} W + k_t v_t^T (128 lanes x 128 fp32 columns),
//     produced by one elected thread as 8 K=16 MMAs on the bf16 H tile and W^T tile
//     in shared memory, plus one K=16 MMA whose A column 0 is k_t and B column 0 is
//     v_t (the rank-1 write, Eq. (10), done by the tensor core);
//   * every thread loads its row of D in 32-column pieces (tcgen05.ld), applies the
//     MUFU tanh and the gate lerp H_t = f H_{t-1} + (1 - f) Z in fp32, and writes
//     the bf16 copy of H_t into the 128-byte-swizzled A tile;
//   * the readout y_t = H_t^T q_t (Eq. (12)) is also a tensor-core product: the same
//     A tile read M-major (M = value column j, K = row i) times a 16-row tile whose
//     row 0 is q_t gives y_t in tensor-memory column 0, lane j; w_r ⊙ v_t is added
//     in fp32 on the way out.  The recurrence batch and the readout batch are
//     committed to separate mbarriers, so step t+1's tanh starts as soon as D is
//     ready while the readout of step t is still running.
// The serial chain of one pair (MMA latency, then tanh of 16384 elements) leaves the
// tensor core or the MUFU idle half of the time; the two blocks of an SM fill each
// other's gaps.  q, k, v arrive in chunks by TMA; gates (f, 1 - f) are computed a chunk
// ahead.  Every wait is bounded; a timeout is decided jointly by the block (OR-reduction
// barrier), tensor memory is released and the block exits.
//
// Schedules.  With at most two pairs per SM every block runs one pair.  With more, a
// wave of whole pairs would leave the last wave partly idle, so the balanced schedule
// lays all pairs' steps end to end and gives each of 2 x SMs blocks an equal stretch; a
// pair cut by a stretch boundary runs its first steps at the start of the later stretch
// and its last steps at the end of the earlier one.  Rows and pairs are independent, so
// the bits are those of one block per pair.  The state H_s crosses between the two
// blocks through the pair's own y rows s .. s+127 (fp32), with a ready tag in row s+128 —
// rows that nothing writes before the taking block has read them — ordered by a release
// store and an acquire load at GPU scope.  The tag carries the launch's epoch (a host
// counter), so nothing needs clearing before the launch.  The block that hands a state
// over has the lower block index and runs those first steps before anything else: with
// blocks started in index order (as the GPU dispatches them) the wait for it ends even if
// not every block were resident at once, and a wait that still runs out is reported as a
// timeout, never a hang.
#include <atomic>
#include <cstring>

#include <cuda_bf16.h>

#include "m2rnn_internal.h"
#include "ptx_util.cuh"

namespace m2rnn {
namespace {

constexpr int kD = 128;        // K = V = 128
constexpr int kTc = 16;        // steps per input chunk
constexpr int kThreads = 256;  // 8 warps: lane quadrant (warp & 3) x column half (warp >> 2)
constexpr uint32_t kTmemCols = 256;  // D: columns 0..127; readout: columns 128..143

// Shared memory layout (bytes); swizzled tiles are 1024-byte aligned.
constexpr int kOffA = 0;                       // H_t bf16, K-major SW128: [2 K-blocks][128][128 B]
constexpr int kOffW = kOffA + 32768;           // W^T bf16, same layout (row j = column j of W)
constexpr int kOffAx = kOffW + 32768;          // rank-1 A: [128 rows x 16] no-swizzle core matrices
constexpr int kOffBx = kOffAx + 4096;          // rank-1 B: same layout
constexpr int kOffQ = kOffBx + 4096;           // readout B: q_t in row 0, [2 K-blocks][16][128 B]
constexpr int kOffIn = kOffQ + 4096;           // 2 stages x {q, k, v} [kTc][128] bf16
constexpr int kStageBytes = 3 * kTc * kD * 2;
constexpr int kOffFg = kOffIn + 2 * kStageBytes;  // float2 [2][kTc]
constexpr int kOffBar = kOffFg + 2 * kTc * 8;     // mma, full[2], never, read; tmem slot
constexpr int kSmemBytes = kOffBar + 64 + 1024;   // + slack to align the base to 1024

__device__ __forceinline__ uint32_t sw128_off(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}
__device__ __forceinline__ uint32_t core_off(int r, int k) {  // no-swizzle, K = 16
  return (uint32_t)((r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Handoff of a pair cut between two blocks (balanced schedule): the block that runs the
// pair's first steps leaves the fp32 state H_s (row i in y row s + i of the pair) and then
// a ready tag (y row s + K, columns 0-1) in the y rows of the pair's later part, which
// nothing else writes before the later block has read them.  The tag holds a fixed high
// word and the launch's epoch, so a tag left by an earlier launch is never taken as ready.
constexpr uint32_t kReadyMagic = 0x4d32524eu;
__device__ __forceinline__ float* handoff_row(float* y, size_t row_base, int s, int N, int n,
                                              int r) {
  return y + ((row_base + s + r) * N + n) * kD;
}
__device__ __forceinline__ void st_release_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// kBalanced = false: block b runs pair b whole (the stretch logic folds away).
// kCache: also keep every state, the bf16 A tile of H_t exactly as the next step's product
// reads it, by one TMA tensor store per step into Hs [B N, T, K, V] (the training forward).
// The store must have read the tile before the next step rewrites it: thread 0 waits for
// that, and the block meets once more per step.
template <bool kBalanced, bool kCache>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_bf16_tc5(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_h,
                 const uint16_t* __restrict__ a,
                 const float* __restrict__ alpha, const float* __restrict__ beta,
                 const uint16_t* __restrict__ W, const float* __restrict__ w_r, const float* H0,
                 float* y, float* H_T, int T, int N, int qk_hs, long long pairs,
                 long long line_per_block, uint32_t epoch, int debug,
                 int* status) {
  extern __shared__ uint8_t smem_raw[];
  // Round the dynamic shared-memory base up to 1024 bytes (128-byte swizzle atoms).
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qd = warp & 3, ch = warp >> 2;
  const int i = 32 * qd + lane;  // row of H owned by this thread
  const int c0 = 64 * ch;        // first of its 64 columns

  uint8_t* sA = smem + kOffA;
  uint8_t* sW = smem + kOffW;
  uint8_t* sAx = smem + kOffAx;
  uint8_t* sBx = smem + kOffBx;
  uint8_t* sQ = smem + kOffQ;
  float2* fgs = reinterpret_cast<float2*>(smem + kOffFg);
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = mma_bar + 1;  // [2]
  uint64_t* never = mma_bar + 3;
  uint64_t* read_bar = mma_bar + 4;  // readout batch of a step done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 5);
  auto stage = [&](int st, int which) {  // which: 0 q, 1 k, 2 v
    return reinterpret_cast<uint16_t*>(smem + kOffIn + st * kStageBytes + which * kTc * kD * 2);
  };

  // This block's stretch [s_line, e_line) of the line of all pairs' steps laid end to end.
  // Balanced launches number the stretches backwards, so that the block handing a pair's
  // state over (the later stretch) has the lower block index and starts no later than the
  // block that waits for it.
  const long long worker =
      kBalanced ? (long long)gridDim.x - 1 - blockIdx.x : (long long)blockIdx.x;
  const long long total = pairs * (long long)T;
  const long long s_line =
      kBalanced ? tc5_cut(worker * line_per_block, total, T) : worker * (long long)T;
  const long long e_line =
      kBalanced ? tc5_cut((worker + 1) * line_per_block, total, T) : s_line + T;

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if (kCache) prefetch_tensormap(&tm_h);
    mbar_init(mma_bar, 1);
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(never, 1);
    mbar_init(read_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  // Zero the rank-1 and readout tiles (only column / row 0 is rewritten each step).
  for (int e = tid; e < (3 * 4096) / 16; e += kThreads)
    reinterpret_cast<uint4*>(sAx)[e] = make_uint4(0u, 0u, 0u, 0u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + ((uint32_t)(32 * qd) << 16);

  const uint32_t idesc_main = umma_idesc_bf16(kD, kD, false);
  const uint32_t idesc_read = umma_idesc_bf16(kD, 16, true);
  // Descriptor bases; per K=16 step only the start-address field (bits 0..13, in
  // 16-byte units) advances by a compile-time offset.
  const uint64_t dA = umma_desc(smem_u32(sA), 16, 1024, 2);
  const uint64_t dW = umma_desc(smem_u32(sW), 16, 1024, 2);
  const uint64_t dAy = umma_desc(smem_u32(sA), 16384, 1024, 2);  // same tile, M-major view
  const uint64_t dQ = umma_desc(smem_u32(sQ), 16, 1024, 2);
  const uint64_t dAx = umma_desc(smem_u32(sAx), 128, 256, 0);
  const uint64_t dBx = umma_desc(smem_u32(sBx), 128, 256, 0);
  // Recurrence batch D = H W + k v^T (8 + 1 MMAs) -> mma_bar; then, when asked, the
  // readout batch y = H^T q (8 MMAs) -> read_bar.  Each barrier gets one commit per call.
  auto issue_mma = [&](bool recur, bool read) {
    tc_fence_after();
    if (recur) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        umma_bf16(tmem, dA + off, dW + off, idesc_main, kk);
      }
      umma_bf16(tmem, dAx, dBx, idesc_main, 1);
    }
    umma_commit(mma_bar);
    if (read) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16(tmem + 128, dAy + (uint64_t)((kk * 2048) >> 4),
                  dQ + (uint64_t)(((kk >> 2) * 2048 + (kk & 3) * 32) >> 4), idesc_read, kk);
      umma_commit(read_bar);
    }
  };

  // Phases consumed so far on each barrier, over all of the block's segments.
  uint32_t mma_ph = 0, read_ph = 0, chunk_base = 0;
  bool abort = false, first_wait = true;
  float2 h[32];

  // Segments in the block's order: the first steps of a pair that another block finishes
  // (state handed off), whole pairs, then the last steps of a pair that another block
  // started (state taken over).  Each step of each pair is run by exactly one block.
  for (long long p = kBalanced ? s_line / T : worker;
       kBalanced ? (!abort && p * (long long)T < e_line) : p == worker; ++p) {
    const long long lo = kBalanced ? (s_line > p * T ? s_line : p * T) - p * T : 0;
    const long long hi = kBalanced ? (e_line < (p + 1) * T ? e_line : (p + 1) * T) - p * T : T;
    const bool to_handoff = lo > 0;      // the line's [lo, T) is this pair's first T - lo steps
    const bool from_handoff = hi < T;    // the line's [0, hi) is this pair's last hi steps
    const int t0 = from_handoff ? T - (int)hi : 0;
    const int t1 = to_handoff ? T - (int)lo : T;
    const int b = (int)(p / N), n = (int)(p - (long long)b * N);
    const size_t row_base = (size_t)b * T;
    const int nsteps = t1 - t0;
    const int nchunks = (nsteps + kTc - 1) / kTc;
    const float al = alpha[n], be = beta[n];
    const float wr_i = w_r[(size_t)n * kD + i];

    // TMA of the segment's chunk cc (one thread) and its gates (threads 0 .. kTc-1).
    auto issue_chunk = [&](int cc) {
      const int st = (int)((chunk_base + cc) & 1);
      mbar_arrive_expect_tx(&full[st], 3u * kTc * kD * 2u);
      tma_load_4d(stage(st, 0), &tm_q, &full[st], 0, n * qk_hs, t0 + cc * kTc, b);
      tma_load_4d(stage(st, 1), &tm_k, &full[st], 0, n * qk_hs, t0 + cc * kTc, b);
      tma_load_4d(stage(st, 2), &tm_v, &full[st], 0, n, t0 + cc * kTc, b);
    };
    auto chunk_gates = [&](int cc) {
      if (tid < kTc) {
        const int t = t0 + cc * kTc + tid;
        const float av = t < t1 ? bf16_bits_to_float(a[(row_base + t) * N + n]) : 0.f;
        fgs[((chunk_base + cc) & 1) * kTc + tid] = gate_fg(av, al, be);
      }
    };
    auto full_parity = [&](int cc) { return (uint32_t)((chunk_base + cc) >> 1) & 1u; };
    auto full_stage = [&](int cc) { return (int)((chunk_base + cc) & 1); };

    // W^T tile: row j, K index l holds W[l][j].
    const uint16_t* Wn = W + (size_t)n * kD * kD;
    for (int e = tid; e < kD * kD; e += kThreads) {
      const int l = e >> 7, j = e & 127;
      *reinterpret_cast<uint16_t*>(sW + sw128_off(j, l, kD)) = Wn[e];
    }
    if (tid == 0) {
      issue_chunk(0);
      if (nchunks > 1) issue_chunk(1);
    }
    chunk_gates(0);
    if (nchunks > 1) chunk_gates(1);
    // Initial state (fp32 registers): H_0, zeros, or the state another block handed off.
    bool ok = true;
    if (from_handoff) {
      if (tid == 0) {
        const unsigned long long* ready = reinterpret_cast<const unsigned long long*>(
            handoff_row(y, row_base, t0, N, n, kD));
        const unsigned long long tag = ((unsigned long long)kReadyMagic << 32) | epoch;
        const long long limit = kWaitLimitCycles + (long long)T * 8192;
        const long long c_start = clock64();
        while (ld_acquire_gpu(ready) != tag) {
          if (clock64() - c_start > limit) {
            ok = false;
            break;
          }
          __nanosleep(2000);
        }
      }
      ok = __syncthreads_and(ok);
      if (ok) {
        const float* hp = handoff_row(y, row_base, t0, N, n, i) + c0;
#pragma unroll
        for (int u = 0; u < 32; ++u) h[u] = __ldcg(reinterpret_cast<const float2*>(hp + 2 * u));
      }
    } else {
      const float* hp = H0 ? H0 + ((size_t)p * kD + i) * kD + c0 : nullptr;
#pragma unroll
      for (int u = 0; u < 32; ++u)
        h[u] = hp ? *reinterpret_cast<const float2*>(hp + 2 * u) : make_float2(0.f, 0.f);
    }
    auto store_a_tile = [&](int blk) {  // columns c0 + 16 blk .. +15 of row i, two 16-byte chunks
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int u = 8 * blk + 4 * hh;
        const uint4 v = make_uint4(pack_bf16x2(h[u].x, h[u].y), pack_bf16x2(h[u + 1].x, h[u + 1].y),
                                   pack_bf16x2(h[u + 2].x, h[u + 2].y),
                                   pack_bf16x2(h[u + 3].x, h[u + 3].y));
        *reinterpret_cast<uint4*>(sA + sw128_off(i, c0 + 16 * blk + 8 * hh, kD)) = v;
      }
    };
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) store_a_tile(blk);

    ok = ok && mbar_wait_bounded(&full[full_stage(0)], full_parity(0), kWaitLimitCycles);
    if (first_wait && (debug & kDebugForceTimeout))
      ok = ok && mbar_wait_bounded(never, 0u, kDebugWaitLimitCycles);
    first_wait = false;
    // Rank-1 operands of the first step: k in A column 0 (column-half 0), v in B column 0.
    if (ok) {
      const int st0 = full_stage(0);
      const uint16_t kv = ch == 0 ? stage(st0, 1)[i] : stage(st0, 2)[i];
      *reinterpret_cast<uint16_t*>((ch == 0 ? sAx : sBx) + core_off(i, 0)) = kv;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    abort = __syncthreads_or(!ok);
    if (!abort && tid == 0) issue_mma(true, false);

    float v_prev = 0.f;  // v_{t-1}[i] for the readout's residual term
    for (int t = t0; t < t1 && !abort; ++t) {
      const int ls = t - t0, cc = ls / kTc, s = ls - cc * kTc, st = full_stage(cc);
      if (s == 0 && cc >= 1) {  // the other stage was last read in chunk cc-1: refill it
        if (tid == 0 && cc + 1 < nchunks) issue_chunk(cc + 1);
        if (cc + 1 < nchunks) chunk_gates(cc + 1);
      }
      ok = mbar_wait_bounded(mma_bar, mma_ph & 1u, kWaitLimitCycles);
      ++mma_ph;
      if (kCache && t > t0) {
        // The A tile is rewritten below: the store of H_{t-1} must have read it.
        if (tid == 0) bulk_wait_group_read<0>();
        __syncthreads();
      }
      tc_fence_after();
      const float2 fg = fgs[st * kTc + s];
      const float2 ff = make_float2(fg.x, fg.x), gg = make_float2(fg.y, fg.y);
      // H_t = f H_{t-1} + (1 - f) tanh(D), 32 columns per tensor-memory wait.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float pv[32];
        tmem_ld16_nowait(t_lane + c0 + 32 * half, pv);
        tmem_ld16_nowait(t_lane + c0 + 32 * half + 16, pv + 16);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float2 z = make_float2(tanh_mufu(pv[2 * u]), tanh_mufu(pv[2 * u + 1]));
          h[16 * half + u] = fma2(gg, z, mul2(ff, h[16 * half + u]));  // Eq. (11)
        }
        if (half == 0 && t > t0) {
          // The readout batch of step t-1 reads the A tile and the q tile that this
          // step rewrites: wait for it, then emit y_{t-1} (column-half 0 lanes j = i).
          ok = ok && mbar_wait_bounded(read_bar, read_ph & 1u, kWaitLimitCycles);
          ++read_ph;
          tc_fence_after();
          if (ch == 0) {
            const float yv = tmem_ld1(t_lane + 128);
            y[((row_base + t - 1) * N + n) * kD + i] = fmaf(wr_i, v_prev, yv);
          }
        }
        store_a_tile(2 * half);
        store_a_tile(2 * half + 1);
      }
      // q_t (readout), and v_t kept for its residual; k_{t+1}, v_{t+1} (next rank-1).
      if (ch == 0) {
        const uint16_t qv = stage(st, 0)[s * kD + i];
        *reinterpret_cast<uint16_t*>(sQ + sw128_off(0, i, 16)) = qv;
        v_prev = bf16_bits_to_float(stage(st, 2)[s * kD + i]);
      }
      const bool has_next = t + 1 < t1;
      if (has_next) {
        const int ln = ls + 1, ccn = ln / kTc, sn = ln - ccn * kTc;
        if (sn == 0)
          ok = ok && mbar_wait_bounded(&full[full_stage(ccn)], full_parity(ccn), kWaitLimitCycles);
        if (ok) {
          const int stn = full_stage(ccn);
          const uint16_t kv = ch == 0 ? stage(stn, 1)[sn * kD + i] : stage(stn, 2)[sn * kD + i];
          *reinterpret_cast<uint16_t*>((ch == 0 ? sAx : sBx) + core_off(i, 0)) = kv;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      abort = __syncthreads_or(!ok);
      if (!abort && tid == 0) {
        issue_mma(has_next, true);
        if (kCache) {  // H_t (bf16, the A tile) into Hs[pair][t]: two 64-column boxes
          tma_store_4d_if(true, &tm_h, smem_u32(sA), 0, 0, t, (int)p);
          tma_store_4d_if(true, &tm_h, smem_u32(sA) + 16384, 64, 0, t, (int)p);
          bulk_commit_group();
        }
      }
    }
    if (abort) break;

    // Readout of the segment's last step; the empty recurrence commit of that step.
    bool ok2 = mbar_wait_bounded(read_bar, read_ph & 1u, kWaitLimitCycles);
    ++read_ph;
    ok2 = mbar_wait_bounded(mma_bar, mma_ph & 1u, kWaitLimitCycles) && ok2;
    ++mma_ph;
    tc_fence_after();
    if (ok2 && ch == 0) {
      const float yv = tmem_ld1(t_lane + 128);
      y[((row_base + t1 - 1) * N + n) * kD + i] = fmaf(wr_i, v_prev, yv);
    }
    if (to_handoff) {
      // State after step t1 - 1 into the later block's y rows, then its ready word.
      float* hp = handoff_row(y, row_base, t1, N, n, i) + c0;
#pragma unroll
      for (int u = 0; u < 32; ++u) __stcg(reinterpret_cast<float2*>(hp + 2 * u), h[u]);
      __syncthreads();
      if (tid == 0 && ok2) {
        __threadfence();
        st_release_gpu(
            reinterpret_cast<unsigned long long*>(handoff_row(y, row_base, t1, N, n, kD)),
            ((unsigned long long)kReadyMagic << 32) | epoch);
      }
    } else if (H_T) {
      float* hp = H_T + ((size_t)p * kD + i) * kD + c0;
#pragma unroll
      for (int u = 0; u < 32; ++u) *reinterpret_cast<float2*>(hp + 2 * u) = h[u];
    }
    chunk_base += (uint32_t)nchunks;
    // The next segment rewrites the A tile: the store of this segment's last state must
    // have read it.
    if (kCache && tid == 0) bulk_wait_group_read<0>();
    abort = __syncthreads_or(!ok2);
  }

  if (abort) {
    if (tid == 0) {
      atomicExch(status, kStatusTimeout);
      // Give a tensor-core batch or TMA copy still in flight a bounded chance to finish.
      mbar_wait_bounded(mma_bar, 0u, kDebugWaitLimitCycles);
      mbar_wait_bounded(mma_bar, 1u, kDebugWaitLimitCycles);
      mbar_wait_bounded(read_bar, 0u, kDebugWaitLimitCycles);
      mbar_wait_bounded(read_bar, 1u, kDebugWaitLimitCycles);
      for (int ci = 0; ci < 2; ++ci) {
        mbar_wait_bounded(&full[ci], 0u, kDebugWaitLimitCycles);
        mbar_wait_bounded(&full[ci], 1u, kDebugWaitLimitCycles);
      }
    }
  }
  if (kCache && tid == 0) bulk_wait_group<0>();  // the kept states are written
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

bool make_map_tc5(EncodeTiledFn enc, CUtensorMap* map, const void* base, int N, int T, int B) {
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * 2 * N,
                                 (cuuint64_t)kD * 2 * N * T};
  const cuuint32_t box[4] = {(cuuint32_t)kD, 1u, (cuuint32_t)kTc, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc5_supports(int K, int V) { return K == kD && V == kD; }

cudaError_t launch_fwd_bf16_tc5(const Problem& p, EncodeTiledFn enc, cudaStream_t stream,
                               bool balanced) {
  CUtensorMap mq, mk, mv, mh;
  if (!make_map_tc5(enc, &mq, p.q, p.Nqk, p.T, p.B) ||
      !make_map_tc5(enc, &mk, p.k, p.Nqk, p.T, p.B) ||
      !make_map_tc5(enc, &mv, p.v, p.N, p.T, p.B))
    return cudaErrorInvalidValue;
  const bool cache = p.Hs != nullptr;
  std::memset(&mh, 0, sizeof(mh));
  if (cache) {
    // Kept states [B N, T, K, V] bf16: a box of 64 columns x 128 rows of one step, with the
    // 128-byte swizzle of the A tile.
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kD, (cuuint64_t)p.T,
                                (cuuint64_t)p.B * p.N};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * kD * 2,
                                   (cuuint64_t)kD * kD * 2 * p.T};
    const cuuint32_t box[4] = {64u, (cuuint32_t)kD, 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    if (enc(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.Hs, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const long long pairs = (long long)p.B * p.N;
  const int qk_hs = p.Nqk == 1 ? 0 : 1;
  long long workers = pairs;
  if (balanced) {
    // Two blocks per SM: what the tensor memory (256 columns each) and shared memory allow.
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return err;
    workers = tc5_balanced_workers(pairs, 2LL * sms);
  }
  const bool bal = workers < pairs;
  static std::atomic<uint32_t> epochs{0};
  const uint32_t epoch = bal ? epochs.fetch_add(1, std::memory_order_relaxed) + 1 : 0u;
  const long long line = bal ? tc5_line_per_block(pairs, p.T, workers) : (long long)p.T;
  auto kern = bal ? (cache ? fwd_bf16_tc5<true, true> : fwd_bf16_tc5<true, false>)
                  : (cache ? fwd_bf16_tc5<false, true> : fwd_bf16_tc5<false, false>);
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  // Balanced: one block per stretch (blocks numbered backwards over the stretches, see the
  // kernel); otherwise one block per pair.
  kern<<<(unsigned)workers, kThreads, kSmemBytes, stream>>>(
      mq, mk, mv, mh, (const uint16_t*)p.a, p.alpha, p.beta, (const uint16_t*)p.W, p.w_r, p.H0,
      p.y, p.H_T, p.T, p.N, qk_hs, pairs, line, epoch, p.debug, p.status);
  return cudaGetLastError();
}

}  // namespace m2rnn
