// attn_fwd_fp8.cu -- exact-attention forward with 8-bit (e4m3) Q, K and V on
// the fifth-generation tensor core (tcgen05.mma kind::f8f6f4).
//
// "Training Transformers and Hybrid models on AMD Instinct MI300X
// Accelerators" (section "Summary") names extending its attention kernel to
// fp8 as the next step.  This is that forward for GB300: the caller stores Q,
// K, V as e4m3 bytes with one fp32 descale factor per tensor (the real value
// is byte value x descale), and the kernel computes
//
//   S = (s qd kd) Q8 K8^T,   O = softmax(S) (vd V8),   L = logsumexp(S)
//
// with both contractions in fp8 and fp32 accumulation.  P is quantised to
// e4m3 for P V; the row sums and L use the unquantised fp32 probabilities.
//
// Design: the bf16 forward's (attn_fwd.cu) -- CTAs taking tasks of two
// 128-row query tiles of one head in turn (heaviest first under the causal
// mask; the grid from fwd_grid), K/V tiles streaming through a two-stage TMA
// ring that runs on across a CTA's tasks, warps 0-3 and 4-7 running the
// softmax of the two tiles, warp 8 issuing TMA, warp 9 issuing tcgen05.mma --
// with 8-bit operands: a 128 x 128 e4m3 tile is one
// 128-byte-swizzled block of 16 KB (head dim 128 only), an MMA takes K = 32,
// and P goes to tensor memory four e4m3 values per 32-bit column.  The row
// maximum is exact (no lazy threshold): P is formed as 2^(x - m + 8), at most
// 256, so that e4m3's normal range (down to 2^-6) covers probabilities down
// to 2^-14 of the row maximum.

#include "f32x2.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace fwd8 {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int HD = 128;           // head dim (bytes per e4m3 row)
constexpr int kTileBytes = 128 * HD;  // one 128-row e4m3 tile: 16 KB
constexpr float kPShift = 8.f;    // P = 2^(x - m + 8) <= 256

constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;
constexpr int kBarKFull = 2;                       // + stage
constexpr int kBarKEmpty = kBarKFull + kStages;    // + stage
constexpr int kBarVFull = kBarKEmpty + kStages;    // + stage
constexpr int kBarVEmpty = kBarVFull + kStages;    // + stage
constexpr int kBarSFull = kBarVEmpty + kStages;    // + tile
constexpr int kBarPReady = kBarSFull + 2;          // + tile
constexpr int kBarOFull = kBarPReady + 2;          // + tile
constexpr int kBarDrain = kBarOFull + 2;
constexpr int kNumBars = kBarDrain + 1;

struct Layout {
  static constexpr int kQ = 0;                       // two query tiles
  static constexpr int kK = kQ + 2 * kTileBytes;     // kStages key tiles
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  // Padded past half of the SM's shared memory: one CTA (owning all 512
  // tensor-memory columns) per SM.
  static constexpr int kRaw = (kAbort + 4 + 15) / 16 * 16;
  static constexpr int kBytes = kRaw > 118784 ? kRaw : 118784;
  static constexpr uint32_t kColO = 0;         // + tile * HD
  static constexpr uint32_t kColS = 2 * HD;    // + tile * 128
};

// Descriptors (128-byte swizzle, one 16 KB block per tile: 128 rows of 128
// bytes): a K-major operand advances 32 bytes (32 e4m3 values) per k-step;
// the MN-major V advances 4 KB (32 rows) per k-step.

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                        float* __restrict__ Lout, int BH, int N, float score_log2, float v_descale,
                        int* err) {
  using Ly = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(err, kDevSmemAlign, 0x400);
    return;
  }

  const int n_tiles = (N + 127) >> 7;
  const int n_pairs = (n_tiles + 1) >> 1;
  const int n_tasks = BH * n_pairs;
  const int G = int(gridDim.x), cta = int(blockIdx.x);
  // Task i: query tiles 2 pair and 2 pair + 1 of head bh against key/value
  // tiles 0 .. n_kv - 1; causal tasks heaviest first, heads interleaved,
  // else head by head.
  struct Task {
    int bh, qt_a, n_kv;
    bool has_b;
  };
  auto task = [&](int i) {
    Task t;
    t.bh = CAUSAL ? i % BH : i / n_pairs;
    t.qt_a = 2 * (CAUSAL ? n_pairs - 1 - i / BH : i % n_pairs);
    t.has_b = t.qt_a + 1 < n_tiles;
    t.n_kv = CAUSAL ? min(n_tiles, t.qt_a + (t.has_b ? 2 : 1)) : n_tiles;
    return t;
  };
  // CTA b of G takes tasks b, 2G-1-b, 2G+b, ... (a snake over rounds); -1 past the end
  auto snake = [&](int k) {
    const long long idx = (k & 1) ? (long long)k * G + (G - 1 - cta) : (long long)k * G + cta;
    return idx < n_tasks ? int(idx) : -1;
  };

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), (i == kBarPReady || i == kBarPReady + 1) ? 128 : 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtx ctx{abort_flag, err, kWaitLimitNs};
  grid_dep_wait();
  grid_dep_launch();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    // g counts key/value tiles across tasks; the query tiles of a task load
    // once the previous task's last S has completed.
    bool ok = true;
    int g = 0;
    for (int k = 0, i = snake(0); ok && i >= 0; i = snake(++k)) {
      const Task tk = task(i);
      if (k > 0 && !(ok = mbar_wait_warp(bar(kBarQEmpty), (k - 1) & 1, ctx, 0x412))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarQFull), (tk.has_b ? 2 : 1) * kTileBytes);
        for (int t = 0; t < (tk.has_b ? 2 : 1); ++t)
          tma_load_3d(sbase + Ly::kQ + t * kTileBytes, &tmQ, bar(kBarQFull), 0,
                      (tk.qt_a + t) * 128, tk.bh);
      }
      __syncwarp();
      for (int j = 0; j < tk.n_kv; ++j, ++g) {
        const int s = g % kStages, n = g / kStages;
        if (g >= kStages && !(ok = mbar_wait_warp(bar(kBarKEmpty + s), (n - 1) & 1, ctx, 0x410)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(kBarKFull + s), kTileBytes);
          tma_load_3d(sbase + Ly::kK + s * kTileBytes, &tmK, bar(kBarKFull + s), 0, j * 128,
                      tk.bh);
        }
        __syncwarp();
        if (g >= kStages && !(ok = mbar_wait_warp(bar(kBarVEmpty + s), (n - 1) & 1, ctx, 0x411)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(kBarVFull + s), kTileBytes);
          tma_load_3d(sbase + Ly::kV + s * kTileBytes, &tmV, bar(kBarVFull + s), 0, j * 128,
                      tk.bh);
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = make_idesc_e4m3(128, 128, 0, 0);  // S = Q K^T
    constexpr uint32_t kIdO = make_idesc_e4m3(128, HD, 0, 1);   // O += P V, V MN-major
    auto issue_s = [&](int t, int stage) {  // elected lane only
      const uint64_t dq = make_sdesc_sw128(sbase + Ly::kQ + t * kTileBytes, 16, 1024);
      const uint64_t dk = make_sdesc_sw128(sbase + Ly::kK + stage * kTileBytes, 16, 1024);
      const uint32_t d = tbase + Ly::kColS + 128 * t;
#pragma unroll
      for (int k = 0; k < HD / 32; ++k)
        mma_ss_f8(d, sdesc_add(dq, k * 32), sdesc_add(dk, k * 32), kIdS, k > 0 ? 1u : 0u);
      tc_commit(bar(kBarSFull + t));
    };
    auto issue_pv = [&](int t, int stage, uint32_t acc) {  // elected lane only
      const uint64_t dv = make_sdesc_sw128(sbase + Ly::kV + stage * kTileBytes, 16384, 1024);
      const uint32_t d = tbase + Ly::kColO + HD * t;
      const uint32_t p = tbase + Ly::kColS + 128 * t;
#pragma unroll
      for (int k = 0; k < 4; ++k)  // 128 keys, 32 per step; P packed 4 per column
        mma_ts_f8(d, p + 8 * k, sdesc_add(dv, k * 4096), kIdO, k > 0 ? 1u : acc);
    };
    // Handshake counts across tasks: g key/value tiles, ca (cb) S/P rounds of
    // tile A (B).  A task's first P V overwrites O_t, which the softmax warps
    // of tile t have read before they signal the first P of this task; the
    // tensor core runs this thread's instructions in issue order, so an S
    // written over P columns comes after the P V that reads them.
    bool ok = true;
    int g = 0, ca = 0, cb = 0;
    for (int k = 0, i = snake(0); ok && i >= 0; i = snake(++k)) {
      const Task tk = task(i);
      const int n_kv = tk.n_kv;
      if (!(ok = mbar_wait_warp(bar(kBarQFull), k & 1, ctx, 0x420))) break;
      if (!(ok = mbar_wait_warp(bar(kBarKFull + g % kStages), (g / kStages) & 1, ctx, 0x421)))
        break;
      tc_fence_after();
      if (elect_one()) {
        issue_s(0, g % kStages);
        if (tk.has_b) issue_s(1, g % kStages);
        if (n_kv == 1) tc_commit(bar(kBarQEmpty));  // the task's last S
        tc_commit(bar(kBarKEmpty + g % kStages));
      }
      __syncwarp();
      for (int j = 0; j < n_kv; ++j, ++g) {
        const int s = g % kStages;
        const bool next = j + 1 < n_kv;
        const int s1 = (g + 1) % kStages, n1 = (g + 1) / kStages;
        const uint32_t acc = j > 0 ? 1u : 0u;
        if (!(ok = mbar_wait_warp(bar(kBarVFull + s), (g / kStages) & 1, ctx, 0x422))) break;
        if (!(ok = mbar_wait_warp(bar(kBarPReady + 0), (ca + j) & 1, ctx, 0x423))) break;
        tc_fence_after();
        if (elect_one()) issue_pv(0, s, acc);
        __syncwarp();
        if (next) {
          if (!(ok = mbar_wait_warp(bar(kBarKFull + s1), n1 & 1, ctx, 0x424))) break;
          tc_fence_after();
          if (elect_one()) issue_s(0, s1);
          __syncwarp();
        }
        if (tk.has_b) {
          if (!(ok = mbar_wait_warp(bar(kBarPReady + 1), (cb + j) & 1, ctx, 0x425))) break;
          tc_fence_after();
          if (elect_one()) {
            issue_pv(1, s, acc);
            if (next) issue_s(1, s1);
          }
          __syncwarp();
        }
        if (elect_one()) {
          if (j + 2 == n_kv) tc_commit(bar(kBarQEmpty));  // the task's last S was issued above
          tc_commit(bar(kBarVEmpty + s));
          if (next) tc_commit(bar(kBarKEmpty + s1));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) {
        tc_commit(bar(kBarOFull + 0));
        if (tk.has_b) tc_commit(bar(kBarOFull + 1));
      }
      __syncwarp();
      ca += n_kv;
      if (tk.has_b) cb += n_kv;
    }
    if (elect_one()) tc_commit(bar(kBarDrain));
    __syncwarp();
    volatile int never = 0;  // this wait ignores the CTA abort flag
    const WaitCtx own{&never, err, kWaitLimitNs};
    mbar_wait_warp(bar(kBarDrain), 0, own, 0x42F);
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;  // 0 = tile A, 1 = tile B
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + Ly::kColS + 128 * t;
    const uint32_t tO = tbase + lane_off + Ly::kColO + HD * t;
    bool ok = true;
    int cs = 0;  // S/P rounds of this tile so far
    int no = 0;  // outputs of this tile so far
    for (int k = 0, i = snake(0); ok && i >= 0; i = snake(++k)) {
      const Task tk = task(i);
      if (t == 1 && !tk.has_b) continue;
      const int bh = tk.bh, n_kv = tk.n_kv;
      const int q_tile0 = (tk.qt_a + t) * 128;
      const int q = q_tile0 + r;
      float m = -INFINITY;  // running (exact) max of the base-2 scaled scores
      float l = 0.f;        // running sum of 2^(x - m + 8), unquantised
      for (int j = 0; j < n_kv; ++j) {
        if (!(ok = mbar_wait_warp(bar(kBarSFull + t), (cs + j) & 1, ctx, 0x430 + t))) break;
        tc_fence_after();
        uint32_t u[128];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&u[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&u[96]));
        tmem_wait_ld();
        const int kv0 = j * 128;
        if ((CAUSAL && kv0 + 127 > q_tile0) || kv0 + 128 > N) {
          const int e_hi = min(CAUSAL ? q - kv0 : 127, N - 1 - kv0);  // last visible column
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > e_hi) u[c] = __float_as_uint(-INFINITY);
        }
        // row maximum: eight chains of three-input maxima (two scores each)
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(u[e]);
#pragma unroll
        for (int e = 8; e < 128; e += 2)
          m8[(e >> 1) & 7] =
              max3f(m8[(e >> 1) & 7], __uint_as_float(u[e]), __uint_as_float(u[e + 1]));
        const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                               fmaxf(m8[6], m8[7]));
        const float m_new = fmaxf(m, mx * score_log2);  // score_log2 > 0
        const bool rescale = m_new > m;
        const float alpha = rescale ? ex2(m - m_new) : 1.f;
        if (rescale) {
          l *= alpha;
          m = m_new;
        }
        // every row has its diagonal (or a first key) visible, so m is finite
        // once a visible key has been seen; before that, all P are 0
        const float mb = (m == -INFINITY) ? 0.f : m - kPShift;
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) {
          // s score_log2 - mb, two scores per instruction
          float x0, x1, x2, x3;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(u[4 * c4]), __uint_as_float(u[4 * c4 + 1])),
                                f32x2(score_log2, score_log2), f32x2(-mb, -mb)),
                      x0, x1);
          f32x2_split(
              fma_f32x2(f32x2(__uint_as_float(u[4 * c4 + 2]), __uint_as_float(u[4 * c4 + 3])),
                        f32x2(score_log2, score_log2), f32x2(-mb, -mb)),
              x2, x3);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          rs[c4 & 3] += (p0 + p1) + (p2 + p3);
          pk[c4] = pack_e4m3x4(p0, p1, p2, p3);
        }
        tmem_st32(tS, pk);
        l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        // O holds P V of earlier tiles (PV(j-1) has completed: its P columns
        // were free for this S).  tcgen05.ld/st are warp-collective, so if any
        // row of the warp moved its maximum the whole warp rescales.
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c4, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(tO + 32 * c4, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarPReady + t));
      }
      if (!ok) break;
      cs += n_kv;
      if (!(ok = mbar_wait_warp(bar(kBarOFull + t), no & 1, ctx, 0x438 + t))) break;
      ++no;
      {
        tc_fence_after();
        const float mult = v_descale / l;
        __nv_bfloat16* orow = O + (size_t(bh) * N + q) * HD;
#pragma unroll
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c4, o);
          tmem_wait_ld();
          if (q < N) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16x2(__uint_as_float(o[8 * c8 + 2 * e]) * mult,
                                    __uint_as_float(o[8 * c8 + 2 * e + 1]) * mult);
              st_global_v4(orow + 32 * c4 + 8 * c8, w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
        if (q < N) Lout[size_t(bh) * N + q] = (m - kPShift + log2f(l)) * 0.69314718055994530942f;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  if (*abort_flag && threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, void* O, float* L, const Shape& s,
                            float score_log2, float v_descale, int* err, cudaStream_t stream) {
  auto kern = attn_fwd_fp8_kernel<CAUSAL>;
  cudaError_t e = set_smem_limit_once<attn_fwd_fp8_kernel<CAUSAL>>(Layout::kBytes);
  if (e != cudaSuccess) return e;
  const long long n_tasks = (long long)((s.n_tiles + 1) / 2) * s.BH;
  const dim3 grid(unsigned(fwd_grid(n_tasks, CAUSAL)));
  return launch_kernel(kern, grid, dim3(kThreads), Layout::kBytes, stream, tmQ, tmK, tmV,
                       reinterpret_cast<__nv_bfloat16*>(O), L, s.BH, s.N, score_log2, v_descale,
                       err);
}

}  // namespace fwd8

cudaError_t launch_fwd_fp8(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, void* O, float* L, const Shape& s,
                           float score_log2, float v_descale, int* err, cudaStream_t stream) {
  if (s.causal)
    return fwd8::launch_t<true>(tmQ, tmK, tmV, O, L, s, score_log2, v_descale, err, stream);
  return fwd8::launch_t<false>(tmQ, tmK, tmV, O, L, s, score_log2, v_descale, err, stream);
}

}  // namespace attn
