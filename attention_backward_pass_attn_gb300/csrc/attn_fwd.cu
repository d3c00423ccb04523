// attn_fwd.cu -- exact-attention forward on sm_103a: O = softmax(s Q K^T) V and
// the row log-sum-exp L, never storing the N x N score matrix.
//
// This is the forward the backward consumes (FlashAttention-2 forward, page
// "Training Transformers and Hybrid models on AMD Instinct MI300X
// Accelerators", section "Flash Attention").  Design for GB300:
//
//  * A task is two 128-row query tiles of one head (A and B) against the K/V
//    tiles they see.  A CTA takes one or more tasks in turn, streaming 128-row
//    K/V tiles through a two-stage TMA ring that runs on across its tasks: the
//    next task's query and first K/V tiles load, and its first S is computed,
//    while this task's last P V and output run.  Both query tiles reuse every
//    K/V tile in shared memory.  The grid (fwd_grid) is persistent, one CTA
//    per SM, without the causal mask or with few tasks; else one CTA per task.
//  * Warp roles: warps 0-3 run the softmax of tile A, warps 4-7 that of tile
//    B (one thread per query row = one TMEM lane), warp 8 issues TMA copies,
//    warp 9 issues tcgen05.mma and owns the tensor-memory allocation.
//  * Tensor memory (512 columns x 128 lanes, fp32): O_A, O_B (d columns each)
//    and S_A, S_B (128 columns each).  S = Q K^T lands in S_x; the softmax
//    threads overwrite its first 64 columns with P in bf16 (two per column),
//    and the tensor core reads P straight from tensor memory for O += P V.
//  * Online softmax in base 2 (log2(e) folded into the scale) with lazy
//    rescaling: the running maximum is only moved (and O rescaled in tensor
//    memory) when it grows by more than 2^8, which keeps P <= 256.
//  * While the softmax of tile A runs, the tensor core works on tile B, and
//    the next S of one tile is computed while the other tile's P V runs.
//  * Causal: a task stops at the last key tile its rows can see; tiles on the
//    diagonal are masked element-wise, each row against the first and last
//    column it may see.  Tasks are taken heaviest first.
//    Without the mask they run head by head, so the CTAs working at one time
//    share K and V in L2.
//  * Mask variants (mask.cuh: a causal sliding window, documents of packed
//    sequences) have their own instantiations: a task starts at the first key
//    tile its first row can see, and each row masks keys below its bound.
//  * Every mbarrier wait is bounded (see ptx.cuh); on expiry the kernel
//    records an error, drains the tensor core and exits normally.

#include "f32x2.cuh"
#include "kernels.h"
#include "mask.cuh"
#include "ptx.cuh"

namespace attn {
namespace fwd {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;

// Barrier indices.
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;
constexpr int kBarKFull = 2;                       // + stage
constexpr int kBarKEmpty = kBarKFull + kStages;    // + stage
constexpr int kBarVFull = kBarKEmpty + kStages;    // + stage
constexpr int kBarVEmpty = kBarVFull + kStages;    // + stage
constexpr int kBarSFull = kBarVEmpty + kStages;    // + tile (0 = A, 1 = B)
constexpr int kBarPReady = kBarSFull + 2;          // + tile
constexpr int kBarOFull = kBarPReady + 2;          // + tile
constexpr int kBarDrain = kBarOFull + 2;
constexpr int kNumBars = kBarDrain + 1;

template <int HD>
struct Layout {
  static constexpr int kTileBytes = 128 * HD * 2;   // one 128-row bf16 tile
  static constexpr int kQ = 0;                       // two query tiles
  static constexpr int kK = kQ + 2 * kTileBytes;     // kStages key tiles
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  // Padded past half of the SM's shared memory so that at most one CTA (which
  // allocates all 512 tensor-memory columns) is resident per SM.
  static constexpr int kRaw = (kAbort + 4 + 15) / 16 * 16;
  static constexpr int kBytes = kRaw > 118784 ? kRaw : 118784;
  // tensor-memory columns
  static constexpr uint32_t kColO = 0;           // + tile * HD
  static constexpr uint32_t kColS = 2 * HD;      // + tile * 128
};

// One task: query tiles qt_a (A) and qt_a + 1 (B, when N reaches it) of head
// bh against key/value tiles kv_lo .. kv_lo + n_kv - 1.
struct Task {
  int bh, qt_a, kv_lo, n_kv;
  bool has_b;
};

// Task i of BH * n_pairs.  Causal: heaviest first (a later pair sees more
// key/value tiles), heads interleaved.  Without the mask every task costs the
// same and tasks run head by head, so the CTAs working at one time share
// their heads' K and V in L2.
template <bool CAUSAL, int MASK>
struct TaskMap {
  int BH, H, N, n_tiles, n_pairs, window;
  const int* doc;  // documents: map [B][N] (device)

  __device__ __forceinline__ Task range(int bh, int pair) const {
    Task t;
    t.bh = bh;
    t.qt_a = 2 * pair;
    t.has_b = t.qt_a + 1 < n_tiles;
    const int kv_end = CAUSAL ? min(n_tiles, t.qt_a + (t.has_b ? 2 : 1)) : n_tiles;
    // Under a window or documents the first row of tile A bounds the first
    // key tile; tile B's rows start no earlier (lower bounds never decrease
    // along a pair), and their extra leading keys are masked per row.
    int lo = 0;
    if (MASK != kMaskPlain) {
      const int* docb = MASK == kMaskDocument ? doc + size_t(bh / H) * N : nullptr;
      lo = first_visible_key(t.qt_a * 128, docb, window, N) / 128;
    }
    t.kv_lo = lo;
    t.n_kv = kv_end - lo;
    return t;
  }
  __device__ __forceinline__ Task task(int i) const {
    if (CAUSAL) return range(i % BH, n_pairs - 1 - i / BH);
    return range(i / n_pairs, i % n_pairs);
  }
};

// CTA b of G takes tasks b, 2G-1-b, 2G+b, 4G-1-b, ... (a snake over rounds,
// which evens out the heavy-first order); -1 past the last task.  With one
// CTA per task (G = the task count) that is task b alone.
__device__ __forceinline__ int snake_task(int k, int b, int G, int n_tasks) {
  const long long idx = (k & 1) ? (long long)k * G + (G - 1 - b) : (long long)k * G + b;
  return idx < n_tasks ? int(idx) : -1;
}

// Descriptor conventions (128-byte swizzle, tiles of 128 rows in 64-column
// blocks of 16 KB): a K-major operand advances 32 bytes per 16-element k-step
// within a block and 16 KB across blocks; an MN-major operand advances 2 KB
// (16 rows) per k-step, its MN extent spanning blocks 16 KB apart (LBO).

template <int HD, bool CAUSAL, int MASK>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                    float* __restrict__ Lout, int BH, int N, float scale_log2, int window_arg,
                    const int* __restrict__ doc, int H, int* err) {
  // The window and document masks have their own instantiations; without
  // them their code compiles away.
  const int window = MASK != kMaskPlain ? window_arg : 0;
  using Ly = Layout<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (sbase & 1023u) {  // uniform over the CTA: every thread returns here
    if (threadIdx.x == 0) report_error(err, kDevSmemAlign, 0x100);
    return;
  }

  const int n_tiles = (N + 127) >> 7;
  const int n_pairs = (n_tiles + 1) >> 1;
  const int n_tasks = BH * n_pairs;
  const int G = int(gridDim.x), cta = int(blockIdx.x);
  const TaskMap<CAUSAL, MASK> tm{BH, H, N, n_tiles, n_pairs, window, doc};

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 128);
      mbar_init(bar(kBarOFull + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
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
  // Everything above overlaps the previous kernel; its results are read below.
  grid_dep_wait();
  grid_dep_launch();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (warp-uniform operands); one lane issues.
    // Key/value tiles run through the ring across tasks (g counts them), so
    // the next task's first tiles load while this one finishes.
    bool ok = true;
    int g = 0;
    for (int k = 0, i = snake_task(0, cta, G, n_tasks); ok && i >= 0;
         i = snake_task(++k, cta, G, n_tasks)) {
      const Task tk = tm.task(i);
      // Both query tiles are free once the previous task's last S completed.
      if (k > 0 && !(ok = mbar_wait_warp(bar(kBarQEmpty), (k - 1) & 1, ctx, 0x112))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarQFull), (tk.has_b ? 2 : 1) * Ly::kTileBytes);
        for (int t = 0; t < (tk.has_b ? 2 : 1); ++t)
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb)
            tma_load_3d(sbase + Ly::kQ + t * Ly::kTileBytes + cb * 16384, &tmQ, bar(kBarQFull),
                        cb * 64, (tk.qt_a + t) * 128, tk.bh);
      }
      __syncwarp();
      for (int j = 0; j < tk.n_kv; ++j, ++g) {
        const int s = g % kStages, n = g / kStages;
        if (g >= kStages && !(ok = mbar_wait_warp(bar(kBarKEmpty + s), (n - 1) & 1, ctx, 0x110)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(kBarKFull + s), Ly::kTileBytes);
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb)
            tma_load_3d(sbase + Ly::kK + s * Ly::kTileBytes + cb * 16384, &tmK,
                        bar(kBarKFull + s), cb * 64, (tk.kv_lo + j) * 128, tk.bh);
        }
        __syncwarp();
        if (g >= kStages && !(ok = mbar_wait_warp(bar(kBarVEmpty + s), (n - 1) & 1, ctx, 0x111)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(kBarVFull + s), Ly::kTileBytes);
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb)
            tma_load_3d(sbase + Ly::kV + s * Ly::kTileBytes + cb * 16384, &tmV,
                        bar(kBarVFull + s), cb * 64, (tk.kv_lo + j) * 128, tk.bh);
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues.  Every
    // descriptor is a per-tile base plus a compile-time k-step offset.
    constexpr uint32_t kIdS = make_idesc_bf16(128, 128, 0, 0);  // S = Q K^T
    constexpr uint32_t kIdO = make_idesc_bf16(128, HD, 0, 1);   // O += P V
    const uint64_t dQa = make_sdesc_sw128(sbase + Ly::kQ, 16, 1024);
    const uint64_t dQb = make_sdesc_sw128(sbase + Ly::kQ + Ly::kTileBytes, 16, 1024);
    auto issue_s = [&](int t, int stage) {  // elected lane only
      const uint64_t dq = t == 0 ? dQa : dQb;
      const uint64_t dk = make_sdesc_sw128(sbase + Ly::kK + stage * Ly::kTileBytes, 16, 1024);
      const uint32_t d = tbase + Ly::kColS + 128 * t;
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
        mma_ss(d, sdesc_add(dq, off), sdesc_add(dk, off), kIdS, k > 0 ? 1u : 0u);
      }
      tc_commit(bar(kBarSFull + t));
    };
    auto issue_pv = [&](int t, int stage, uint32_t acc) {  // elected lane only
      const uint64_t dv = make_sdesc_sw128(sbase + Ly::kV + stage * Ly::kTileBytes, 16384, 1024);
      const uint32_t d = tbase + Ly::kColO + HD * t;
      const uint32_t p = tbase + Ly::kColS + 128 * t;
#pragma unroll
      for (int k = 0; k < 8; ++k)  // 128 keys, 16 per step; P packed 2 per column
        mma_ts(d, p + 8 * k, sdesc_add(dv, k * 2048), kIdO, k > 0 ? 1u : acc);
    };
    // Handshake counts across tasks: g key/value tiles, ca (cb) S/P rounds of
    // tile A (B).  A task's first P V overwrites O_t; the softmax warps of
    // tile t read the previous task's O_t before they signal the first P of
    // this one, so the P-ready wait covers that hazard.  Tensor-core
    // instructions of this thread run in issue order, so an S written into
    // the columns that hold P comes after the P V that reads them.
    bool ok = true;
    int g = 0, ca = 0, cb = 0;
    for (int k = 0, i = snake_task(0, cta, G, n_tasks); ok && i >= 0;
         i = snake_task(++k, cta, G, n_tasks)) {
      const Task tk = tm.task(i);
      const int n_kv = tk.n_kv;
      if (!(ok = mbar_wait_warp(bar(kBarQFull), k & 1, ctx, 0x120))) break;
      if (!(ok = mbar_wait_warp(bar(kBarKFull + g % kStages), (g / kStages) & 1, ctx, 0x121)))
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
        if (!(ok = mbar_wait_warp(bar(kBarVFull + s), (g / kStages) & 1, ctx, 0x122))) break;
        if (!(ok = mbar_wait_warp(bar(kBarPReady + 0), (ca + j) & 1, ctx, 0x123))) break;
        tc_fence_after();
        if (elect_one()) issue_pv(0, s, acc);
        __syncwarp();
        if (next) {
          if (!(ok = mbar_wait_warp(bar(kBarKFull + s1), n1 & 1, ctx, 0x124))) break;
          tc_fence_after();
          if (elect_one()) issue_s(0, s1);
          __syncwarp();
        }
        if (tk.has_b) {
          if (!(ok = mbar_wait_warp(bar(kBarPReady + 1), (cb + j) & 1, ctx, 0x125))) break;
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
    // Wait until every MMA issued above has completed before teardown.
    if (elect_one()) tc_commit(bar(kBarDrain));
    __syncwarp();
    volatile int never = 0;  // this wait ignores the CTA abort flag
    const WaitCtx own{&never, err, kWaitLimitNs};
    mbar_wait_warp(bar(kBarDrain), 0, own, 0x12F);
  } else {
    // ------------------------------------------------------------ softmax
    // 0 = tile A, 1 = tile B.  The mask changes no value (softmax warps are
    // 0-7) but bounds t for the compiler: fewer registers spill, and the
    // kernel measured 1-3 % faster on the causal workloads.
    const int t = (warp >> 2) & 1;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + Ly::kColS + 128 * t;
    const uint32_t tO = tbase + lane_off + Ly::kColO + HD * t;
    bool ok = true;
    int c = 0;   // S/P rounds of this tile so far
    int no = 0;  // outputs of this tile so far
    for (int k = 0, i = snake_task(0, cta, G, n_tasks); ok && i >= 0;
         i = snake_task(++k, cta, G, n_tasks)) {
      const Task tk = tm.task(i);
      if (t == 1 && !tk.has_b) continue;
      const int q_tile0 = (tk.qt_a + t) * 128;
      const int q = q_tile0 + r;
      // first key this row may see (window, document)
      const int* docb = MASK == kMaskDocument ? doc + size_t(tk.bh / H) * N : nullptr;
      const int lo_q = MASK != kMaskPlain ? first_visible_key(q, docb, window, N) : 0;
      float m = -INFINITY;  // running max of the base-2 scaled scores
      float l = 0.f;        // running sum of 2^(x - m)
      for (int j = 0; j < tk.n_kv; ++j) {
        if (!(ok = mbar_wait_warp(bar(kBarSFull + t), (c + j) & 1, ctx, 0x130 + t))) break;
        tc_fence_after();
        uint32_t u[128];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&u[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&u[96]));
        tmem_wait_ld();
        const int kv0 = (tk.kv_lo + j) * 128;
        // masked: above the diagonal, beyond N, or before the first key the
        // row may see (sliding window, document)
        const bool below = MASK != kMaskPlain && kv0 < lo_q;
        if ((CAUSAL && kv0 + 127 > q_tile0) || kv0 + 128 > N || below) {
          // the row sees columns e_lo .. e_hi of this tile
          const int e_hi = min(CAUSAL ? q - kv0 : 127, N - 1 - kv0);
          const int e_lo = below ? lo_q - kv0 : 0;
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e > e_hi || e < e_lo) u[e] = __float_as_uint(-INFINITY);
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
        const float mt = mx * scale_log2;  // scale > 0, so the max commutes with it
        const float m_new = fmaxf(m, mt);
        // Lazy rescale: move the reference maximum (and rescale l and O by
        // 2^(m - m_new)) only when the maximum grew by more than 8 in base 2.
        const bool rescale = m_new > m + 8.f;
        const float alpha = rescale ? ex2(m - m_new) : 1.f;
        if (rescale) {
          l *= alpha;
          m = m_new;
        }
        const float mb = (m == -INFINITY) ? 0.f : m;
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2) {
            float x0, x1;  // s scale_log2 - mb for two scores in one instruction
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(u[64 * h + 2 * c2]),
                                        __uint_as_float(u[64 * h + 2 * c2 + 1])),
                                  f32x2(scale_log2, scale_log2), f32x2(-mb, -mb)), x0, x1);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            rs[c2 & 3] += p0 + p1;
            pk[c2] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + 32 * h, pk);
        }
        l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        // tcgen05.ld/st are warp-collective: if any row of the warp moved its
        // maximum, the whole warp rescales (alpha = 1 leaves the other rows
        // unchanged).  O holds P V of earlier tiles; PV(j-1) has completed.
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c4, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + 32 * c4, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarPReady + t));
      }
      if (!ok) break;
      c += tk.n_kv;
      if (!(ok = mbar_wait_warp(bar(kBarOFull + t), no & 1, ctx, 0x138 + t))) break;
      ++no;
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = O + (size_t(tk.bh) * N + q) * HD;
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
              w4[e] = pack_bf16x2(__uint_as_float(o[8 * c8 + 2 * e]) * inv_l,
                                  __uint_as_float(o[8 * c8 + 2 * e + 1]) * inv_l);
            st_global_v4(orow + 32 * c4 + 8 * c8, w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (q < N) Lout[size_t(tk.bh) * N + q] = (m + log2f(l)) * 0.69314718055994530942f;
      // O_t has been read into registers (tmem_wait_ld above) before this
      // warp signals the next task's first P.
      tc_fence_before();
    }
  }

  // ---------------------------------------------------------------- teardown
  if (*abort_flag && threadIdx.x == 0) {
    // Give copies still in flight time to land before the CTA retires.
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

template <int HD, bool CAUSAL, int MASK>
static cudaError_t launch_t(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, void* O, float* L, const Shape& s,
                            float scale, int* err, cudaStream_t stream) {
  using Ly = Layout<HD>;
  auto kern = attn_fwd_kernel<HD, CAUSAL, MASK>;
  cudaError_t e = set_smem_limit_once<attn_fwd_kernel<HD, CAUSAL, MASK>>(Ly::kBytes);
  if (e != cudaSuccess) return e;
  const long long n_tasks = (long long)((s.n_tiles + 1) / 2) * s.BH;
  const dim3 grid(unsigned(fwd_grid(n_tasks, CAUSAL)));
  const float scale_log2 = scale * 1.4426950408889634f;
  return launch_kernel(kern, grid, dim3(kThreads), Ly::kBytes, stream, tmQ, tmK, tmV,
                       reinterpret_cast<__nv_bfloat16*>(O), L, s.BH, s.N, scale_log2, s.window,
                       s.doc, s.H, err);
}

}  // namespace fwd

cudaError_t launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       void* O, float* L, const Shape& s, float scale, int* err,
                       cudaStream_t stream) {
  const int mask = !s.causal ? kMaskPlain
                   : s.doc        ? kMaskDocument
                   : s.window > 0 ? kMaskWindow
                                  : kMaskPlain;
  if (s.d == 64) {
    if (!s.causal) return fwd::launch_t<64, false, kMaskPlain>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
    if (mask == kMaskDocument)
      return fwd::launch_t<64, true, kMaskDocument>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
    if (mask == kMaskWindow)
      return fwd::launch_t<64, true, kMaskWindow>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
    return fwd::launch_t<64, true, kMaskPlain>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
  }
  if (!s.causal) return fwd::launch_t<128, false, kMaskPlain>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
  if (mask == kMaskDocument)
    return fwd::launch_t<128, true, kMaskDocument>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
  if (mask == kMaskWindow)
    return fwd::launch_t<128, true, kMaskWindow>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
  return fwd::launch_t<128, true, kMaskPlain>(tmQ, tmK, tmV, O, L, s, scale, err, stream);
}

}  // namespace attn
