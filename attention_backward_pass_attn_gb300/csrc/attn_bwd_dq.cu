// attn_bwd_dq.cu -- dQ of exact attention by a separate query-stationary pass.
//
// The backward of "Training Transformers and Hybrid models on AMD Instinct
// MI300X Accelerators" (section "Flash Attention") needs dQ_i = s sum_j dS_ij
// k_j, a sum over key tiles, while its main kernel walks key tiles and holds
// dK and dV.  The fused design (attn_bwd_main.cuh with FUSED_DQ) adds each
// key tile's partial into an fp32 accumulator.  This pass is the other way:
// it holds dQ instead, and recomputes what it needs per key/value tile
// (section "Harnessing the MI300 Hardware Specs": the backward recomputes
// the forward's activations):
//
//    S   = Q K^T                 (tensor memory, 128 x 128 fp32)
//    P   = 2^(S s log2e - L log2e)      softmax warps, kept in registers
//    dP  = dO V^T                (into the same tensor-memory columns)
//    dS  = P o (dP - D)          softmax warps, bf16, back into those columns
//    dQ += dS K                  (A operand read from tensor memory)
//
// and writes dQ = bf16(s dQ) once: no accumulator in HBM, no reductions, and
// the result does not depend on any summation order across CTAs.  Its price
// is two extra contractions per (query tile, key tile) pair: S and dP are
// formed here and in the main kernel.  Which way is faster is measured.
//
// Design (GB300): one CTA owns two 128-row query tiles of one head (A, B),
// with Q and dO of both resident in shared memory, and streams 128-row K
// tiles through a two-stage TMA ring and V tiles through one stage.  Warps
// 0-3 are the softmax of tile A and 4-7 that of tile B (one thread per query
// row = one tensor-memory lane), warp 8 issues TMA, warp 9 issues
// tcgen05.mma and owns the tensor memory: dQ_A, dQ_B (d columns each) and
// one 128-column block per tile that holds S, then dP, then dS.  While the
// softmax warps of one tile work, the tensor core runs the other tile's
// contractions.  The causal mask, the sliding window and documents bound the
// key tiles each pair visits exactly as in the forward kernel.

#include "kernels.h"
#include "mask.cuh"
#include "ptx.cuh"

namespace attn {
namespace bwdq {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;

constexpr int kBarQFull = 0;     // Q and dO of both tiles
constexpr int kBarKFull = 1;     // + K stage (2)
constexpr int kBarKEmpty = 3;    // + K stage
constexpr int kBarVFull = 5;
constexpr int kBarVEmpty = 6;
constexpr int kBarSFull = 7;     // + tile: S in tensor memory
constexpr int kBarPDone = 9;     // + tile: S read, P in registers (128 arrivals)
constexpr int kBarDPFull = 11;   // + tile: dP in tensor memory
constexpr int kBarDSReady = 13;  // + tile: dS packed in tensor memory (128 arrivals)
constexpr int kBarDQFull = 15;   // every dQ contraction done
constexpr int kBarDrain = 16;
constexpr int kNumBars = 17;

template <int HD>
struct Layout {
  static constexpr int kTileBytes = 128 * HD * 2;  // one 128-row bf16 tile
  static constexpr int kQ = 0;                      // Q_A, Q_B
  static constexpr int kDO = kQ + 2 * kTileBytes;   // dO_A, dO_B
  static constexpr int kK = kDO + 2 * kTileBytes;   // two stages
  static constexpr int kV = kK + 2 * kTileBytes;    // one stage
  static constexpr int kBar = kV + kTileBytes;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  // At least half of the SM's shared memory: one CTA (owning all 512
  // tensor-memory columns) per SM.
  static constexpr int kRaw = (kAbort + 4 + 15) / 16 * 16;
  static constexpr int kBytes = kRaw > 118784 ? kRaw : 118784;
  static constexpr uint32_t kColDQ = 0;      // + tile * HD
  static constexpr uint32_t kColS = 2 * HD;  // + tile * 128: S, then dP, then dS
};

// Descriptor conventions as in the other kernels (128-byte swizzle, tiles of
// 128 rows in 64-column blocks of 16 KB): a K-major operand advances 32 bytes
// per 16-element k-step within a block and 16 KB across blocks; an MN-major
// operand advances 2 KB (16 rows) per k-step, its MN extent spanning blocks
// 16 KB apart (LBO).

template <int HD, bool CAUSAL, int MASK>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdO, const float* __restrict__ L2ws,
                       const float* __restrict__ Dws, __nv_bfloat16* __restrict__ dQ, int BH,
                       int N, float scale_log2, float scale, int window_arg,
                       const int* __restrict__ doc, int H, int* err) {
  const int window = MASK != kMaskPlain ? window_arg : 0;
  using Ly = Layout<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (sbase & 1023u) {  // uniform over the CTA: every thread returns here
    if (threadIdx.x == 0) report_error(err, kDevSmemAlign, 0x300);
    return;
  }

  const int n_tiles = (N + 127) >> 7;
  const int Npad = n_tiles * 128;
  const int n_pairs = (n_tiles + 1) >> 1;
  // Causal: pairs heaviest first across all heads; otherwise head by head,
  // so that the CTAs resident at one time share their heads' K and V in L2.
  const int bh = CAUSAL ? int(blockIdx.x % BH) : int(blockIdx.x / n_pairs);
  const int pair = CAUSAL ? (n_pairs - 1 - int(blockIdx.x / BH)) : int(blockIdx.x % n_pairs);
  const int qt_a = 2 * pair;
  const bool has_b = qt_a + 1 < n_tiles;
  // Key/value tiles kv_lo .. kv_lo + n_kv - 1, as in the forward.
  const int kv_end = CAUSAL ? min(n_tiles, qt_a + (has_b ? 2 : 1)) : n_tiles;
  const int lo_key = qt_a * 128 - window + 1;
  int kv_lo = (CAUSAL && window > 0 && lo_key > 0) ? lo_key / 128 : 0;
  int n_kv = kv_end - kv_lo;
  const int* docb = MASK == kMaskDocument ? doc + size_t(bh / H) * N : nullptr;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      const bool per_row = (i == kBarPDone || i == kBarPDone + 1 || i == kBarDSReady ||
                            i == kBarDSReady + 1);
      mbar_init(bar(i), per_row ? 128 : 1);
    }
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
    tma_prefetch_desc(&tmdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtx ctx{abort_flag, err, kWaitLimitNs};
  // Everything above overlaps the previous kernel; its results are read below.
  grid_dep_wait();
  grid_dep_launch();
  if (MASK == kMaskDocument) {  // row lower bounds never decrease along the tile pair
    kv_lo = first_visible_key(qt_a * 128, docb, window, N) / 128;
    n_kv = kv_end - kv_lo;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      const int nt = has_b ? 2 : 1;
      mbar_arrive_expect_tx(bar(kBarQFull), 2 * nt * Ly::kTileBytes);
      for (int t = 0; t < nt; ++t)
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb) {
          tma_load_3d(sbase + Ly::kQ + t * Ly::kTileBytes + cb * 16384, &tmQ, bar(kBarQFull),
                      cb * 64, (qt_a + t) * 128, bh);
          tma_load_3d(sbase + Ly::kDO + t * Ly::kTileBytes + cb * 16384, &tmdO, bar(kBarQFull),
                      cb * 64, (qt_a + t) * 128, bh);
        }
    }
    __syncwarp();
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1, n = j >> 1;
      // K(j) reuses the stage of K(j-2), free once its last dQ contraction is done.
      if (j >= 2 && !mbar_wait_warp(bar(kBarKEmpty + s), (n - 1) & 1, ctx, 0x310)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarKFull + s), Ly::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(sbase + Ly::kK + s * Ly::kTileBytes + cb * 16384, &tmK, bar(kBarKFull + s),
                      cb * 64, (kv_lo + j) * 128, bh);
      }
      __syncwarp();
      // V(j) replaces V(j-1) once both dP contractions of j-1 are done.
      if (j >= 1 && !mbar_wait_warp(bar(kBarVEmpty), (j - 1) & 1, ctx, 0x311)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarVFull), Ly::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(sbase + Ly::kV + cb * 16384, &tmV, bar(kBarVFull), cb * 64,
                      (kv_lo + j) * 128, bh);
      }
      __syncwarp();
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per key/value tile j: dP_A, dP_B (each once its softmax warps have read
    // S), then dQ_A += dS_A K and S_A(j+1), then dQ_B and S_B(j+1).  The next
    // S goes into the columns the dQ contraction just read its dS from: the
    // tensor core runs one CTA's contractions in issue order.
    constexpr uint32_t kIdS = make_idesc_bf16(128, 128, 0, 0);  // S = Q K^T, dP = dO V^T
    constexpr uint32_t kIdQ = make_idesc_bf16(128, HD, 0, 1);   // dQ += dS K, K MN-major
    auto issue_nt = [&](int t, uint32_t a_base, uint32_t b_base, int bar_id) {
      const uint64_t da = make_sdesc_sw128(a_base + t * Ly::kTileBytes, 16, 1024);
      const uint64_t db = make_sdesc_sw128(b_base, 16, 1024);
      const uint32_t d = tbase + Ly::kColS + 128 * t;
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
        mma_ss(d, sdesc_add(da, off), sdesc_add(db, off), kIdS, k > 0 ? 1u : 0u);
      }
      tc_commit(bar(bar_id + t));
    };
    auto issue_s = [&](int t, int ks) {  // S_t = Q_t K^T; elected lane only
      issue_nt(t, sbase + Ly::kQ, sbase + Ly::kK + ks * Ly::kTileBytes, kBarSFull);
    };
    auto issue_dp = [&](int t) {  // dP_t = dO_t V^T; elected lane only
      issue_nt(t, sbase + Ly::kDO, sbase + Ly::kV, kBarDPFull);
    };
    auto issue_dq = [&](int t, int ks, uint32_t acc) {  // dQ_t += dS_t K; elected lane only
      const uint64_t dk = make_sdesc_sw128(sbase + Ly::kK + ks * Ly::kTileBytes, 16384, 1024);
      const uint32_t d = tbase + Ly::kColDQ + HD * t;
      const uint32_t p = tbase + Ly::kColS + 128 * t;
#pragma unroll
      for (int k = 0; k < 8; ++k)  // 128 keys, 16 per step; dS packed 2 per column
        mma_ts(d, p + 8 * k, sdesc_add(dk, k * 2048), kIdQ, k > 0 ? 1u : acc);
    };
    bool ok = mbar_wait_warp(bar(kBarQFull), 0, ctx, 0x320) &&
              mbar_wait_warp(bar(kBarKFull), 0, ctx, 0x321);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_s(0, 0);
        if (has_b) issue_s(1, 0);
      }
      __syncwarp();
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ks = j & 1;
        const bool next = j + 1 < n_kv;
        const int ks1 = (j + 1) & 1, n1 = (j + 1) >> 1;
        const uint32_t acc = j > 0 ? 1u : 0u;
        if (!(ok = mbar_wait_warp(bar(kBarVFull), j & 1, ctx, 0x322))) break;
        if (!(ok = mbar_wait_warp(bar(kBarPDone + 0), j & 1, ctx, 0x323))) break;
        tc_fence_after();
        if (elect_one()) issue_dp(0);
        __syncwarp();
        if (has_b) {
          if (!(ok = mbar_wait_warp(bar(kBarPDone + 1), j & 1, ctx, 0x324))) break;
          tc_fence_after();
          if (elect_one()) issue_dp(1);
          __syncwarp();
        }
        if (elect_one()) tc_commit(bar(kBarVEmpty));
        __syncwarp();
        if (!(ok = mbar_wait_warp(bar(kBarDSReady + 0), j & 1, ctx, 0x325))) break;
        tc_fence_after();
        if (elect_one()) issue_dq(0, ks, acc);
        __syncwarp();
        if (next) {
          if (!(ok = mbar_wait_warp(bar(kBarKFull + ks1), n1 & 1, ctx, 0x326))) break;
          tc_fence_after();
          if (elect_one()) issue_s(0, ks1);
          __syncwarp();
        }
        if (has_b) {
          if (!(ok = mbar_wait_warp(bar(kBarDSReady + 1), j & 1, ctx, 0x327))) break;
          tc_fence_after();
          if (elect_one()) {
            issue_dq(1, ks, acc);
            if (next) issue_s(1, ks1);
          }
          __syncwarp();
        }
        if (elect_one()) tc_commit(bar(kBarKEmpty + ks));
        __syncwarp();
      }
      if (ok && elect_one()) tc_commit(bar(kBarDQFull));
      __syncwarp();
    }
    // Wait until every MMA issued above has completed before teardown.
    if (elect_one()) tc_commit(bar(kBarDrain));
    __syncwarp();
    volatile int never = 0;  // this wait ignores the CTA abort flag
    const WaitCtx own{&never, err, kWaitLimitNs};
    mbar_wait_warp(bar(kBarDrain), 0, own, 0x32F);
  } else {
    // ------------------------------------------------------------ softmax / dS
    const int t = warp >> 2;  // 0 = tile A, 1 = tile B
    const int r = threadIdx.x & 127;
    if (t == 0 || has_b) {
      const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
      const uint32_t tS = tbase + lane_off + Ly::kColS + 128 * t;
      const uint32_t tQ = tbase + lane_off + Ly::kColDQ + HD * t;
      const int q_tile0 = (qt_a + t) * 128;
      const int q = q_tile0 + r;
      // this row's L log2(e) (+inf on rows past N, so their P is 0) and D
      const float l2 = L2ws[size_t(bh) * Npad + q];
      const float dd = Dws[size_t(bh) * Npad + q];
      // first key this row may see (window, document)
      const int lo_q = MASK != kMaskPlain ? first_visible_key(q, docb, window, N) : 0;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        if (!(ok = mbar_wait_warp(bar(kBarSFull + t), j & 1, ctx, 0x330 + t))) break;
        tc_fence_after();
        const int kv0 = (kv_lo + j) * 128;
        // masked: above the diagonal, beyond N, or before the row's first key
        const bool below = MASK != kMaskPlain && kv0 < lo_q;
        const bool edge = (CAUSAL && kv0 + 127 > q_tile0) || kv0 + 128 > N || below;
        // P = 2^(S s log2e - L log2e), packed bf16, kept in registers until dS
        uint32_t pk[64];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t u[64];
          tmem_ld32(tS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
          tmem_ld32(tS + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          tmem_wait_ld();
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2) {
            float p0 = ex2(fmaf(__uint_as_float(u[2 * c2]), scale_log2, -l2));
            float p1 = ex2(fmaf(__uint_as_float(u[2 * c2 + 1]), scale_log2, -l2));
            if (edge) {
              const int kv = kv0 + 64 * h + 2 * c2;
              if ((CAUSAL && kv > q) || kv >= N || (below && kv < lo_q)) p0 = 0.f;
              if ((CAUSAL && kv + 1 > q) || kv + 1 >= N || (below && kv + 1 < lo_q)) p1 = 0.f;
            }
            pk[32 * h + c2] = pack_bf16x2(p0, p1);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(kBarPDone + t));
        if (!(ok = mbar_wait_warp(bar(kBarDPFull + t), j & 1, ctx, 0x332 + t))) break;
        tc_fence_after();
        // dS = P o (dP - D): the difference in fp32, packed once to bf16x2,
        // times the packed P; written over the first 64 columns (two keys
        // per column), which the h = 0 load has already read.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t u[64];
          tmem_ld32(tS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
          tmem_ld32(tS + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          tmem_wait_ld();
          uint32_t ds[32];
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2)
            ds[c2] = mul_bf16x2(pk[32 * h + c2], pack_bf16x2(__uint_as_float(u[2 * c2]) - dd,
                                                              __uint_as_float(u[2 * c2 + 1]) - dd));
          tmem_st32(tS + 32 * h, ds);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarDSReady + t));
      }
      if (ok && mbar_wait_warp(bar(kBarDQFull), 0, ctx, 0x338 + t)) {
        tc_fence_after();
        __nv_bfloat16* orow = dQ + (size_t(bh) * N + q) * HD;
#pragma unroll
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(tQ + 32 * c4, o);
          tmem_wait_ld();
          if (q < N) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16x2(__uint_as_float(o[8 * c8 + 2 * e]) * scale,
                                    __uint_as_float(o[8 * c8 + 2 * e + 1]) * scale);
              st_global_v4(orow + 32 * c4 + 8 * c8, w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      }
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
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, void* dQ,
                            const Workspace& ws, const Shape& s, float scale, int* err,
                            cudaStream_t stream) {
  using Ly = Layout<HD>;
  auto kern = attn_bwd_dq_kernel<HD, CAUSAL, MASK>;
  cudaError_t e = set_smem_limit_once<attn_bwd_dq_kernel<HD, CAUSAL, MASK>>(Ly::kBytes);
  if (e != cudaSuccess) return e;
  const int n_pairs = (s.n_tiles + 1) / 2;
  const dim3 grid(unsigned(n_pairs) * unsigned(s.BH));
  return launch_kernel(kern, grid, dim3(kThreads), Ly::kBytes, stream, tmQ, tmK, tmV, tmdO,
                       static_cast<const float*>(ws.L2), static_cast<const float*>(ws.D),
                       reinterpret_cast<__nv_bfloat16*>(dQ), s.BH, s.N,
                       scale * 1.4426950408889634f, scale, s.window, s.doc, s.H, err);
}

}  // namespace bwdq

cudaError_t launch_bwd_dq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, void* dQ, const Workspace& ws, const Shape& s,
                          float scale, int* err, cudaStream_t stream) {
  const int mask = !s.causal ? kMaskPlain
                   : s.doc        ? kMaskDocument
                   : s.window > 0 ? kMaskWindow
                                  : kMaskPlain;
#define ATTN_DQ(HD_, C_, M_) \
  bwdq::launch_t<HD_, C_, M_>(tmQ, tmK, tmV, tmdO, dQ, ws, s, scale, err, stream)
  if (s.d == 64) {
    if (!s.causal) return ATTN_DQ(64, false, kMaskPlain);
    if (mask == kMaskDocument) return ATTN_DQ(64, true, kMaskDocument);
    if (mask == kMaskWindow) return ATTN_DQ(64, true, kMaskWindow);
    return ATTN_DQ(64, true, kMaskPlain);
  }
  if (!s.causal) return ATTN_DQ(128, false, kMaskPlain);
  if (mask == kMaskDocument) return ATTN_DQ(128, true, kMaskDocument);
  if (mask == kMaskWindow) return ATTN_DQ(128, true, kMaskWindow);
  return ATTN_DQ(128, true, kMaskPlain);
#undef ATTN_DQ
}

}  // namespace attn
