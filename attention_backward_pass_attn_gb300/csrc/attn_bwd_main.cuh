// attn_bwd_main.cuh -- the fused main kernel of the exact-attention backward
// (step 2 of attn_bwd) and its host-side launcher template.  Included by
// attn_bwd.cu (the instantiations that also reduce dQ) and attn_bwd_split.cu
// (the instantiations that leave dQ to the separate query-stationary pass of
// attn_bwd_dq.cu), so the two families compile in parallel.
//
// Per 128-row key/value tile, looping over the 128-row query tiles that see
// it, five (or four) tcgen05.mma contractions:
//    S^T = K Q^T              (tensor memory, 128 x 128 fp32)
//    P^T = 2^(S^T s log2e - L log2e)    softmax warps, written back as bf16
//    dP^T = V dO^T            (tensor memory)
//    dV  += P^T dO            (A operand read from tensor memory)
//    dS^T = P^T o (dP^T - D)  softmax warps, bf16 into shared memory (for
//                             dQ) or back into the dP^T columns
//    dK  += dS^T Q            (A operand from shared memory, or from tensor
//                              memory where dQ does not take the dP^T columns)
//    dQ_i = dS K              (FUSED_DQ only: tensor memory, then staged
//                              through shared memory and added into the fp32
//                              accumulator by TMA reduce-add)
// dK and dV stay in tensor memory for the whole loop and are written once, by
// TMA tile stores from the dS^T tile (the item's epilogue).
//
// Warp roles (14 warps): 0-3 drain dQ from tensor memory into the
// accumulator (idle without FUSED_DQ); 4-7 and 8-11 each own 64 of the 128
// query columns of S^T/dP^T (one key row = one tensor-memory lane per
// thread); 12 issues TMA; 13 issues tcgen05.mma and owns the tensor-memory
// allocation.  The grid is persistent: each CTA walks a list of (head,
// key/value tile) work items, and all barrier phases continue from one item
// to the next.  Tensor memory (512 columns): dV | dK | S^T (P^T) | dP^T |
// (dQ: its own columns for d = 64, the dP^T columns for d = 128).  Shared
// memory: K, V, two stages of Q (with its per-row L and D vectors), dO (two
// stages, except for d = 128 with FUSED_DQ, where the dQ staging buffers take
// the room of the second), the dS^T tile (which also stages dV and dK at the
// end of an item) and, with FUSED_DQ, two 16 KB fp32 staging buffers for the
// dQ reduction.
//
// Work items are ordered heaviest first over all heads under the causal
// mask, and in L2-sized groups of heads without it.  Mask variants (a causal
// sliding window; documents of packed sequences, see mask.cuh) have their
// own instantiations: items end at the last query tile that still sees the
// key/value tile, and the softmax warps zero P outside the mask on the edge
// tiles; with documents, the preprocessing step tabulates those ranges and a
// one-CTA sort (attn_bwd_order_kernel) orders the items by size.
#pragma once

#include "f32x2.cuh"
#include "kernels.h"
#include "mask.cuh"
#include "ptx.cuh"

namespace attn {
namespace bwd {

constexpr int kThreads = 448;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;

// Item-level barriers (one phase per work item of the CTA).
constexpr int kBarKFull = 0;
constexpr int kBarVFull = 1;
constexpr int kBarKEmpty = 2;
constexpr int kBarVEmpty = 3;
constexpr int kBarAccFull = 4;    // dK, dV complete in tensor memory
constexpr int kBarAccEmpty = 5;   // dK, dV read out by the epilogue
// Tile-level barriers (one phase per query tile the CTA processes).
constexpr int kBarQFull = 6;      // + stage
constexpr int kBarQEmpty = 8;     // + stage
constexpr int kBarDOFull = 10;    // + dO stage
constexpr int kBarDOEmpty = 12;   // + dO stage
constexpr int kBarSFull = 14;
constexpr int kBarPReady = 15;
constexpr int kBarDPFull = 16;
constexpr int kBarDSReady = 17;
constexpr int kBarDSFree = 18;
constexpr int kBarDQFull = 19;
constexpr int kBarDQFree = 20;
constexpr int kBarDrain = 21;
// The item epilogue stages dV and dK through the shared dS^T tile (two turns
// for d = 128, one for d = 64): written by the softmax warps of a turn, then
// stored by TMA, after which the tile is free again.  One pair per turn, so
// that each barrier completes one phase per item.
constexpr int kBarEpiFull = 22;   // + turn
constexpr int kBarEpiFree = 24;   // + turn
constexpr int kNumBars = 26;
constexpr int kDrainBarrierId = 1;  // named barrier of the 128 dQ-drain threads

// Work items are (head, key/value tile) pairs.  Heads are taken in groups
// of HG whose query, dO and dQ-accumulator tiles fit in L2 together; within
// a group the index runs key/value-tile major, i = jt * hg + (bh - first
// head), so under the causal mask (a smaller jt sees more query tiles) each
// group goes heaviest first.  The grid is persistent (at most one CTA per
// SM); CTA b of G takes items b, 2G-1-b, 2G+b, 4G-1-b, ... (a snake over
// rounds, which evens out the heavy-first order).  Returns -1 past the last
// item.
__device__ __forceinline__ int snake_item(int k, int b, int G, int n_items) {
  const int idx = (k & 1) ? k * G + (G - 1 - b) : k * G + b;
  return idx < n_items ? idx : -1;
}

struct ItemMap {
  int BH, n_tiles, HG;
  __device__ __forceinline__ void decode(int i, int& jt, int& bh) const {
    const int per_group = HG * n_tiles;
    const int gr = i / per_group, r = i - gr * per_group;
    const int hg = BH - gr * HG < HG ? BH - gr * HG : HG;  // heads in this group
    jt = r / hg;
    bh = gr * HG + (r - jt * hg);
  }
};

template <int HD, bool FUSED_DQ>
struct Layout {
  static constexpr int kTileBytes = 128 * HD * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;          // + stage * kTileBytes
  // dO: two stages, so that the next dO arrives while this one is in use;
  // one for d = 128 when the dQ staging buffers below fill shared memory.
  static constexpr int kDOStages = (HD == 64 || !FUSED_DQ) ? 2 : 1;
  static constexpr int kDO = kQ + 2 * kTileBytes;     // + stage * kTileBytes
  static constexpr int kDS = kDO + kDOStages * kTileBytes;  // 128 x 128 bf16, two 16 KB blocks
  static constexpr int kStage = kDS + 32768;          // 2 x (128 rows x 32 fp32), swizzled
  static constexpr int kVec = kStage + (FUSED_DQ ? 32768 : 0);         // stage s: L2 at +1024 s, D at +1024 s + 512
  static constexpr int kBar = kVec + 2048;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  // At least half of the SM's shared memory: one CTA (owning all 512
  // tensor-memory columns) per SM.
  static constexpr int kRaw = (kAbort + 4 + 15) / 16 * 16;
  static constexpr int kBytes = kRaw > 118784 ? kRaw : 118784;
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = HD;
  static constexpr uint32_t kColS = 2 * HD;
  static constexpr uint32_t kColDP = 2 * HD + 128;
  // d = 64 leaves 128 of the 512 columns free: dQ gets its own columns, so the
  // next dP does not wait for the drain.  d = 128 has no room: dQ reuses the
  // dP columns once the softmax warps have read them.
  static constexpr bool kSeparateDq = HD == 64;
  static constexpr uint32_t kColDQ = kSeparateDq ? 2 * HD + 256 : kColDP;
  // Where dQ shares the dP^T columns, dQ_i is issued before dK, so that its
  // drain overlaps dK's contraction instead of holding back the next dP; dK
  // then reads dS^T from shared memory (dQ has overwritten the columns).
  // Elsewhere dK reads dS^T from the dP^T columns, packed there by the
  // softmax warps, and no shared dS^T is needed without dQ.
  static constexpr bool kDqFirst = FUSED_DQ && !kSeparateDq;
  // Turns of the item epilogue through the 32 KB dS^T tile: dV then dK for
  // d = 128 (32 KB each), both at once for d = 64.
  static constexpr int kEpiTurns = HD == 128 ? 2 : 1;
};

// Descriptor conventions (128-byte swizzle, tiles of 128 rows in 64-column
// blocks of 16 KB): a K-major operand advances 32 bytes per 16-element k-step
// within a block and 16 KB across blocks; an MN-major operand advances 2 KB
// (16 rows) per k-step, its MN extent spanning blocks 16 KB apart (LBO).

template <int HD, bool CAUSAL, int MASK, bool FUSED_DQ>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmAcc,
                         const __grid_constant__ CUtensorMap tmDK,
                         const __grid_constant__ CUtensorMap tmDV, const float* __restrict__ L2ws,
                         const float* __restrict__ Dws, int BH,
                         int N, int head_group, int window_arg, const int* __restrict__ doc,
                         int H, const int2* __restrict__ items, const int* __restrict__ qend,
                         const int* __restrict__ order, float scale, float scale_log2,
                         int* err) {
  // The window and document masks have their own instantiations; without
  // them their code compiles away.
  const int window = MASK != kMaskPlain ? window_arg : 0;
  using Ly = Layout<HD, FUSED_DQ>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(err, kDevSmemAlign, 0x200);
    return;
  }

  const int n_tiles = (N + 127) >> 7;
  const int Npad = n_tiles * 128;
  const int n_items = BH * n_tiles;
  const ItemMap imap{BH, n_tiles, head_group};
  // With documents the items come from the sorted list (heaviest first).
  auto decode_item = [&](int idx, int& jt, int& bh) {
    if (MASK == kMaskDocument) {
      const int id = order[idx];
      bh = id / n_tiles;
      jt = id - bh * n_tiles;
    } else {
      imap.decode(idx, jt, bh);
    }
  };
  // Query tiles of the item with key/value tile jt: it0 .. it0 + n_it - 1.
  // Under the causal mask they start at the diagonal; under a sliding window
  // they end at the last query that still sees a key of the tile,
  // jt * 128 + 127 + window - 1; with documents the preprocessing step has
  // tabulated where they end (read only after griddepcontrol.wait).
  auto item_tiles = [&](int jt, int bh) {
    if (MASK == kMaskDocument) {
      const int last = items[size_t(bh) * n_tiles + jt].x;
      return (last < jt ? jt : (last >= n_tiles ? n_tiles - 1 : last)) - jt + 1;
    }
    int last = n_tiles - 1;
    if (CAUSAL && window > 0) {
      const int lq = (jt * 128 + 126 + window) >> 7;
      if (lq < last) last = lq;
    }
    return last - (CAUSAL ? jt : 0) + 1;
  };
  const int G = gridDim.x, b = blockIdx.x;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      // arrivals per phase: the 256 softmax threads, the 128 drain threads,
      // or one (a TMA transaction or a tcgen05.commit)
      const uint32_t count =
          (i == kBarPReady || i == kBarDSReady || i == kBarAccEmpty) ? 256
          : (i == kBarDQFree)                                          ? 128
          : (i == kBarEpiFull || i == kBarEpiFull + 1)                 ? 256 / Ly::kEpiTurns
                                                                       : 1;
      mbar_init(bar(i), count);
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
    if (FUSED_DQ) tma_prefetch_desc(&tmAcc);
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
    // Per item: V (free once the previous item's last dP is done), K (free
    // once its last dK/dQ is done); per query tile g: dO(g) (its stage is free
    // once the dV of the tile that last held it is done) and Q(g+1) with its
    // L and D vectors (two
    // stages, free once dK(g-1) is done) -- for the last tile of an item,
    // Q(g+1) is the first query tile of the next item.
    auto load_q = [&](int g, int qbh, int qt) {  // elected lane only
      const int s = g & 1;
      mbar_arrive_expect_tx(bar(kBarQFull + s), Ly::kTileBytes + 1024);
#pragma unroll
      for (int cb = 0; cb < HD / 64; ++cb)
        tma_load_3d(sbase + Ly::kQ + s * Ly::kTileBytes + cb * 16384, &tmQ, bar(kBarQFull + s),
                    cb * 64, qt * 128, qbh);
      const size_t vo = size_t(qbh) * Npad + size_t(qt) * 128;
      bulk_load(sbase + Ly::kVec + s * 1024, L2ws + vo, 512, bar(kBarQFull + s));
      bulk_load(sbase + Ly::kVec + s * 1024 + 512, Dws + vo, 512, bar(kBarQFull + s));
    };
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int it0 = CAUSAL ? jt : 0, n_it = item_tiles(jt, bh);
      const int next = snake_item(k + 1, b, G, n_items);
      int njt = 0, nbh = 0;
      if (next >= 0) decode_item(next, njt, nbh);
      if (k > 0 && !(ok = mbar_wait_warp(bar(kBarVEmpty), (k - 1) & 1, ctx, 0x212))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarVFull), Ly::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(sbase + Ly::kV + cb * 16384, &tmV, bar(kBarVFull), cb * 64, jt * 128, bh);
      }
      __syncwarp();
      if (k > 0 && !(ok = mbar_wait_warp(bar(kBarKEmpty), (k - 1) & 1, ctx, 0x213))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarKFull), Ly::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(sbase + Ly::kK + cb * 16384, &tmK, bar(kBarKFull), cb * 64, jt * 128, bh);
        if (k == 0) load_q(0, bh, it0);
        // Warm L2 (and the address translation) for the next item: a new head
        // is often a cold region, and its first tiles are needed right at the
        // item switch.
        if (next >= 0) {
          const int nq = CAUSAL ? njt : 0;
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb) {
            tma_prefetch_3d(&tmK, cb * 64, njt * 128, nbh);
            tma_prefetch_3d(&tmV, cb * 64, njt * 128, nbh);
            tma_prefetch_3d(&tmQ, cb * 64, nq * 128, nbh);
            tma_prefetch_3d(&tmdO, cb * 64, nq * 128, nbh);
          }
          const size_t vo = size_t(nbh) * Npad + size_t(nq) * 128;
          bulk_prefetch(L2ws + vo, 512);
          bulk_prefetch(Dws + vo, 512);
        }
      }
      __syncwarp();
      for (int it = 0; it < n_it; ++it, ++g) {
        const int ds_ = g % Ly::kDOStages, dn = g / Ly::kDOStages;
        if (dn > 0 &&
            !(ok = mbar_wait_warp(bar(kBarDOEmpty + ds_), (dn - 1) & 1, ctx, 0x211)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(kBarDOFull + ds_), Ly::kTileBytes);
#pragma unroll
          for (int cb = 0; cb < HD / 64; ++cb)
            tma_load_3d(sbase + Ly::kDO + ds_ * Ly::kTileBytes + cb * 16384, &tmdO,
                        bar(kBarDOFull + ds_), cb * 64, (it0 + it) * 128, bh);
        }
        __syncwarp();
        int qbh = bh, qt = it0 + it + 1;
        if (it + 1 == n_it) {
          if (next < 0) continue;
          qbh = nbh;
          qt = CAUSAL ? njt : 0;
        }
        const int gn = g + 1;
        if (gn >= 2 &&
            !(ok = mbar_wait_warp(bar(kBarQEmpty + (gn & 1)), ((gn >> 1) - 1) & 1, ctx, 0x210)))
          break;
        if (elect_one()) load_q(gn, qbh, qt);
        __syncwarp();
      }
      item = next;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues.  Every
    // descriptor is a per-tile base plus a compile-time k-step offset.
    constexpr uint32_t kIdS = make_idesc_bf16(128, 128, 0, 0);   // S^T, dP^T
    constexpr uint32_t kIdV = make_idesc_bf16(128, HD, 0, 1);    // dV, dK
    constexpr uint32_t kIdQ = make_idesc_bf16(128, HD, 1, 1);    // dQ = dS K
    const uint64_t dK_k = make_sdesc_sw128(sbase + Ly::kK, 16, 1024);        // K, K-major
    const uint64_t dK_mn = make_sdesc_sw128(sbase + Ly::kK, 16384, 1024);    // K, MN-major
    const uint64_t dV_k = make_sdesc_sw128(sbase + Ly::kV, 16, 1024);
    const uint64_t dS_k = make_sdesc_sw128(sbase + Ly::kDS, 16, 1024);       // dS^T, K-major
    const uint64_t dS_mn = make_sdesc_sw128(sbase + Ly::kDS, 16384, 1024);   // dS, MN-major
    const uint32_t tS = tbase + Ly::kColS, tDP = tbase + Ly::kColDP;
    const uint32_t tDV = tbase + Ly::kColDV, tDK = tbase + Ly::kColDK;
    const uint32_t tDQ = tbase + Ly::kColDQ;
    // Issue order per query tile:  dP, dV, S(next), dQ, dK (d = 128 with dQ;
    // else dK, dQ).  S(next) goes right
    // behind dV (which has consumed P from the S columns; the softmax warps
    // keep P in registers), so the softmax warps compute the next tile's P
    // while the tensor core runs dK and dQ.  The first S of an item waits for
    // its K.
    auto issue_s = [&](int stage) {  // S^T = K Q^T; elected lane only
      const uint64_t dq = make_sdesc_sw128(sbase + Ly::kQ + stage * Ly::kTileBytes, 16, 1024);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
        mma_ss(tS, sdesc_add(dK_k, off), sdesc_add(dq, off), kIdS, k > 0 ? 1u : 0u);
      }
      tc_commit(bar(kBarSFull));
    };
    // d = 128 with dQ: dQ_i = dS K into the dP^T columns (the softmax warps
    // have read them), then dK += dS^T Q, both from the shared dS^T tile.
    // Otherwise dK += dS^T Q with dS^T read from the dP^T columns (packed there
    // by the softmax warps), then (d = 64) dQ_i = dS K into its own columns.
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int n_it = item_tiles(jt, bh);
      if (!(ok = mbar_wait_warp(bar(kBarKFull), k & 1, ctx, 0x220))) break;
      if (!(ok = mbar_wait_warp(bar(kBarQFull + (g & 1)), (g >> 1) & 1, ctx, 0x221))) break;
      tc_fence_after();
      if (elect_one()) issue_s(g & 1);
      __syncwarp();
      if (!(ok = mbar_wait_warp(bar(kBarVFull), k & 1, ctx, 0x227))) break;
      for (int it = 0; it < n_it; ++it, ++g) {
        const int s = g & 1;
        const bool last = it + 1 == n_it;
        const uint32_t sQ = sbase + Ly::kQ + s * Ly::kTileBytes;
        const int ds_ = g % Ly::kDOStages;
        const uint32_t sDO = sbase + Ly::kDO + ds_ * Ly::kTileBytes;
        const uint64_t dQ_mn = make_sdesc_sw128(sQ, 16384, 1024);
        const uint64_t dO_k = make_sdesc_sw128(sDO, 16, 1024);
        const uint64_t dO_mn = make_sdesc_sw128(sDO, 16384, 1024);
        const uint32_t acc0 = it > 0 ? 1u : 0u;
        // dP^T = V dO^T.  When dQ shares the dP columns, they held the previous
        // dQ: wait for its drain.  (Otherwise the previous dP has been read:
        // the softmax warps signalled DS_READY, which the last tile waited on.)
        if (!(ok = mbar_wait_warp(bar(kBarDOFull + ds_), (g / Ly::kDOStages) & 1, ctx, 0x222)))
          break;
        if (FUSED_DQ && !Ly::kSeparateDq && g > 0 &&
            !(ok = mbar_wait_warp(bar(kBarDQFree), (g - 1) & 1, ctx, 0x223)))
          break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tDP, sdesc_add(dV_k, off), sdesc_add(dO_k, off), kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(kBarDPFull));
          if (last) tc_commit(bar(kBarVEmpty));
        }
        __syncwarp();
        // dV += P^T dO, P^T read from tensor memory: query block kk/4 was
        // packed by the softmax warps of that half into its own first 32
        // columns.  The first dV of an item overwrites the accumulator: the
        // previous item's epilogue must have read it.
        if (!(ok = mbar_wait_warp(bar(kBarPReady), g & 1, ctx, 0x224))) break;
        if (it == 0 && k > 0 &&
            !(ok = mbar_wait_warp(bar(kBarAccEmpty), (k - 1) & 1, ctx, 0x228)))
          break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tDV, tS + 64 * (kk >> 2) + 8 * (kk & 3), sdesc_add(dO_mn, kk * 2048), kIdV,
                   kk > 0 ? 1u : acc0);
          tc_commit(bar(kBarDOEmpty + ds_));
        }
        __syncwarp();
        // S of the item's next query tile into the S columns, behind dV
        if (!last) {
          const int s1 = (g + 1) & 1;
          if (!(ok = mbar_wait_warp(bar(kBarQFull + s1), ((g + 1) >> 1) & 1, ctx, 0x226)))
            break;
          tc_fence_after();
          if (elect_one()) issue_s(s1);
          __syncwarp();
        }
        if (!(ok = mbar_wait_warp(bar(kBarDSReady), g & 1, ctx, 0x225))) break;
        tc_fence_after();
        if constexpr (Ly::kDqFirst) {
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tDQ, sdesc_add(dS_mn, kk * 2048), sdesc_add(dK_mn, kk * 2048), kIdQ,
                     kk > 0 ? 1u : 0u);
            tc_commit(bar(kBarDQFull));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_ss(tDK, sdesc_add(dS_k, off), sdesc_add(dQ_mn, kk * 2048), kIdV,
                     kk > 0 ? 1u : acc0);
            }
            tc_commit(bar(kBarQEmpty + s));
          }
          __syncwarp();
        } else {
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // dS^T packed like P^T, in the dP^T columns
              mma_ts(tDK, tDP + 64 * (kk >> 2) + 8 * (kk & 3), sdesc_add(dQ_mn, kk * 2048),
                     kIdV, kk > 0 ? 1u : acc0);
            tc_commit(bar(kBarQEmpty + s));
          }
          __syncwarp();
        }
        if constexpr (FUSED_DQ && !Ly::kDqFirst) {
          // With its own columns, dQ waits only for the previous dQ's drain.
          if (Ly::kSeparateDq && g > 0 &&
              !(ok = mbar_wait_warp(bar(kBarDQFree), (g - 1) & 1, ctx, 0x223)))
            break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tDQ, sdesc_add(dS_mn, kk * 2048), sdesc_add(dK_mn, kk * 2048), kIdQ,
                     kk > 0 ? 1u : 0u);
            tc_commit(bar(kBarDQFull));
          }
          __syncwarp();
        }
        // dK (and dQ) have read the dS^T tile; the item's last tile also
        // releases K and hands the accumulators to the epilogue.
        if (elect_one()) {
          tc_commit(bar(kBarDSFree));
          if (last) {
            tc_commit(bar(kBarKEmpty));
            tc_commit(bar(kBarAccFull));
          }
        }
        __syncwarp();
      }
      item = snake_item(k + 1, b, G, n_items);
    }
    if (elect_one()) tc_commit(bar(kBarDrain));
    __syncwarp();
    volatile int never = 0;  // this wait ignores the CTA abort flag
    const WaitCtx own{&never, err, kWaitLimitNs};
    mbar_wait_warp(bar(kBarDrain), 0, own, 0x22F);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS
    const int h = (warp - 4) >> 2;       // query half: columns 64h .. 64h+63
    const int r = threadIdx.x & 127;     // key row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + Ly::kColS + 64 * h;
    const uint32_t tDP = tbase + lane_off + Ly::kColDP + 64 * h;
    const uint32_t sDSrow = sbase + Ly::kDS + h * 16384 + r * 128;
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int it0 = CAUSAL ? jt : 0, n_it = item_tiles(jt, bh);
      const int doc_edge = MASK == kMaskDocument ? items[size_t(bh) * n_tiles + jt].y : n_tiles;
      // with documents: this thread's key jt*128 + r is seen by queries below
      // q_lim only (the end of its document, and of the window)
      int q_lim = N;
      if (MASK == kMaskDocument) {
        const int kg = jt * 128 + r;
        q_lim = qend[size_t(bh) * Npad + kg];
        if (window > 0 && kg + window < q_lim) q_lim = kg + window;
      }
      for (int it = 0; it < n_it; ++it, ++g) {
        const int s = g & 1, qt = it0 + it;
        if (!(ok = mbar_wait_warp(bar(kBarQFull + s), (g >> 1) & 1, ctx, 0x230))) break;
        if (!(ok = mbar_wait_warp(bar(kBarSFull), g & 1, ctx, 0x231))) break;
        tc_fence_after();
        const float* L2v = reinterpret_cast<const float*>(smem + Ly::kVec + s * 1024) + 64 * h;
        const float* Dv =
            reinterpret_cast<const float*>(smem + Ly::kVec + s * 1024 + 512) + 64 * h;
        // P stays in registers (packed bf16) for the dS phase: the tensor
        // core overwrites these S columns with the next S once dV has read it.
        uint32_t pk[32];
        {
          uint32_t u[64];
          tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
          tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          tmem_wait_ld();
          const bool diag = CAUSAL && qt == jt;
          // key rows past N (the zero-filled tail of the last tile) get P = 0:
          // their K and V rows are zero, and 2^(-L) must not reach dS
          const bool dead_key = jt * 128 + r >= N;
          // sliding window: query column q of this tile sees key row r only
          // while (qt - jt) * 128 + q - r < window
          const int dq_tile = (qt - jt) * 128;
          const bool wedge = MASK == kMaskWindow && CAUSAL && window > 0 && dq_tile + 127 >= window;
          // documents (and a window with them): from the tabulated first query
          // tile on, some query columns cannot see every key of the tile
          const bool dedge = MASK == kMaskDocument && qt >= doc_edge;
          const float4* L2v4 = reinterpret_cast<const float4*>(L2v);
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 l = L2v4[c4];  // one broadcast load for four query columns
            // y = L - s scale log2e for two columns per instruction; P = 2^-y
            float y0, y1, y2, y3;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(u[4 * c4]), __uint_as_float(u[4 * c4 + 1])),
                                  f32x2(-scale_log2, -scale_log2), f32x2(l.x, l.y)),
                        y0, y1);
            f32x2_split(
                fma_f32x2(f32x2(__uint_as_float(u[4 * c4 + 2]), __uint_as_float(u[4 * c4 + 3])),
                          f32x2(-scale_log2, -scale_log2), f32x2(l.z, l.w)),
                y2, y3);
            float p0 = ex2(-y0), p1 = ex2(-y1), p2 = ex2(-y2), p3 = ex2(-y3);
            if (diag) {  // key row r is visible to query columns >= r only
              const int q0 = 64 * h + 4 * c4;
              if (q0 < r) p0 = 0.f;
              if (q0 + 1 < r) p1 = 0.f;
              if (q0 + 2 < r) p2 = 0.f;
              if (q0 + 3 < r) p3 = 0.f;
            }
            if (wedge) {
              const int dq0 = dq_tile + 64 * h + 4 * c4 - r;
              if (dq0 >= window) p0 = 0.f;
              if (dq0 + 1 >= window) p1 = 0.f;
              if (dq0 + 2 >= window) p2 = 0.f;
              if (dq0 + 3 >= window) p3 = 0.f;
            }
            if (dedge) {  // query columns at or past q_lim cannot see this key
              const int q0 = qt * 128 + 64 * h + 4 * c4;
              if (q0 >= q_lim) p0 = 0.f;
              if (q0 + 1 >= q_lim) p1 = 0.f;
              if (q0 + 2 >= q_lim) p2 = 0.f;
              if (q0 + 3 >= q_lim) p3 = 0.f;
            }
            pk[2 * c4] = pack_bf16x2(p0, p1);
            pk[2 * c4 + 1] = pack_bf16x2(p2, p3);
          }
          if (dead_key) {  // only in the last, ragged key tile
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = 0u;
          }
          tmem_st32(tS, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kBarPReady));
        }
        if (!(ok = mbar_wait_warp(bar(kBarDPFull), g & 1, ctx, 0x232))) break;
        // dQ reads dS from the shared-memory tile: the previous one must be done,
        // and at an item's first tile so must the previous item's epilogue
        if (FUSED_DQ && g > 0 &&
            !(ok = mbar_wait_warp(bar(kBarDSFree), (g - 1) & 1, ctx, 0x233)))
          break;
        if (FUSED_DQ && it == 0 && k > 0 &&
            !(ok = mbar_wait_warp(bar(kBarEpiFree + Ly::kEpiTurns - 1), (k - 1) & 1, ctx,
                                  0x234)))
          break;
        tc_fence_after();
        {
          const float4* Dv4 = reinterpret_cast<const float4*>(Dv);
          // two 32-column chunks of dP^T.  Where dK reads it from tensor memory,
          // dS^T goes back into the dP^T columns this warp has read, packed two
          // queries per column as P^T is; with dQ, into row r of the shared
          // dS^T tile (128-byte swizzle: 16-byte chunk c lands at c ^ (r % 8)).
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t u[32];
            tmem_ld32(tDP + 32 * ch, u);
            tmem_wait_ld();
            // dS = P o (dP - D): the difference in fp32, packed once to
            // bf16x2, times the packed bf16 P with one bf16x2 multiply per pair.
            uint32_t ds[16];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 dd = Dv4[8 * ch + c4];  // one broadcast load for four columns
              // dP - D for two columns per instruction (a product by -1 is exact)
              float e0, e1, e2, e3;
              f32x2_split(fma_f32x2(f32x2(dd.x, dd.y), f32x2(-1.f, -1.f),
                                    f32x2(__uint_as_float(u[4 * c4]), __uint_as_float(u[4 * c4 + 1]))),
                          e0, e1);
              f32x2_split(
                  fma_f32x2(f32x2(dd.z, dd.w), f32x2(-1.f, -1.f),
                            f32x2(__uint_as_float(u[4 * c4 + 2]), __uint_as_float(u[4 * c4 + 3]))),
                  e2, e3);
              ds[2 * c4] = mul_bf16x2(pk[16 * ch + 2 * c4], pack_bf16x2(e0, e1));
              ds[2 * c4 + 1] = mul_bf16x2(pk[16 * ch + 2 * c4 + 1], pack_bf16x2(e2, e3));
            }
            if constexpr (!Ly::kDqFirst) tmem_st16(tDP + 16 * ch, ds);
            if constexpr (FUSED_DQ) {
#pragma unroll
              for (int c = 0; c < 4; ++c)
                st_shared_v4(sDSrow + (((4 * ch + c) ^ (r & 7)) << 4), ds[4 * c], ds[4 * c + 1],
                             ds[4 * c + 2], ds[4 * c + 3]);
            }
          }
          tmem_wait_st();
          if constexpr (FUSED_DQ) fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(bar(kBarDSReady));
        }
      }
      if (!ok) break;
      // Epilogue of the item: dV (half 0) and dK (half 1, times the softmax
      // scale) from tensor memory, rounded to bf16 into the shared dS^T tile
      // (its two 16 KB blocks are the 64-column boxes of the output tile map,
      // with the same 128-byte swizzle) and written by TMA tile stores, which
      // leave out the rows past N.  One elected warp per turn issues them;
      // their shared-memory reads complete before the tile is used again.
      if (!(ok = mbar_wait_warp(bar(kBarAccFull), k & 1, ctx, 0x238 + h))) break;
      tc_fence_after();
      const uint32_t tAcc = tbase + lane_off + (h == 0 ? Ly::kColDV : Ly::kColDK);
      const float mult = h == 0 ? 1.f : scale;
      for (int turn = 0; ok && turn < Ly::kEpiTurns; ++turn) {
        if (Ly::kEpiTurns == 1 || h == turn) {
          // The tile's previous contents: this item's dS^T (the contractions
          // have completed: AccFull), then the previous turn's store -- of this
          // item for turn 1, of the previous item for turn 0.
          const int prev_turn = turn > 0 ? turn - 1 : Ly::kEpiTurns - 1;
          const int prev_item = turn > 0 ? k : k - 1;
          if (prev_item >= 0 &&
              !(ok = mbar_wait_warp(bar(kBarEpiFree + prev_turn), prev_item & 1, ctx, 0x23A)))
            break;
          const uint32_t row = sbase + Ly::kDS + (HD == 64 ? h * 16384 : 0) + r * 128;
#pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t o[32];
            tmem_ld32(tAcc + 32 * c4, o);
            tmem_wait_ld();
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {  // 16-byte chunk j of 64-column block c4 / 2
              const int j = 4 * (c4 & 1) + c8;
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16x2(__uint_as_float(o[8 * c8 + 2 * e]) * mult,
                                    __uint_as_float(o[8 * c8 + 2 * e + 1]) * mult);
              st_shared_v4(row + (c4 >> 1) * 16384 + ((j ^ (r & 7)) << 4), w4[0], w4[1], w4[2],
                           w4[3]);
            }
          }
          tc_fence_before();
          mbar_arrive(bar(kBarAccEmpty));  // this thread's accumulator columns are read
          fence_proxy_async_smem();
          mbar_arrive(bar(kBarEpiFull + turn));
        }
        if (warp == 4 + 4 * (Ly::kEpiTurns == 2 ? turn : 0)) {  // the turn's issuing warp
          if (!(ok = mbar_wait_warp(bar(kBarEpiFull + turn), k & 1, ctx, 0x23B))) break;
          if (elect_one()) {
            if constexpr (HD == 128) {
              const CUtensorMap* map = turn == 0 ? &tmDV : &tmDK;
              tma_store_3d(map, sbase + Ly::kDS, 0, jt * 128, bh);
              tma_store_3d(map, sbase + Ly::kDS + 16384, 64, jt * 128, bh);
            } else {
              tma_store_3d(&tmDV, sbase + Ly::kDS, 0, jt * 128, bh);
              tma_store_3d(&tmDK, sbase + Ly::kDS + 16384, 0, jt * 128, bh);
            }
            bulk_commit_group();
            bulk_wait_group_read<0>();
            mbar_arrive(bar(kBarEpiFree + turn));
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      item = snake_item(k + 1, b, G, n_items);
    }
    bulk_wait_group_all();  // the epilogue's stores complete before the CTA retires
  } else if (FUSED_DQ) {
    // ------------------------------------------------------------ dQ drain
    // Tensor memory -> registers -> swizzled fp32 staging tile -> TMA
    // reduce-add into the accumulator, 32 columns (16 KB) per box, two
    // staging buffers.  Thread 0 issues the reductions and owns their groups.
    const int r = threadIdx.x;  // query row within the tile = TMEM lane
    const uint32_t tDQ = tbase + (uint32_t(warp * 32) << 16) + Ly::kColDQ;
    const bool issuer = threadIdx.x == 0;
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int it0 = CAUSAL ? jt : 0, n_it = item_tiles(jt, bh);
      for (int it = 0; it < n_it; ++it, ++g) {
        const int qt = it0 + it;
        // The four drain warps agree before any named barrier below, so that a
        // wait that gave up in one warp stops all of them.
        const bool got = mbar_wait_warp(bar(kBarDQFull), g & 1, ctx, 0x240);
        if (!(ok = named_barrier_and(kDrainBarrierId, 128, got))) break;
        tc_fence_after();
        // 32-column chunks.  For d = 128, chunks 0-2 are loaded, chunk 0
        // staged, chunk 3 loaded into chunk 0's registers, and only then are
        // the columns released to the MMA warp (the register budget does not
        // hold all four).
        auto stage = [&](int c, const uint32_t (&v)[32]) {
          const uint32_t buf = sbase + Ly::kStage + (c & 1) * 16384;
          // the reduction that last read this buffer (two boxes ago) is done
          if (issuer) bulk_wait_group_read<1>();
          named_barrier_sync(kDrainBarrierId, 128);
          const uint32_t row = buf + r * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(row + ((j ^ (r & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                         v[4 * j + 3]);
          fence_proxy_async_smem();
          named_barrier_sync(kDrainBarrierId, 128);
          if (issuer) {
            tma_reduce_add_2d(&tmAcc, buf, 32 * c, bh * Npad + qt * 128);
            bulk_commit_group();
          }
        };
        uint32_t a0[32], a1[32];
        tmem_ld32(tDQ, a0);
        tmem_ld32(tDQ + 32, a1);
        if constexpr (HD == 128) {
          uint32_t a2[32];
          tmem_ld32(tDQ + 64, a2);
          tmem_wait_ld();
          stage(0, a0);
          tmem_ld32(tDQ + 96, a0);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(kBarDQFree));
          stage(1, a1);
          stage(2, a2);
          stage(3, a0);
        } else {
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(kBarDQFree));
          stage(0, a0);
          stage(1, a1);
        }
      }
      item = snake_item(k + 1, b, G, n_items);
    }
    if (issuer) bulk_wait_group_all();  // reductions complete before the CTA retires
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

// Streaming multiprocessors of the current device (cached per device).
static int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// L2 size of the current device in bytes (cached per device).
static size_t l2_bytes() {
  static size_t cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return size_t(32) << 20;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0)
      n = 32 << 20;
    cached[dev] = size_t(n);
  }
  return cached[dev];
}

// Heads per work-item group: as many as keep the group's Q, dO (bf16) and,
// when the kernel reduces dQ, the dQ accumulator (fp32) -- 8 bytes per
// element of a head, else 4 -- within half the L2.
// Without the mask every item of a head walks all its query tiles, so
// grouping turns most Q/dO reads into L2 hits (measured +13% at N = 8192,
// d = 128).  Under the causal mask, grouping measured slower (-4 to -9%):
// all heads form one group there, and the order stays heaviest first.
static int head_group(const Shape& s, int bytes_per_element) {
  if (s.causal) return s.BH;
  const size_t per_head = size_t(s.Npad) * s.d * bytes_per_element;
  size_t hg = (l2_bytes() / 2) / per_head;
  if (hg < 1) hg = 1;
  if (hg > size_t(s.BH)) hg = size_t(s.BH);
  return int(hg);
}

template <int HD, bool CAUSAL, int MASK, bool FUSED_DQ>
static cudaError_t launch_main_t(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                 const CUtensorMap& tmAcc, void* dK, void* dV,
                                 const Workspace& ws, const Shape& s, float scale, int* err,
                                 cudaStream_t stream) {
  using Ly = Layout<HD, FUSED_DQ>;
  auto kern = attn_bwd_main_kernel<HD, CAUSAL, MASK, FUSED_DQ>;
  cudaError_t e =
      set_smem_limit_once<attn_bwd_main_kernel<HD, CAUSAL, MASK, FUSED_DQ>>(Ly::kBytes);
  if (e != cudaSuccess) return e;
  // dK and dV are written by TMA tile stores: [BH][N][d] bf16, like Q.
  CUtensorMap tmDK, tmDV;
  if (make_tile_map(&tmDK, dK, s) || make_tile_map(&tmDV, dV, s)) return cudaErrorInvalidValue;
  // Persistent grid: at most one CTA per SM, each walking its work items.
  const long long n_items = (long long)s.n_tiles * s.BH;
  const dim3 grid(unsigned(n_items < num_sms() ? n_items : num_sms()));
  return launch_kernel(kern, grid, dim3(kThreads), Ly::kBytes, stream, tmQ, tmK, tmV, tmdO, tmAcc,
                       tmDK, tmDV, ws.L2, ws.D, s.BH, s.N,
                       head_group(s, FUSED_DQ ? 8 : 4), s.window, s.doc, s.H,
                       static_cast<const int2*>(ws.items), static_cast<const int*>(ws.qend),
                       static_cast<const int*>(ws.order), scale, scale * 1.4426950408889634f,
                       err);
}

// The main kernel's instantiation for a validated shape: head dim, mask and
// whether it also reduces dQ (FUSED_DQ) or leaves dQ to the separate pass.
template <bool FUSED_DQ>
static cudaError_t launch_main_any(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                   const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                   const CUtensorMap& tmAcc, void* dK, void* dV,
                                   const Workspace& ws, const Shape& s, float scale, int* err,
                                   cudaStream_t stream) {
  const int mask = !s.causal ? kMaskPlain
                   : s.doc        ? kMaskDocument
                   : s.window > 0 ? kMaskWindow
                                  : kMaskPlain;
#define ATTN_MAIN(HD_, C_, M_)                                                               \
  launch_main_t<HD_, C_, M_, FUSED_DQ>(tmQ, tmK, tmV, tmdO, tmAcc, dK, dV, ws, s, scale, err, \
                                       stream)
  if (s.d == 64) {
    if (!s.causal) return ATTN_MAIN(64, false, kMaskPlain);
    if (mask == kMaskDocument) return ATTN_MAIN(64, true, kMaskDocument);
    if (mask == kMaskWindow) return ATTN_MAIN(64, true, kMaskWindow);
    return ATTN_MAIN(64, true, kMaskPlain);
  }
  if (!s.causal) return ATTN_MAIN(128, false, kMaskPlain);
  if (mask == kMaskDocument) return ATTN_MAIN(128, true, kMaskDocument);
  if (mask == kMaskWindow) return ATTN_MAIN(128, true, kMaskWindow);
  return ATTN_MAIN(128, true, kMaskPlain);
#undef ATTN_MAIN
}

}  // namespace bwd
}  // namespace attn
