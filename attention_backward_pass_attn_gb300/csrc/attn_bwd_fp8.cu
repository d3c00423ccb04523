// attn_bwd_fp8.cu -- the exact-attention backward with 8-bit (e4m3) operands
// on the fifth-generation tensor core (tcgen05.mma kind::f8f6f4).
//
// The fp8 extension that "Training Transformers and Hybrid models on AMD
// Instinct MI300X Accelerators" (section "Summary") names as the next step for
// its attention kernel, for the backward: Q, K, V and dO arrive as e4m3 bytes
// with one fp32 descale factor each, and all five contractions per tile pair
// run on 8-bit operands with fp32 accumulation:
//
//   S^T  = K8 Q8^T                     (scores, scaled by s qd kd)
//   P^T  = exp(S^T - L)  -> e4m3(256 P^T) in tensor memory
//   dP^T = V8 dO8^T                    (scaled by vd dod)
//   dV  += (256 P)^T dO8               -> dV = acc dod / 256
//   dS^T = P^T o (dP^T - D)  -> e4m3(ds_scale dS^T) in shared memory
//   dK  += (ds_scale dS)^T Q8          -> dK = acc s qd / ds_scale
//   dQ_i = (ds_scale dS) K8            -> fp32 accumulator (TMA reduce-add),
//                                         dQ = acc s kd / ds_scale
//
// dS spans a wider range than P (it carries dP - D), so its 8-bit rounding
// uses a scale the caller supplies -- the delayed scaling of fp8 training:
// the kernel reports the largest |dS| it met (ds_amax), from which the
// caller derives the next call's scale.  P is scaled by 256: P <= 1 (L is
// the exact log-sum-exp), so 256 P stays below e4m3's 448 and its normal
// range covers probabilities down to 2^-14.
//
// Design: the bf16 backward main kernel's (attn_bwd_main.cuh) -- persistent
// CTAs walking (head, 128-row key/value tile) items, warps 0-3 draining dQ,
// warps 4-11 forming P and dS (one key row per thread), warp 12 issuing TMA
// and warp 13 tcgen05.mma -- with 8-bit tiles: a 128 x 128 e4m3 tile is one
// 16 KB block of 128-byte-swizzled rows, an MMA takes K = 32, P^T goes to
// tensor memory four values per 32-bit column, and the dS^T tile is one 16 KB
// block read K-major for dK and MN-major for dQ.  Head dim 128; the causal
// mask or none.

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace bwd8 {

constexpr int kThreads = 448;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;
constexpr int HD = 128;
constexpr int kTile = 128 * HD;  // one 128 x 128 e4m3 tile: 16 KB
constexpr float kPScale = 256.f;

constexpr int kBarKFull = 0;
constexpr int kBarVFull = 1;
constexpr int kBarKEmpty = 2;
constexpr int kBarVEmpty = 3;
constexpr int kBarAccFull = 4;
constexpr int kBarAccEmpty = 5;
constexpr int kBarQFull = 6;    // + stage
constexpr int kBarQEmpty = 8;   // + stage
constexpr int kBarDOFull = 10;  // + stage
constexpr int kBarDOEmpty = 12; // + stage
constexpr int kBarSFull = 14;
constexpr int kBarPReady = 15;
constexpr int kBarDPFull = 16;
constexpr int kBarDSReady = 17;
constexpr int kBarDSFree = 18;
constexpr int kBarDQFull = 19;
constexpr int kBarDQFree = 20;
constexpr int kBarDrain = 21;
constexpr int kNumBars = 22;
constexpr int kDrainBarrierId = 1;

struct Layout {
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;        // + stage * kTile
  static constexpr int kDO = kQ + 2 * kTile;   // + stage * kTile
  static constexpr int kDS = kDO + 2 * kTile;  // 128 x 128 e4m3
  static constexpr int kStage = kDS + kTile;   // 2 x (128 rows x 32 fp32), swizzled
  static constexpr int kVec = kStage + 32768;  // stage s: L2 at +1024 s, D at +1024 s + 512
  static constexpr int kBar = kVec + 2048;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kRaw = (kAbort + 4 + 15) / 16 * 16;
  static constexpr int kBytes = kRaw > 118784 ? kRaw : 118784;
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = HD;
  static constexpr uint32_t kColS = 2 * HD;
  static constexpr uint32_t kColDP = 2 * HD + 128;
  static constexpr uint32_t kColDQ = kColDP;  // dQ reuses the dP columns once read
};

__device__ __forceinline__ int snake_item(int k, int b, int G, int n_items) {
  const int idx = (k & 1) ? k * G + (G - 1 - b) : k * G + b;
  return idx < n_items ? idx : -1;
}

// Descriptors: 128-byte swizzle, one 16 KB block per 128 x 128 e4m3 tile.
// K-major: +32 bytes per 32-element k-step; MN-major: +4 KB (32 rows).

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmdO,
                        const __grid_constant__ CUtensorMap tmAcc, const float* __restrict__ L2ws,
                        const float* __restrict__ Dws, __nv_bfloat16* __restrict__ dK,
                        __nv_bfloat16* __restrict__ dV, int BH, int N, int head_group,
                        float score_log2, float dp_mult, float ds_scale, float dk_mult,
                        float dv_mult, float* __restrict__ ds_amax, int* err) {
  using Ly = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(err, kDevSmemAlign, 0x500);
    return;
  }
  const int n_tiles = (N + 127) >> 7;
  const int Npad = n_tiles * 128;
  const int n_items = BH * n_tiles;
  // items: groups of head_group heads, key/value-tile major within a group
  auto decode_item = [&](int i, int& jt, int& bh) {
    const int per_group = head_group * n_tiles;
    const int gr = i / per_group, r = i - gr * per_group;
    const int hg = BH - gr * head_group < head_group ? BH - gr * head_group : head_group;
    jt = r / hg;
    bh = gr * head_group + (r - jt * hg);
  };
  auto item_tiles = [&](int jt) { return n_tiles - (CAUSAL ? jt : 0); };
  const int G = gridDim.x, b = blockIdx.x;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sbase + Ly::kBar + 8 * i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kNumBars; ++i) {
      const uint32_t count =
          (i == kBarPReady || i == kBarDSReady || i == kBarAccEmpty) ? 256
          : (i == kBarDQFree)                                          ? 128
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
    tma_prefetch_desc(&tmAcc);
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
    auto load_q = [&](int g, int qbh, int qt) {  // elected lane only
      const int s = g & 1;
      mbar_arrive_expect_tx(bar(kBarQFull + s), kTile + 1024);
      tma_load_3d(sbase + Ly::kQ + s * kTile, &tmQ, bar(kBarQFull + s), 0, qt * 128, qbh);
      const size_t vo = size_t(qbh) * Npad + size_t(qt) * 128;
      bulk_load(sbase + Ly::kVec + s * 1024, L2ws + vo, 512, bar(kBarQFull + s));
      bulk_load(sbase + Ly::kVec + s * 1024 + 512, Dws + vo, 512, bar(kBarQFull + s));
    };
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int it0 = CAUSAL ? jt : 0, n_it = item_tiles(jt);
      const int next = snake_item(k + 1, b, G, n_items);
      int njt = 0, nbh = 0;
      if (next >= 0) decode_item(next, njt, nbh);
      if (k > 0 && !(ok = mbar_wait_warp(bar(kBarVEmpty), (k - 1) & 1, ctx, 0x512))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarVFull), kTile);
        tma_load_3d(sbase + Ly::kV, &tmV, bar(kBarVFull), 0, jt * 128, bh);
      }
      __syncwarp();
      if (k > 0 && !(ok = mbar_wait_warp(bar(kBarKEmpty), (k - 1) & 1, ctx, 0x513))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(kBarKFull), kTile);
        tma_load_3d(sbase + Ly::kK, &tmK, bar(kBarKFull), 0, jt * 128, bh);
        if (k == 0) load_q(0, bh, it0);
      }
      __syncwarp();
      for (int it = 0; it < n_it; ++it, ++g) {
        const int ds_ = g & 1, dn = g >> 1;
        if (dn > 0 && !(ok = mbar_wait_warp(bar(kBarDOEmpty + ds_), (dn - 1) & 1, ctx, 0x511)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(kBarDOFull + ds_), kTile);
          tma_load_3d(sbase + Ly::kDO + ds_ * kTile, &tmdO, bar(kBarDOFull + ds_), 0,
                      (it0 + it) * 128, bh);
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
            !(ok = mbar_wait_warp(bar(kBarQEmpty + (gn & 1)), ((gn >> 1) - 1) & 1, ctx, 0x510)))
          break;
        if (elect_one()) load_q(gn, qbh, qt);
        __syncwarp();
      }
      item = next;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = make_idesc_e4m3(128, 128, 0, 0);  // S^T, dP^T
    constexpr uint32_t kIdV = make_idesc_e4m3(128, HD, 0, 1);   // dV, dK
    constexpr uint32_t kIdQ = make_idesc_e4m3(128, HD, 1, 1);   // dQ = dS K
    const uint64_t dK_k = make_sdesc_sw128(sbase + Ly::kK, 16, 1024);
    const uint64_t dK_mn = make_sdesc_sw128(sbase + Ly::kK, 16384, 1024);
    const uint64_t dV_k = make_sdesc_sw128(sbase + Ly::kV, 16, 1024);
    const uint64_t dS_k = make_sdesc_sw128(sbase + Ly::kDS, 16, 1024);
    const uint64_t dS_mn = make_sdesc_sw128(sbase + Ly::kDS, 16384, 1024);
    const uint32_t tS = tbase + Ly::kColS, tDP = tbase + Ly::kColDP;
    const uint32_t tDV = tbase + Ly::kColDV, tDK = tbase + Ly::kColDK;
    const uint32_t tDQ = tbase + Ly::kColDQ;
    auto issue_s = [&](int stage) {  // S^T = K Q^T; elected lane only
      const uint64_t dq = make_sdesc_sw128(sbase + Ly::kQ + stage * kTile, 16, 1024);
#pragma unroll
      for (int k = 0; k < HD / 32; ++k)
        mma_ss_f8(tS, sdesc_add(dK_k, k * 32), sdesc_add(dq, k * 32), kIdS, k > 0 ? 1u : 0u);
      tc_commit(bar(kBarSFull));
    };
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int n_it = item_tiles(jt);
      if (!(ok = mbar_wait_warp(bar(kBarKFull), k & 1, ctx, 0x520))) break;
      if (!(ok = mbar_wait_warp(bar(kBarQFull + (g & 1)), (g >> 1) & 1, ctx, 0x521))) break;
      tc_fence_after();
      if (elect_one()) issue_s(g & 1);
      __syncwarp();
      if (!(ok = mbar_wait_warp(bar(kBarVFull), k & 1, ctx, 0x527))) break;
      for (int it = 0; it < n_it; ++it, ++g) {
        const int s = g & 1;
        const bool last = it + 1 == n_it;
        const uint32_t sQ = sbase + Ly::kQ + s * kTile;
        const uint32_t sDO = sbase + Ly::kDO + s * kTile;
        const uint64_t dQ_mn = make_sdesc_sw128(sQ, 16384, 1024);
        const uint64_t dO_k = make_sdesc_sw128(sDO, 16, 1024);
        const uint64_t dO_mn = make_sdesc_sw128(sDO, 16384, 1024);
        const uint32_t acc0 = it > 0 ? 1u : 0u;
        if (!(ok = mbar_wait_warp(bar(kBarDOFull + s), (g >> 1) & 1, ctx, 0x522))) break;
        // dP^T reuses the columns of the previous dQ: wait for its drain
        if (g > 0 && !(ok = mbar_wait_warp(bar(kBarDQFree), (g - 1) & 1, ctx, 0x523))) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < HD / 32; ++kk)
            mma_ss_f8(tDP, sdesc_add(dV_k, kk * 32), sdesc_add(dO_k, kk * 32), kIdS,
                      kk > 0 ? 1u : 0u);
          tc_commit(bar(kBarDPFull));
          if (last) tc_commit(bar(kBarVEmpty));
        }
        __syncwarp();
        // dV += (256 P)^T dO: query block kk/2 was packed by the softmax warps
        // of that half into the first 16 columns of its 64.
        if (!(ok = mbar_wait_warp(bar(kBarPReady), g & 1, ctx, 0x524))) break;
        if (it == 0 && k > 0 &&
            !(ok = mbar_wait_warp(bar(kBarAccEmpty), (k - 1) & 1, ctx, 0x528)))
          break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_f8(tDV, tS + 64 * (kk >> 1) + 8 * (kk & 1), sdesc_add(dO_mn, kk * 4096), kIdV,
                      kk > 0 ? 1u : acc0);
          tc_commit(bar(kBarDOEmpty + s));
        }
        __syncwarp();
        if (!last) {
          const int s1 = (g + 1) & 1;
          if (!(ok = mbar_wait_warp(bar(kBarQFull + s1), ((g + 1) >> 1) & 1, ctx, 0x526)))
            break;
          tc_fence_after();
          if (elect_one()) issue_s(s1);
          __syncwarp();
        }
        if (!(ok = mbar_wait_warp(bar(kBarDSReady), g & 1, ctx, 0x525))) break;
        tc_fence_after();
        if (elect_one()) {
          // dQ first: its drain (which frees the dP^T columns for the next
          // tile) then overlaps dK's contraction
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dQ = dS K
            mma_ss_f8(tDQ, sdesc_add(dS_mn, kk * 4096), sdesc_add(dK_mn, kk * 4096), kIdQ,
                      kk > 0 ? 1u : 0u);
          tc_commit(bar(kBarDQFull));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dK += dS^T Q
            mma_ss_f8(tDK, sdesc_add(dS_k, kk * 32), sdesc_add(dQ_mn, kk * 4096), kIdV,
                      kk > 0 ? 1u : acc0);
          tc_commit(bar(kBarQEmpty + s));
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
    volatile int never = 0;
    const WaitCtx own{&never, err, kWaitLimitNs};
    mbar_wait_warp(bar(kBarDrain), 0, own, 0x52F);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P and dS
    const int h = (warp - 4) >> 2;    // query half: columns 64h .. 64h+63
    const int r = threadIdx.x & 127;  // key row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + Ly::kColS + 64 * h;
    const uint32_t tDP = tbase + lane_off + Ly::kColDP + 64 * h;
    const uint32_t sDSrow = sbase + Ly::kDS + r * 128;
    float amax = 0.f;  // the largest |dS| this thread forms
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int it0 = CAUSAL ? jt : 0, n_it = item_tiles(jt);
      for (int it = 0; it < n_it; ++it, ++g) {
        const int s = g & 1, qt = it0 + it;
        if (!(ok = mbar_wait_warp(bar(kBarQFull + s), (g >> 1) & 1, ctx, 0x530))) break;
        if (!(ok = mbar_wait_warp(bar(kBarSFull), g & 1, ctx, 0x531))) break;
        tc_fence_after();
        const float* L2v = reinterpret_cast<const float*>(smem + Ly::kVec + s * 1024) + 64 * h;
        const float* Dv =
            reinterpret_cast<const float*>(smem + Ly::kVec + s * 1024 + 512) + 64 * h;
        // P^T in registers (packed bf16) for dS; 256 P^T in e4m3 to tensor memory
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
          uint32_t p8[16];
          const float4* L2v4 = reinterpret_cast<const float4*>(L2v);
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 l = L2v4[c4];
            float p0 = ex2(fmaf(__uint_as_float(u[4 * c4]), score_log2, -l.x));
            float p1 = ex2(fmaf(__uint_as_float(u[4 * c4 + 1]), score_log2, -l.y));
            float p2 = ex2(fmaf(__uint_as_float(u[4 * c4 + 2]), score_log2, -l.z));
            float p3 = ex2(fmaf(__uint_as_float(u[4 * c4 + 3]), score_log2, -l.w));
            if (diag) {  // key row r is visible to query columns >= r only
              const int q0 = 64 * h + 4 * c4;
              if (q0 < r) p0 = 0.f;
              if (q0 + 1 < r) p1 = 0.f;
              if (q0 + 2 < r) p2 = 0.f;
              if (q0 + 3 < r) p3 = 0.f;
            }
            pk[2 * c4] = pack_bf16x2(p0, p1);
            pk[2 * c4 + 1] = pack_bf16x2(p2, p3);
            p8[c4] = pack_e4m3x4(p0 * kPScale, p1 * kPScale, p2 * kPScale, p3 * kPScale);
          }
          if (dead_key) {  // only in the last, ragged key tile
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = 0u;
#pragma unroll
            for (int c = 0; c < 16; ++c) p8[c] = 0u;
          }
          tmem_st16(tS, p8);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kBarPReady));
        }
        if (!(ok = mbar_wait_warp(bar(kBarDPFull), g & 1, ctx, 0x532))) break;
        if (g > 0 && !(ok = mbar_wait_warp(bar(kBarDSFree), (g - 1) & 1, ctx, 0x533))) break;
        tc_fence_after();
        {
          const float4* Dv4 = reinterpret_cast<const float4*>(Dv);
          // two 32-column chunks of dP^T; this half's 64 bytes of row r of the
          // dS^T tile are 16-byte chunks 4h .. 4h+3, chunk c landing at c ^ (r % 8)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t u[32];
            tmem_ld32(tDP + 32 * ch, u);
            tmem_wait_ld();
            uint32_t q8[8];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 dd = Dv4[8 * ch + c4];
              float ds[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint32_t pw = pk[16 * ch + 2 * c4 + (e >> 1)];
                const float p = (e & 1) ? bf16hi_to_f32(pw) : bf16lo_to_f32(pw);
                const float dv = e == 0 ? dd.x : (e == 1 ? dd.y : (e == 2 ? dd.z : dd.w));
                ds[e] = p * fmaf(__uint_as_float(u[4 * c4 + e]), dp_mult, -dv);
                amax = fmaxf(amax, fabsf(ds[e]));
              }
              q8[c4] = pack_e4m3x4(ds[0] * ds_scale, ds[1] * ds_scale, ds[2] * ds_scale,
                                   ds[3] * ds_scale);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c)
              st_shared_v4(sDSrow + (((4 * h + 2 * ch + c) ^ (r & 7)) << 4), q8[4 * c],
                           q8[4 * c + 1], q8[4 * c + 2], q8[4 * c + 3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(bar(kBarDSReady));
        }
      }
      if (!ok) break;
      // epilogue of the item: half 0 writes dV, half 1 writes dK
      if (!(ok = mbar_wait_warp(bar(kBarAccFull), k & 1, ctx, 0x538 + h))) break;
      tc_fence_after();
      const int kv = jt * 128 + r;
      const uint32_t tAcc = tbase + lane_off + (h == 0 ? Ly::kColDV : Ly::kColDK);
      const float mult = h == 0 ? dv_mult : dk_mult;
      __nv_bfloat16* orow = (h == 0 ? dV : dK) + (size_t(bh) * N + kv) * HD;
#pragma unroll
      for (int c4 = 0; c4 < HD / 32; ++c4) {
        uint32_t o[32];
        tmem_ld32(tAcc + 32 * c4, o);
        tmem_wait_ld();
        if (kv < N) {
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
      tc_fence_before();
      mbar_arrive(bar(kBarAccEmpty));
      item = snake_item(k + 1, b, G, n_items);
    }
    // the largest |dS| of the warp into the caller's word (non-negative
    // floats order like their bit patterns)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0 && ds_amax)
      atomicMax(reinterpret_cast<unsigned int*>(ds_amax), __float_as_uint(amax));
  } else {
    // ------------------------------------------------------------ dQ drain
    const int r = threadIdx.x;
    const uint32_t tDQ = tbase + (uint32_t(warp * 32) << 16) + Ly::kColDQ;
    const bool issuer = threadIdx.x == 0;
    bool ok = true;
    int g = 0;
    for (int k = 0, item = snake_item(0, b, G, n_items); ok && item >= 0; ++k) {
      int jt, bh;
      decode_item(item, jt, bh);
      const int it0 = CAUSAL ? jt : 0, n_it = item_tiles(jt);
      for (int it = 0; it < n_it; ++it, ++g) {
        const int qt = it0 + it;
        const bool got = mbar_wait_warp(bar(kBarDQFull), g & 1, ctx, 0x540);
        if (!(ok = named_barrier_and(kDrainBarrierId, 128, got))) break;
        tc_fence_after();
        auto stage = [&](int c, const uint32_t (&v)[32]) {
          const uint32_t buf = sbase + Ly::kStage + (c & 1) * 16384;
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
        uint32_t a0[32], a1[32], a2[32];
        tmem_ld32(tDQ, a0);
        tmem_ld32(tDQ + 32, a1);
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
      }
      item = snake_item(k + 1, b, G, n_items);
    }
    if (issuer) bulk_wait_group_all();
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

// The value of one E4M3 byte (finite codes): sign, 4-bit exponent with bias
// 7, 3-bit mantissa; exponent 0 holds the subnormals m 2^-9.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const uint32_t e = (byte >> 3) & 0xFu, m = byte & 7u;
  const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : float(m) * 0.001953125f;
  return __uint_as_float(__float_as_uint(mag) | ((byte & 0x80u) << 24));
}

// D_i = dod <dO8_i, O_i> (O in bf16), L_i log2(e) (+inf on padded rows), the
// dQ accumulator zeroed, and the |dS| maximum word cleared.  Eight threads per
// row, 16 values each.
__global__ void __launch_bounds__(256)
    attn_bwd_fp8_preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                   const uint8_t* __restrict__ dO8, const float* __restrict__ L,
                                   float* __restrict__ L2ws, float* __restrict__ Dws,
                                   float* __restrict__ acc, int BH, int N, int Npad,
                                   size_t acc_vec4, float do_descale,
                                   float* __restrict__ ds_amax) {
  const size_t rows = size_t(BH) * Npad;
  const size_t nthreads = size_t(gridDim.x) * blockDim.x;
  const size_t gt = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  grid_dep_wait();
  grid_dep_launch();
  if (gt == 0 && ds_amax) *ds_amax = 0.f;
  // warp w covers rows 4 w .. 4 w + 3 per pass (8 lanes per row)
  for (size_t base = (gt / 32) * 4; base < rows; base += (nthreads / 32) * 4) {
    const size_t row = base + lane / 8;
    const int part = lane % 8;
    float dot = 0.f;
    const int q = int(row % Npad);
    if (row < rows && q < N) {
      const size_t off = (size_t(row / Npad) * N + q) * HD + part * 16;
      const uint4 o0 = __ldg(reinterpret_cast<const uint4*>(O + off));
      const uint4 o1 = __ldg(reinterpret_cast<const uint4*>(O + off + 8));
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(dO8 + off));
      const uint32_t ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
      const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int w = 0; w < 4; ++w)  // bytes 4w .. 4w+3 against O values 4w .. 4w+3
        dot += e4m3_to_f32(gv[w] & 0xFF) * bf16lo_to_f32(ov[2 * w]) +
               e4m3_to_f32((gv[w] >> 8) & 0xFF) * bf16hi_to_f32(ov[2 * w]) +
               e4m3_to_f32((gv[w] >> 16) & 0xFF) * bf16lo_to_f32(ov[2 * w + 1]) +
               e4m3_to_f32(gv[w] >> 24) * bf16hi_to_f32(ov[2 * w + 1]);
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (row < rows && part == 0) {
      const bool valid = q < N;
      Dws[row] = valid ? dot * do_descale : 0.f;
      L2ws[row] = valid ? __ldg(L + size_t(row / Npad) * N + q) * 1.4426950408889634f : INFINITY;
    }
  }
  float4* a4 = reinterpret_cast<float4*>(acc);
  for (size_t i = gt; i < acc_vec4; i += nthreads) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

static int num_sms_fp8() {
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

static int head_group_fp8(const Shape& s) {
  if (s.causal) return s.BH;
  int l2 = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0)
    l2 = 32 << 20;
  // Q, dO (1 byte each) and the dQ accumulator (4 bytes) per element
  size_t hg = (size_t(l2) / 2) / (size_t(s.Npad) * s.d * 6);
  if (hg < 1) hg = 1;
  if (hg > size_t(s.BH)) hg = size_t(s.BH);
  return int(hg);
}

template <bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO,
                            const CUtensorMap& tmAcc, void* dK, void* dV, const Workspace& ws,
                            const Shape& s, const Fp8BwdScales& sc, float* ds_amax, int* err,
                            cudaStream_t stream) {
  auto kern = attn_bwd_fp8_kernel<CAUSAL>;
  cudaError_t e = set_smem_limit_once<attn_bwd_fp8_kernel<CAUSAL>>(Layout::kBytes);
  if (e != cudaSuccess) return e;
  const long long n_items = (long long)s.n_tiles * s.BH;
  const dim3 grid(unsigned(n_items < num_sms_fp8() ? n_items : num_sms_fp8()));
  return launch_kernel(kern, grid, dim3(kThreads), Layout::kBytes, stream, tmQ, tmK, tmV, tmdO,
                       tmAcc, static_cast<const float*>(ws.L2), static_cast<const float*>(ws.D),
                       reinterpret_cast<__nv_bfloat16*>(dK), reinterpret_cast<__nv_bfloat16*>(dV),
                       s.BH, s.N, head_group_fp8(s), sc.score_log2, sc.dp_mult, sc.ds_scale,
                       sc.dk_mult, sc.dv_mult, ds_amax, err);
}

}  // namespace bwd8

cudaError_t launch_bwd_fp8_preprocess(const void* O, const void* dO8, const float* L,
                                      const Workspace& ws, const Shape& s, float do_descale,
                                      float* ds_amax, cudaStream_t stream) {
  const size_t rows = size_t(s.BH) * s.Npad;
  const size_t acc_vec4 = size_t(s.BH) * s.Npad * s.d / 4;
  size_t blocks = (rows * 8 + 255) / 256;
  const size_t acc_blocks = (acc_vec4 + 255) / 256;
  if (acc_blocks > blocks) blocks = acc_blocks;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) blocks = 1;
  return launch_kernel(bwd8::attn_bwd_fp8_preprocess_kernel, dim3(unsigned(blocks)), dim3(256), 0,
                       stream, reinterpret_cast<const __nv_bfloat16*>(O),
                       static_cast<const uint8_t*>(dO8), L, ws.L2, ws.D, ws.acc, s.BH, s.N,
                       s.Npad, acc_vec4, do_descale, ds_amax);
}

cudaError_t launch_bwd_fp8_main(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                const CUtensorMap& tmAcc, void* dK, void* dV, const Workspace& ws,
                                const Shape& s, const Fp8BwdScales& sc, float* ds_amax, int* err,
                                cudaStream_t stream) {
  if (s.causal)
    return bwd8::launch_t<true>(tmQ, tmK, tmV, tmdO, tmAcc, dK, dV, ws, s, sc, ds_amax, err,
                                stream);
  return bwd8::launch_t<false>(tmQ, tmK, tmV, tmdO, tmAcc, dK, dV, ws, s, sc, ds_amax, err,
                               stream);
}

}  // namespace attn
