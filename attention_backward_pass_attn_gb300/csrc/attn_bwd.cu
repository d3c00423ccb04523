// attn_bwd.cu -- exact-attention backward on sm_103a.
//
// The FlashAttention-2 backward of "Training Transformers and Hybrid models
// on AMD Instinct MI300X Accelerators" (section "Flash Attention"), with the
// forward's probabilities recomputed instead of stored (section "Harnessing
// the MI300 Hardware Specs": the backward is harder partly because of this
// activation recomputation).  Kernels, in stream order:
//
//  1. attn_bwd_preprocess_kernel: D_i = <dO_i, O_i>, L_i log2(e), and (when
//     the main kernel reduces dQ) a zeroed fp32 dQ accumulator (HBM-bound).
//  2. attn_bwd_main_kernel (attn_bwd_main.cuh): per (head, 128-row key/value
//     tile), dK and dV, and -- in the instantiations launched from this file
//     -- each dQ tile's partial dS K, added into the fp32 accumulator by TMA
//     reduce-add.
//  3. attn_bwd_dq_convert_kernel: dQ = bf16(s * accumulator) (HBM-bound).
//
// The other way to form dQ -- a separate query-stationary pass that
// recomputes S and dP per key/value tile and keeps dQ in tensor memory, with
// no accumulator and no reductions -- is in attn_bwd_dq.cu, with its main
// kernel instantiations in attn_bwd_split.cu.
//
// The dQ reduction is the costly exchange of the fused design: every
// key/value tile adds a 128 x d fp32 partial into each query tile's
// accumulator.  Done as one red.global per thread and 16 bytes it saturated
// the load/store path that the softmax warps also use; as TMA tensor
// reduce-adds of 16 KB boxes it is a handful of instructions per tile and
// runs on the copy engine.  Every kernel is launched with programmatic
// dependent launch: its set-up overlaps the previous kernel, and it waits
// (griddepcontrol.wait) before reading.

#include "attn_bwd_main.cuh"

namespace attn {
namespace bwd {

// ------------------------------------------------------------------ step 1
// One row per HD/8 threads (16 bytes each); rows beyond N get D = 0 and
// L2 = +inf so that their recomputed probabilities are exactly 0.  Each
// thread issues the loads of kUnroll rows before using any of them (memory
// parallelism), then the accumulator is zeroed with 16-byte stores.
constexpr int kUnroll = 4;

template <int HD>
__global__ void __launch_bounds__(256)
    attn_bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                               const __nv_bfloat16* __restrict__ dO, const float* __restrict__ L,
                               float* __restrict__ L2ws, float* __restrict__ Dws,
                               float* __restrict__ acc, int BH, int N, int Npad,
                               size_t acc_vec4, const int* __restrict__ doc, int H, int window,
                               int2* __restrict__ items, int* __restrict__ qend) {
  constexpr int TPR = HD / 8;  // threads per row
  const size_t rows = size_t(BH) * Npad;
  const size_t units = rows * TPR;
  const size_t nthreads = size_t(gridDim.x) * blockDim.x;
  const size_t gt = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  grid_dep_wait();  // O and L come from the forward
  grid_dep_launch();
  // Warp w covers units [w*32*kUnroll, (w+1)*32*kUnroll) per pass, so the
  // shuffle groups of TPR lanes stay inside one row.
  for (size_t base = (gt / 32) * 32 * kUnroll; base < units; base += nthreads * kUnroll) {
    uint4 a[kUnroll], c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t id = base + size_t(u) * 32 + lane;
      const size_t row = id / TPR;
      const int q = int(row % Npad);
      a[u] = c[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows && q < N) {
        const size_t off = (size_t(row / Npad) * N + q) * HD + int(id % TPR) * 8;
        a[u] = __ldg(reinterpret_cast<const uint4*>(O + off));
        c[u] = __ldg(reinterpret_cast<const uint4*>(dO + off));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t id = base + size_t(u) * 32 + lane;
      const size_t row = id / TPR;
      const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
      const uint32_t cv[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dot += bf16lo_to_f32(av[e]) * bf16lo_to_f32(cv[e]) +
               bf16hi_to_f32(av[e]) * bf16hi_to_f32(cv[e]);
#pragma unroll
      for (int o = TPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (row < rows && id % TPR == 0) {
        const int bh = int(row / Npad), q = int(row % Npad);
        const bool valid = q < N;
        Dws[row] = valid ? dot : 0.f;
        L2ws[row] = valid ? __ldg(L + size_t(bh) * N + q) * 1.4426950408889634f : INFINITY;
      }
    }
  }
  float4* a4 = reinterpret_cast<float4*>(acc);
  for (size_t i = gt; i < acc_vec4; i += nthreads) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // With documents: for key/value tile jt of head bh, the last query tile
  // whose first row still sees a key of the tile, and the first query tile
  // whose last row does not see the tile's first key (from there on the
  // main kernel masks element-wise).  Row lower bounds never decrease, so
  // both are binary searches over query tiles.
  if (doc) {
    const int n_tiles = Npad >> 7;
    for (size_t i = gt; i < size_t(BH) * n_tiles; i += nthreads) {
      const int bh = int(i / n_tiles), jt = int(i % n_tiles);
      const int* docb = doc + size_t(bh / H) * N;
      int a = jt, z = n_tiles - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (first_visible_key(mid * 128, docb, window, N) <= jt * 128 + 127)
          a = mid;
        else
          z = mid - 1;
      }
      const int last = a;
      int e0 = jt, e1 = last + 1;
      while (e0 < e1) {
        const int mid = (e0 + e1) >> 1;
        const int qlast = mid * 128 + 127 < N - 1 ? mid * 128 + 127 : N - 1;
        if (first_visible_key(qlast, docb, window, N) > jt * 128)
          e1 = mid;
        else
          e0 = mid + 1;
      }
      items[i] = make_int2(last, e0);
    }
    // Per key position k: one past the last query of k's document, the first
    // position after k whose document starts after k (binary search; N if
    // k's document runs to the end).  Queries from there on cannot see k.
    for (size_t i = gt; i < size_t(BH) * Npad; i += nthreads) {
      const int bh = int(i / Npad), k = int(i % Npad);
      const int* docb = doc + size_t(bh / H) * N;
      int a = k + 1, z = N;  // answer in [k + 1, N]
      if (k >= N) a = z = N;
      while (a < z) {
        const int mid = (a + z) >> 1;
        if (first_visible_key(mid, docb, 0, N) > k)
          z = mid;
        else
          a = mid + 1;
      }
      qend[i] = a;
    }
  }
}

// ------------------------------------------------------------------ step 3
// The accumulator is [BH][Npad][HD] fp32 (row-major); a unit is 8 consecutive
// values of one row.  Each thread loads kUnroll units before storing any.
template <int HD>
__global__ void __launch_bounds__(256)
    attn_bwd_dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dQ,
                               int BH, int N, int Npad, float scale) {
  const size_t units = size_t(BH) * Npad * (HD / 8);
  const size_t nthreads = size_t(gridDim.x) * blockDim.x;
  grid_dep_wait();  // the accumulator is complete once the main kernel is
  grid_dep_launch();
  for (size_t base = size_t(blockIdx.x) * blockDim.x + threadIdx.x; base < units;
       base += nthreads * kUnroll) {
    float4 a[kUnroll], c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t id = base + size_t(u) * nthreads;
      if (id < units) {
        a[u] = __ldcs(reinterpret_cast<const float4*>(acc + id * 8));
        c[u] = __ldcs(reinterpret_cast<const float4*>(acc + id * 8 + 4));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t id = base + size_t(u) * nthreads;
      if (id >= units) continue;
      const size_t row = id / (HD / 8);
      const int q = int(row % Npad), bh = int(row / Npad);
      if (q >= N) continue;
      st_global_v4(dQ + (size_t(bh) * N + q) * HD + int(id % (HD / 8)) * 8,
                   pack_bf16x2(a[u].x * scale, a[u].y * scale),
                   pack_bf16x2(a[u].z * scale, a[u].w * scale),
                   pack_bf16x2(c[u].x * scale, c[u].y * scale),
                   pack_bf16x2(c[u].z * scale, c[u].w * scale));
    }
  }
}

// ------------------------------------------------------------------ self-test
// A wait that nothing can satisfy: the bounded wait must give up, record a
// timeout and let the kernel exit normally.
__global__ void attn_watchdog_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t barrier;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&barrier), 1);
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtx ctx{&abort_flag, err, limit_ns};
  mbar_wait(smem_u32(&barrier), 0, ctx, 0xD06);
}

static unsigned grid_for(size_t work_items, int per_block) {
  size_t blocks = (work_items + per_block - 1) / per_block;
  const size_t cap = 152 * 16;  // a few full waves of 256-thread blocks
  if (blocks > cap) blocks = cap;
  return unsigned(blocks > 0 ? blocks : 1);
}

}  // namespace bwd

cudaError_t launch_bwd_preprocess(const void* O, const void* dO, const float* L,
                                  const Workspace& ws, const Shape& s, bool zero_acc,
                                  cudaStream_t stream) {
  const size_t rows = size_t(s.BH) * s.Npad;
  const size_t acc_vec4 = zero_acc ? size_t(s.BH) * s.Npad * s.d / 4 : 0;
  const size_t work = rows * (s.d / 8) > acc_vec4 ? rows * (s.d / 8) : acc_vec4;
  const unsigned grid = bwd::grid_for(work, 256);
  auto o = reinterpret_cast<const __nv_bfloat16*>(O);
  auto g = reinterpret_cast<const __nv_bfloat16*>(dO);
  auto kern = s.d == 64 ? bwd::attn_bwd_preprocess_kernel<64> : bwd::attn_bwd_preprocess_kernel<128>;
  return launch_kernel(kern, dim3(grid), dim3(256), 0, stream, o, g, L, ws.L2, ws.D, ws.acc, s.BH,
                       s.N, s.Npad, acc_vec4, s.doc, s.H, s.window, ws.items, ws.qend);
}

cudaError_t launch_bwd_main(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO,
                            const CUtensorMap& tmAcc, void* dK, void* dV, const Workspace& ws,
                            const Shape& s, float scale, int* err, cudaStream_t stream) {
  return bwd::launch_main_any<true>(tmQ, tmK, tmV, tmdO, tmAcc, dK, dV, ws, s, scale, err,
                                    stream);
}

namespace bwd {

// Counting sort of the work items by query-tile count, most first, in one CTA
// (bucket counts in shared memory; counts at or above kOrderBins share the
// last bucket, which only coarsens the order).
constexpr int kOrderBins = 8192;

__global__ void __launch_bounds__(1024)
    attn_bwd_order_kernel(const int2* __restrict__ items, int n_tiles, int n_items,
                          int* __restrict__ order) {
  __shared__ int bins[kOrderBins];
  __shared__ int partial[1024];
  grid_dep_wait();  // the item table comes from the preprocessing step
  grid_dep_launch();
  auto weight = [&](int id) {
    const int jt = id % n_tiles;
    int w = items[id].x - jt + 1;
    w = w < 1 ? 1 : (w >= kOrderBins ? kOrderBins - 1 : w);
    return kOrderBins - 1 - w;  // heaviest in bucket 0
  };
  for (int i = threadIdx.x; i < kOrderBins; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  for (int id = threadIdx.x; id < n_items; id += blockDim.x) atomicAdd(&bins[weight(id)], 1);
  __syncthreads();
  // exclusive prefix sum over the buckets: each thread sums a run of 8
  constexpr int kRun = kOrderBins / 1024;
  int run = 0;
  for (int j = 0; j < kRun; ++j) run += bins[threadIdx.x * kRun + j];
  partial[threadIdx.x] = run;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan of the run sums
    const int v = threadIdx.x >= off ? partial[threadIdx.x - off] : 0;
    __syncthreads();
    partial[threadIdx.x] += v;
    __syncthreads();
  }
  int base = partial[threadIdx.x] - run;
  for (int j = 0; j < kRun; ++j) {
    const int c = bins[threadIdx.x * kRun + j];
    bins[threadIdx.x * kRun + j] = base;
    base += c;
  }
  __syncthreads();
  for (int id = threadIdx.x; id < n_items; id += blockDim.x)
    order[atomicAdd(&bins[weight(id)], 1)] = id;
}

}  // namespace bwd

cudaError_t launch_bwd_order(const Workspace& ws, const Shape& s, cudaStream_t stream) {
  return launch_kernel(bwd::attn_bwd_order_kernel, dim3(1), dim3(1024), 0, stream,
                       static_cast<const int2*>(ws.items), s.n_tiles, s.BH * s.n_tiles, ws.order);
}

cudaError_t launch_bwd_dq_convert(void* dQ, const Workspace& ws, const Shape& s, float scale,
                                  cudaStream_t stream) {
  const size_t units = size_t(s.BH) * s.Npad * (s.d / 8);
  const unsigned grid = bwd::grid_for(units, 256);
  auto q = reinterpret_cast<__nv_bfloat16*>(dQ);
  auto kern = s.d == 64 ? bwd::attn_bwd_dq_convert_kernel<64> : bwd::attn_bwd_dq_convert_kernel<128>;
  return launch_kernel(kern, dim3(grid), dim3(256), 0, stream, static_cast<const float*>(ws.acc), q,
                       s.BH, s.N, s.Npad, scale);
}

cudaError_t launch_watchdog_selftest(int* err, uint64_t limit_ns, cudaStream_t stream) {
  bwd::attn_watchdog_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn

