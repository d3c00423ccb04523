// ssd.cu -- the Mamba-2 state-space layer (scalar-decay selective scan) and
// its backward pass on sm_103a.
//
// "Training Transformers and Hybrid models on AMD Instinct MI300X
// Accelerators" (section "Mamba-2") trains hybrid models whose second hot
// kernel, beside the attention backward, is the Mamba-2 backward: a prefix
// scan over the sequence, a reverse scan of the state gradient, and block
// reductions of dA and dB/dC.  Per batch element b and head h (group g of B
// and C), with state h_t in R^{N x P}:
//
//   h_t = exp(dt_t A) h_{t-1} + dt_t B_t x_t^T,   y_t = h_t^T C_t + D x_t
//
// The GB300 design splits the sequence into chunks of Lc = 64 steps, so the
// sequential scan runs over chunks only (T / 64 steps of an N x P state, one
// thread per state element) and everything inside a chunk is dense algebra
// over 64 x 64, 64 x N and N x P tiles held in shared memory.  With cs the
// chunk-local inclusive cumulative sum of dt A, e_in[i] = exp(cs_i) and
// e_out[j] = exp(cs_end - cs_j):
//
//   1. ssd_chunk_state_kernel, per (b, h, chunk): the chunk's own state
//      contribution S = sum_j e_out[j] dt_j B_j x_j^T, its state-gradient
//      contribution R = sum_i e_in[i] C_i dy_i^T (both stored transposed,
//      [P][N]), and its decay exp(cs_end).
//   2. ssd_state_scan_kernel, per (b, h, state element): the prefix scan
//      H_in[c] = exp(cs_end[c-1]) H_in[c-1] + S[c-1] and the reverse scan
//      dH_out[c] = exp(cs_end[c+1]) dH_out[c+1] + R[c+1], in place.
//   3. ssd_chunk_bwd_kernel, per (b, h, chunk): with H_in and dH_out known,
//      every gradient of the chunk -- dx, ddt (through the chunk's decays,
//      cs), and the head's own dB, dC and share of dA, dD -- from the masked,
//      decayed 64 x 64 matrices C B^T and dy x^T.
//   4. ssd_reduce_kernel: dB, dC summed over the heads of each group and dA,
//      dD over batches and chunks, each in a fixed order -- the pages' block
//      exchange, done without atomics so every output is bitwise repeatable.
//   (ssd_chunk_fwd_kernel: y from H_in and the chunk, for the forward.)
//
// The arithmetic is fp32 on the CUDA cores (inputs x, B, C, dy in bf16).  The
// tile products are register-blocked outer products over shared memory read
// with 16-byte loads; rows are padded by four floats so that eight
// consecutive rows fall in distinct 16-byte bank groups.

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace ssd {

constexpr int Lc = 64;  // chunk length
constexpr int kThreads = 256;
constexpr int kVecs = 10;

// Shared-memory layout of the chunk kernels, in floats.  Row-major tiles:
// X, DY [Lc][P]; B, C [Lc][N]; the states H, dH transposed [P][N]; M1, M2
// [Lc][Lc].  Every row stride is the width plus 4.
template <int N, int P>
struct SLayout {
  static constexpr int XS = P + 4;
  static constexpr int BS = N + 4;
  static constexpr int HS = N + 4;  // H^T, dH^T rows (one per channel p)
  static constexpr int MS = Lc + 4;
  static constexpr int oX = 0;
  static constexpr int oDY = oX + Lc * XS;
  static constexpr int oB = oDY + Lc * XS;
  static constexpr int oC = oB + Lc * BS;
  static constexpr int oH = oC + Lc * BS;
  static constexpr int odH = oH + P * HS;
  static constexpr int oM1 = odH + P * HS;
  static constexpr int oM2 = oM1 + Lc * MS;
  static constexpr int oVec = oM2 + Lc * MS;  // kVecs vectors of Lc
  static constexpr int oColPart = oVec + kVecs * Lc;  // [16][Lc] partial column sums
  static constexpr int oRed = oColPart + 16 * Lc;
  static constexpr int kFloats = oRed + 16;  // red: per-warp sums of <dH, H> and dy . x
  static constexpr int kBytes = kFloats * 4;
};
// The chunk-state kernel's smaller layout (X, DY, B, C and the vectors
// only), so that two of its CTAs fit on an SM.
template <int N, int P>
struct SLayoutState {
  static constexpr int XS = P + 4;
  static constexpr int BS = N + 4;
  static constexpr int oX = 0;
  static constexpr int oDY = oX + Lc * XS;
  static constexpr int oB = oDY + Lc * XS;
  static constexpr int oC = oB + Lc * BS;
  static constexpr int oVec = oC + Lc * BS;
  static constexpr int kFloats = oVec + kVecs * Lc;
  static constexpr int kBytes = kFloats * 4;
};
// vectors
constexpr int vDT = 0, vCS = 1, vEIN = 2, vEOUT = 3, vROW = 4, vCOL = 5, vE = 6, vF = 7;

struct Dims {
  int Bt, T, H, G, nc;
};

__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float get(const float4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// A chunk's rows of a [Bt][T][X][W] bf16 tensor (index xi along X), held in
// registers between load() and store(), so that a kernel issues the loads of
// all its tiles before it waits for any.  store() writes them to shared
// memory as fp32 rows of stride `ld`, four values per thread and step; rows
// past T are zero.
template <int W>
struct RowTile {
  static constexpr int kIter = Lc * W / 4 / kThreads;  // 4-value groups per thread
  static_assert(kIter * kThreads * 4 == Lc * W, "tile not a whole number of passes");
  uint2 r[kIter];
  __device__ __forceinline__ void load(const uint16_t* src, const Dims& d, int X, int b, int t0,
                                       int xi) {
#pragma unroll
    for (int k = 0; k < kIter; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int i = idx / (W / 4), w = (idx - i * (W / 4)) * 4;
      const int t = t0 + i;
      r[k] = t < d.T
                 ? *reinterpret_cast<const uint2*>(src + ((size_t(b) * d.T + t) * X + xi) * W + w)
                 : make_uint2(0u, 0u);
    }
  }
  __device__ __forceinline__ void store(float* dst, int ld) const {
#pragma unroll
    for (int k = 0; k < kIter; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int i = idx / (W / 4), w = (idx - i * (W / 4)) * 4;
      *reinterpret_cast<float4*>(dst + i * ld + w) =
          make_float4(__uint_as_float(r[k].x << 16), __uint_as_float(r[k].x & 0xFFFF0000u),
                      __uint_as_float(r[k].y << 16), __uint_as_float(r[k].y & 0xFFFF0000u));
    }
  }
};

// A transposed state [P][N] fp32 of one chunk, held in registers between
// load() and store() (rows of stride N + 4 in shared memory).
template <int N, int P>
struct StateTile {
  static constexpr int kIter = N * P / 4 / kThreads;
  float4 v[kIter];
  __device__ __forceinline__ void load(const float* __restrict__ src) {
#pragma unroll
    for (int k = 0; k < kIter; ++k) v[k] = ld4(src + (threadIdx.x + k * kThreads) * 4);
  }
  __device__ __forceinline__ void store(float* dst) const {
#pragma unroll
    for (int k = 0; k < kIter; ++k) {
      const int e = (threadIdx.x + k * kThreads) * 4;
      *reinterpret_cast<float4*>(dst + (e / N) * (N + 4) + e % N) = v[k];
    }
  }
};

// dt of the chunk, cs = inclusive cumulative sum of dt A, e_in = exp(cs),
// e_out = exp(cs_end - cs).  Steps past T have dt = 0 (no decay, no input).
__device__ __forceinline__ void chunk_decays(float* vec, const float* __restrict__ dt,
                                             const Dims& d, int b, int h, int t0, float A) {
  float* vdt = vec + vDT * Lc;
  float* vcs = vec + vCS * Lc;
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    const int t_a = t0 + 2 * l, t_b = t0 + 2 * l + 1;
    const float da = t_a < d.T ? dt[(size_t(b) * d.T + t_a) * d.H + h] : 0.f;
    const float db = t_b < d.T ? dt[(size_t(b) * d.T + t_b) * d.H + h] : 0.f;
    vdt[2 * l] = da;
    vdt[2 * l + 1] = db;
    const float la = da * A, lb = db * A;
    float s = la + lb;  // inclusive scan of pair sums over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, s, o);
      if (l >= o) s += u;
    }
    vcs[2 * l + 1] = s;
    vcs[2 * l] = s - lb;
  }
  __syncthreads();
  const float cs_end = vcs[Lc - 1];
  for (int i = threadIdx.x; i < Lc; i += kThreads) {
    vec[vEIN * Lc + i] = __expf(vcs[i]);
    vec[vEOUT * Lc + i] = __expf(cs_end - vcs[i]);
  }
}

// Sum over the 16 threads of a half-warp that share ty (lanes tx = 0..15).
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// C B^T (or dy x^T): acc[a][q] += sum_k Arow(i0 + a)[k] Brow(tx + 16 q)[k]
// over K values, both operands rows of stride `ld` (k contiguous).
template <int K>
__device__ __forceinline__ void rows_dot(float (&acc)[4][4], const float* A, const float* Bm,
                                         int ld, int i0, int tx) {
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 av[4], bv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) av[a] = ld4(A + (i0 + a) * ld + k);
#pragma unroll
    for (int q = 0; q < 4; ++q) bv[q] = ld4(Bm + (tx + 16 * q) * ld + k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(get(av[a], kk), get(bv[q], kk), acc[a][q]);
  }
}

// ------------------------------------------------------------------ step 1
// S^T[p][n] = sum_j e_out[j] dt_j x_j[p] B_j[n] (and, for the backward,
// R^T[p][n] = sum_i e_in[i] dy_i[p] C_i[n]); dec = exp(cs_end).
template <int N, int P, bool BWD>
__global__ void __launch_bounds__(kThreads)
    ssd_chunk_state_kernel(const uint16_t* __restrict__ x, const float* __restrict__ dt,
                           const float* __restrict__ A, const uint16_t* __restrict__ Bm,
                           const uint16_t* __restrict__ Cm, const uint16_t* __restrict__ dy,
                           float* __restrict__ S, float* __restrict__ R,
                           float* __restrict__ dec, Dims d) {
  using Ly = SLayoutState<N, P>;
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int t0 = c * Lc;
  float* vec = sm + Ly::oVec;
  grid_dep_wait();
  grid_dep_launch();
  // every tile's loads go out before the decays are formed and before any
  // tile is stored
  RowTile<P> inX, inDY;
  RowTile<N> inB, inC;
  inX.load(x, d, d.H, b, t0, h);
  inB.load(Bm, d, d.G, b, t0, g);
  if (BWD) {
    inDY.load(dy, d, d.H, b, t0, h);
    inC.load(Cm, d, d.G, b, t0, g);
  }
  chunk_decays(vec, dt, d, b, h, t0, A[h]);
  inX.store(sm + Ly::oX, Ly::XS);
  inB.store(sm + Ly::oB, Ly::BS);
  if (BWD) {
    inDY.store(sm + Ly::oDY, Ly::XS);
    inC.store(sm + Ly::oC, Ly::BS);
  }
  __syncthreads();
  const size_t chunk = (size_t(b) * d.H + h) * d.nc + c;
  if (threadIdx.x == 0) dec[chunk] = __expf(vec[vCS * Lc + Lc - 1]);
  // thread tile: 4 channels p = p0 + a x NU groups of 4 states n = n0 + 64 u
  constexpr int NU = N / 64;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int p0 = ty * 4, n0 = tx * 4;
  auto product = [&](const float* Rows, int rld, const float* Cols, const float* wv,
                     float* out) {
    float acc[4][NU][4] = {};
    for (int j = 0; j < Lc; ++j) {
      const float w = wv[j];
      const float4 xv = ld4(Rows + j * rld + p0);
      float4 bv[NU];
#pragma unroll
      for (int u = 0; u < NU; ++u) bv[u] = ld4(Cols + j * Ly::BS + n0 + 64 * u);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float xa = get(xv, a) * w;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          acc[a][u][0] = fmaf(xa, bv[u].x, acc[a][u][0]);
          acc[a][u][1] = fmaf(xa, bv[u].y, acc[a][u][1]);
          acc[a][u][2] = fmaf(xa, bv[u].z, acc[a][u][2]);
          acc[a][u][3] = fmaf(xa, bv[u].w, acc[a][u][3]);
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < NU; ++u)
        *reinterpret_cast<float4*>(out + (p0 + a) * N + n0 + 64 * u) =
            make_float4(acc[a][u][0], acc[a][u][1], acc[a][u][2], acc[a][u][3]);
  };
  // weights e_out[j] dt_j for S, e_in[i] for R (the vector region past the
  // named vectors is free here)
  float* wS = vec + vROW * Lc;
  for (int j = threadIdx.x; j < Lc; j += kThreads) wS[j] = vec[vEOUT * Lc + j] * vec[vDT * Lc + j];
  __syncthreads();
  product(sm + Ly::oX, Ly::XS, sm + Ly::oB, wS, S + chunk * N * P);
  if (BWD) product(sm + Ly::oDY, Ly::XS, sm + Ly::oC, vec + vEIN * Lc, R + chunk * N * P);
}

// ------------------------------------------------------------------ step 2
// The prefix scan of the states over chunks (S becomes H_in, the state
// entering each chunk) and, for the backward, the reverse scan of the state
// gradient (R becomes dH_out, the gradient of the state leaving each chunk
// from the chunks after it).  Each thread carries four consecutive state
// elements of one (b, h) with 16-byte accesses, so a block reads and writes
// 4 KB runs of each chunk's state; every element's multiply-adds are those of
// a one-element scan, in the same order.
__device__ __forceinline__ float4 scan_step(float a, float4 carry, float4 v) {
  return make_float4(fmaf(a, carry.x, v.x), fmaf(a, carry.y, v.y), fmaf(a, carry.z, v.z),
                     fmaf(a, carry.w, v.w));
}

__global__ void __launch_bounds__(kThreads)
    ssd_state_scan_kernel(float* __restrict__ S, float* __restrict__ R,
                          const float* __restrict__ dec, int NP, Dims d, int bwd) {
  const int e = 4 * (blockIdx.x * kThreads + threadIdx.x);  // NP is a multiple of 4 kThreads
  const int h = blockIdx.y, b = blockIdx.z;
  grid_dep_wait();
  grid_dep_launch();
  if (e >= NP) return;
  const size_t base = (size_t(b) * d.H + h) * d.nc;
  auto at = [&](float* M, int c) { return reinterpret_cast<float4*>(M + (base + c) * NP + e); };
  // Sixteen chunks' values are loaded before any is used: the loads do not
  // depend on the carry, only the multiply-adds do.
  constexpr int U = 16;
  float4 carry = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < d.nc; c0 += U) {
    float4 v[U];
    float a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u;
      v[u] = c < d.nc ? *at(S, c) : make_float4(0.f, 0.f, 0.f, 0.f);
      a[u] = c < d.nc ? dec[base + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u;
      if (c < d.nc) *at(S, c) = carry;
      carry = scan_step(a[u], carry, v[u]);
    }
  }
  if (!bwd) return;
  carry = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = d.nc - 1; c0 >= 0; c0 -= U) {
    float4 v[U];
    float a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 - u;
      v[u] = c >= 0 ? *at(R, c) : make_float4(0.f, 0.f, 0.f, 0.f);
      a[u] = c >= 0 ? dec[base + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 - u;
      if (c >= 0) *at(R, c) = carry;
      carry = scan_step(a[u], carry, v[u]);
    }
  }
}

// ------------------------------------------------------------------ step 3
// Writes dx, ddt of the chunk, and the head's own dB, dC ([Bt][T][H][N]) and
// dA, dD shares ([Bt][H][chunks]) for step 4 to sum.
template <int N, int P>
__global__ void __launch_bounds__(kThreads)
    ssd_chunk_bwd_kernel(const uint16_t* __restrict__ x, const float* __restrict__ dt,
                         const float* __restrict__ A, const uint16_t* __restrict__ Bm,
                         const uint16_t* __restrict__ Cm, const float* __restrict__ D,
                         const uint16_t* __restrict__ dy, const float* __restrict__ Hin,
                         const float* __restrict__ dHout, float* __restrict__ dx,
                         float* __restrict__ ddt, float* __restrict__ dBh,
                         float* __restrict__ dCh, float* __restrict__ dApart,
                         float* __restrict__ dDpart, Dims d) {
  using Ly = SLayout<N, P>;
  constexpr int NU = N / 64;
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int t0 = c * Lc;
  float* vec = sm + Ly::oVec;
  float* red = sm + Ly::oRed;
  const float Ah = A[h], Dh = D[h];
  const size_t chunk = (size_t(b) * d.H + h) * d.nc + c;
  grid_dep_wait();
  grid_dep_launch();
  // every tile's loads go out before the decays are formed and before any
  // tile is stored
  RowTile<P> inX, inDY;
  RowTile<N> inB, inC;
  StateTile<N, P> inH, indH;
  inX.load(x, d, d.H, b, t0, h);
  inDY.load(dy, d, d.H, b, t0, h);
  inB.load(Bm, d, d.G, b, t0, g);
  inC.load(Cm, d, d.G, b, t0, g);
  inH.load(Hin + chunk * N * P);
  indH.load(dHout + chunk * N * P);
  chunk_decays(vec, dt, d, b, h, t0, Ah);
  inX.store(sm + Ly::oX, Ly::XS);
  inDY.store(sm + Ly::oDY, Ly::XS);
  inB.store(sm + Ly::oB, Ly::BS);
  inC.store(sm + Ly::oC, Ly::BS);
  inH.store(sm + Ly::oH);
  indH.store(sm + Ly::odH);
  __syncthreads();
  const float* Xs = sm + Ly::oX;
  const float* DYs = sm + Ly::oDY;
  const float* Bs = sm + Ly::oB;
  const float* Cs = sm + Ly::oC;
  const float* HT = sm + Ly::oH;    // H^T[p][n]
  const float* dHT = sm + Ly::odH;  // dH^T[p][n]
  float* M1 = sm + Ly::oM1;         // C B^T o W  (M1[i][j], j <= i)
  float* M2 = sm + Ly::oM2;         // dy x^T o W
  const float* vdt = vec + vDT * Lc;
  const float* vcs = vec + vCS * Lc;
  const float* ein = vec + vEIN * Lc;
  const float* eout = vec + vEOUT * Lc;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  // Row block (of 4 rows) of this half-warp in the triangular steps B-D.  B
  // and C run over rows i >= j, D over j <= i, so a low block costs more in
  // B and C and less in D.  Warps w and w + 4 share an SM sub-partition:
  // warp w takes blocks 2w, 2w + 1 and warp w + 4 blocks 14 - 2w, 15 - 2w,
  // which gives every sub-partition the same share of the triangles.
  const int warp_id = threadIdx.x >> 5;
  const int rb = 2 * (warp_id < 4 ? warp_id : 11 - warp_id) + (ty & 1);

  // ---- A: C B^T and dy x^T, masked and decayed; the pair sums for ddt.
  // Thread tile: rows i = 4 ty + a, columns j = tx + 16 q.
  {
    const int i0 = ty * 4;
    float cb[4][4] = {}, yx[4][4] = {};
    rows_dot<N>(cb, Cs, Bs, Ly::BS, i0, tx);
    rows_dot<P>(yx, DYs, Xs, Ly::XS, i0, tx);
    float row[4] = {0.f, 0.f, 0.f, 0.f}, col[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + a, j = tx + 16 * q;
        const float w = j <= i ? __expf(vcs[i] - vcs[j]) : 0.f;
        const float m1 = cb[a][q] * w, m2 = yx[a][q] * w;
        M1[i * Ly::MS + j] = m1;
        M2[i * Ly::MS + j] = m2;
        const float gp = m1 * yx[a][q];  // G_ij / dt_j
        row[a] = fmaf(gp, vdt[j], row[a]);
        col[q] += gp;
      }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float s = sum16(row[a]);
      if (tx == 0) vec[vROW * Lc + i0 + a] = s;  // one writer per row
    }
    // column sums over the 16 row blocks, added in a fixed order below so
    // that ddt is bitwise repeatable
    float* colpart = sm + Ly::oColPart;
#pragma unroll
    for (int q = 0; q < 4; ++q) colpart[ty * Lc + tx + 16 * q] = col[q];
  }
  __syncthreads();
  if (threadIdx.x < Lc) {
    const float* colpart = sm + Ly::oColPart;
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) s += colpart[r * Lc + threadIdx.x];
    vec[vCOL * Lc + threadIdx.x] = s;
  }

  // ---- B: dx_j = dt_j (sum_i M1[i][j] dy_i + e_out[j] dH^T B_j) + D dy_j.
  // Thread tile: rows j = 4 rb + a, channels p = tx + 16 e.
  {
    const int j0 = rb * 4;
    float in[4][4] = {}, out[4][4] = {};
    for (int i = j0; i < Lc; ++i) {  // M1[i][j] = 0 for i < j
      const float4 mv = ld4(M1 + i * Ly::MS + j0);
      float yv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) yv[e] = DYs[i * Ly::XS + tx + 16 * e];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) in[a][e] = fmaf(get(mv, a), yv[e], in[a][e]);
    }
    // sum_n B_j[n] dH[n][p]: rows of B and of dH^T, n contiguous
#pragma unroll 2
    for (int n = 0; n < N; n += 4) {
      float4 bv[4], hv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) bv[a] = ld4(Bs + (j0 + a) * Ly::BS + n);
#pragma unroll
      for (int e = 0; e < 4; ++e) hv[e] = ld4(dHT + (tx + 16 * e) * Ly::HS + n);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) out[a][e] = fmaf(get(bv[a], kk), get(hv[e], kk), out[a][e]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = j0 + a, t = t0 + j;
      if (t >= d.T) continue;
      float* row = dx + ((size_t(b) * d.T + t) * d.H + h) * P;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = tx + 16 * e;
        row[p] = vdt[j] * (in[a][e] + eout[j] * out[a][e]) + Dh * DYs[j * Ly::XS + p];
      }
    }
  }

  // ---- C: dB_j = dt_j (sum_i M2[i][j] C_i + e_out[j] dH x_j),
  //         F_j / dt_j = B_j . (e_out[j] dH x_j)
  // Thread tile: rows j = 4 rb + a, states n = 4 tx + 64 u + e.
  {
    const int j0 = rb * 4, n0 = tx * 4;
    float in[4][NU][4] = {}, out[4][NU][4] = {};
    for (int i = j0; i < Lc; ++i) {
      const float4 mv = ld4(M2 + i * Ly::MS + j0);
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const float4 cv = ld4(Cs + i * Ly::BS + n0 + 64 * u);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float m = get(mv, a);
          in[a][u][0] = fmaf(m, cv.x, in[a][u][0]);
          in[a][u][1] = fmaf(m, cv.y, in[a][u][1]);
          in[a][u][2] = fmaf(m, cv.z, in[a][u][2]);
          in[a][u][3] = fmaf(m, cv.w, in[a][u][3]);
        }
      }
    }
    // sum_p x_j[p] dH[n][p]: x rows (p contiguous) against dH^T rows p
    for (int p = 0; p < P; p += 4) {
      float4 xv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) xv[a] = ld4(Xs + (j0 + a) * Ly::XS + p);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const float4 hv = ld4(dHT + (p + kk) * Ly::HS + n0 + 64 * u);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float xa = get(xv[a], kk);
            out[a][u][0] = fmaf(xa, hv.x, out[a][u][0]);
            out[a][u][1] = fmaf(xa, hv.y, out[a][u][1]);
            out[a][u][2] = fmaf(xa, hv.z, out[a][u][2]);
            out[a][u][3] = fmaf(xa, hv.w, out[a][u][3]);
          }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = j0 + a, t = t0 + j;
      float f = 0.f;
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const float4 bv = ld4(Bs + j * Ly::BS + n0 + 64 * u);
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float inter = eout[j] * out[a][u][e];
          f = fmaf(get(bv, e), inter, f);
          o[e] = vdt[j] * (in[a][u][e] + inter);
        }
        if (t < d.T)
          *reinterpret_cast<float4*>(dBh + ((size_t(b) * d.T + t) * d.H + h) * N + n0 +
                                     64 * u) = make_float4(o[0], o[1], o[2], o[3]);
      }
      f = sum16(f);
      if (tx == 0) vec[vF * Lc + j] = f;
    }
  }

  // ---- D: dC_i = sum_j M2[i][j] dt_j B_j + e_in[i] H dy_i,
  //         E_i = C_i . (e_in[i] H dy_i)
  // Thread tile: rows i = 4 rb + a, states n = 4 tx + 64 u + e.
  {
    const int i0 = rb * 4, n0 = tx * 4;
    float in[4][NU][4] = {}, out[4][NU][4] = {};
    for (int j = 0; j <= i0 + 3; j += 4) {  // M2[i][j] = 0 for j > i
      float4 mv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) mv[a] = ld4(M2 + (i0 + a) * Ly::MS + j);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float w = vdt[j + kk];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const float4 bv = ld4(Bs + (j + kk) * Ly::BS + n0 + 64 * u);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float m = get(mv[a], kk) * w;
            in[a][u][0] = fmaf(m, bv.x, in[a][u][0]);
            in[a][u][1] = fmaf(m, bv.y, in[a][u][1]);
            in[a][u][2] = fmaf(m, bv.z, in[a][u][2]);
            in[a][u][3] = fmaf(m, bv.w, in[a][u][3]);
          }
        }
      }
    }
    // sum_p dy_i[p] H[n][p]: dy rows against H^T rows p
    for (int p = 0; p < P; p += 4) {
      float4 yv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) yv[a] = ld4(DYs + (i0 + a) * Ly::XS + p);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const float4 hv = ld4(HT + (p + kk) * Ly::HS + n0 + 64 * u);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float ya = get(yv[a], kk);
            out[a][u][0] = fmaf(ya, hv.x, out[a][u][0]);
            out[a][u][1] = fmaf(ya, hv.y, out[a][u][1]);
            out[a][u][2] = fmaf(ya, hv.z, out[a][u][2]);
            out[a][u][3] = fmaf(ya, hv.w, out[a][u][3]);
          }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + a, t = t0 + i;
      float e_ = 0.f;
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const float4 cv = ld4(Cs + i * Ly::BS + n0 + 64 * u);
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float inter = ein[i] * out[a][u][e];
          e_ = fmaf(get(cv, e), inter, e_);
          o[e] = in[a][u][e] + inter;
        }
        if (t < d.T)
          *reinterpret_cast<float4*>(dCh + ((size_t(b) * d.T + t) * d.H + h) * N + n0 +
                                     64 * u) = make_float4(o[0], o[1], o[2], o[3]);
      }
      e_ = sum16(e_);
      if (tx == 0) vec[vE * Lc + i] = e_;
    }
  }

  // ---- E: <dH, H> (the entering state carried through the whole chunk)
  // and this chunk's share of dD = sum dy . x
  {
    float fh = 0.f, dd = 0.f;
    for (int idx = threadIdx.x; idx < N * P; idx += kThreads) {
      const int p = idx / N, n = idx - p * N;
      fh = fmaf(dHT[p * Ly::HS + n], HT[p * Ly::HS + n], fh);
    }
    for (int idx = threadIdx.x; idx < Lc * P; idx += kThreads) {
      const int i = idx / P, p = idx - i * P;
      dd = fmaf(DYs[i * Ly::XS + p], Xs[i * Ly::XS + p], dd);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      fh += __shfl_xor_sync(0xffffffffu, fh, o);
      dd += __shfl_xor_sync(0xffffffffu, dd, o);
    }
    // warp sums into fixed slots, added in order by warp 0 below
    if ((threadIdx.x & 31) == 0) {
      red[threadIdx.x >> 5] = fh;
      red[8 + (threadIdx.x >> 5)] = dd;
    }
  }
  __syncthreads();

  // ---- F: d(cs_k), its suffix sums d(l_r) = sum_{k >= r} d(cs_k), ddt, and
  // the chunk's dA and dD shares
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    float fhs = 0.f, dds = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      fhs += red[w];
      dds += red[8 + w];
    }
    const float fh = fhs * __expf(vcs[Lc - 1]);
    // sum_j F_j, F_j = dt_j * (F_j / dt_j)
    float fsum = vdt[2 * l] * vec[vF * Lc + 2 * l] + vdt[2 * l + 1] * vec[vF * Lc + 2 * l + 1];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fsum += __shfl_xor_sync(0xffffffffu, fsum, o);
    float dcs[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int k = 2 * l + u;
      dcs[u] = vec[vROW * Lc + k] - vdt[k] * vec[vCOL * Lc + k] + vec[vE * Lc + k] -
               vdt[k] * vec[vF * Lc + k] + (k == Lc - 1 ? fsum + fh : 0.f);
    }
    // suffix sums over k: reverse inclusive scan of the pair sums
    float s = dcs[0] + dcs[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_down_sync(0xffffffffu, s, o);
      if (l + o < 32) s += u;
    }
    const float dl0 = s;           // d(l) at k = 2l
    const float dl1 = s - dcs[0];  // d(l) at k = 2l + 1
    float da = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = 2 * l + u;
      const float dl = u == 0 ? dl0 : dl1;
      const int t = t0 + r;
      const float direct = vec[vCOL * Lc + r] + vec[vF * Lc + r];
      if (t < d.T) ddt[(size_t(b) * d.T + t) * d.H + h] = fmaf(Ah, dl, direct);
      da = fmaf(vdt[r], dl, da);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
    if (l == 0) {
      dApart[chunk] = da;
      dDpart[chunk] = dds;
    }
  }
}

// ------------------------------------------------------------------ step 4
// dB, dC: the sum over the heads of each group (in head order) of the
// per-head values; dA, dD: the sum over batches and chunks (in order) of the
// per-chunk shares.  Blocks past the dB/dC part take one head each.
template <int N>
__global__ void __launch_bounds__(kThreads)
    ssd_reduce_kernel(const float* __restrict__ dBh, const float* __restrict__ dCh,
                      const float* __restrict__ dApart, const float* __restrict__ dDpart,
                      float* __restrict__ dB, float* __restrict__ dC, float* __restrict__ dA,
                      float* __restrict__ dD, Dims d, unsigned bc_blocks) {
  grid_dep_wait();
  grid_dep_launch();
  if (blockIdx.x < bc_blocks) {
    const int hpg = d.H / d.G;
    const size_t n_out = size_t(d.Bt) * d.T * d.G * N / 4;  // float4 units
    for (size_t u = size_t(blockIdx.x) * kThreads + threadIdx.x; u < n_out;
         u += size_t(bc_blocks) * kThreads) {
      const size_t e = u * 4;
      const int n = int(e % N);
      const size_t btg = e / N;  // (b * T + t) * G + g
      const int g = int(btg % d.G);
      const size_t bt = btg / d.G;
      float4 sb = make_float4(0.f, 0.f, 0.f, 0.f), sc = sb;
      for (int k = 0; k < hpg; ++k) {
        const size_t src = (bt * d.H + size_t(g) * hpg + k) * N + n;
        const float4 vb = ld4(dBh + src), vc = ld4(dCh + src);
        sb.x += vb.x; sb.y += vb.y; sb.z += vb.z; sb.w += vb.w;
        sc.x += vc.x; sc.y += vc.y; sc.z += vc.z; sc.w += vc.w;
      }
      *reinterpret_cast<float4*>(dB + e) = sb;
      *reinterpret_cast<float4*>(dC + e) = sc;
    }
    return;
  }
  // one block per head; thread k sums a fixed stride of the (b, chunk)
  // shares, then a fixed tree over the block
  const int h = int(blockIdx.x - bc_blocks);
  __shared__ float sa[kThreads], sd[kThreads];
  float a = 0.f, dd = 0.f;
  const int per_head = d.Bt * d.nc;
  for (int k = threadIdx.x; k < per_head; k += kThreads) {
    const int b = k / d.nc, c = k - b * d.nc;
    const size_t ch = (size_t(b) * d.H + h) * d.nc + c;
    a += dApart[ch];
    dd += dDpart[ch];
  }
  sa[threadIdx.x] = a;
  sd[threadIdx.x] = dd;
  __syncthreads();
  for (int s = kThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      sa[threadIdx.x] += sa[threadIdx.x + s];
      sd[threadIdx.x] += sd[threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    dA[h] = sa[0];
    dD[h] = sd[0];
  }
}

// ------------------------------------------------------------------ forward
// y_i = sum_{j <= i} (C_i . B_j) exp(cs_i - cs_j) dt_j x_j + e_in[i] H^T C_i + D x_i
template <int N, int P>
__global__ void __launch_bounds__(kThreads)
    ssd_chunk_fwd_kernel(const uint16_t* __restrict__ x, const float* __restrict__ dt,
                         const float* __restrict__ A, const uint16_t* __restrict__ Bm,
                         const uint16_t* __restrict__ Cm, const float* __restrict__ D,
                         const float* __restrict__ Hin, float* __restrict__ y, Dims d) {
  using Ly = SLayout<N, P>;
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int t0 = c * Lc;
  float* vec = sm + Ly::oVec;
  const size_t chunk = (size_t(b) * d.H + h) * d.nc + c;
  grid_dep_wait();
  grid_dep_launch();
  // every tile's loads go out before the decays are formed and before any
  // tile is stored
  RowTile<P> inX;
  RowTile<N> inB, inC;
  StateTile<N, P> inH;
  inX.load(x, d, d.H, b, t0, h);
  inB.load(Bm, d, d.G, b, t0, g);
  inC.load(Cm, d, d.G, b, t0, g);
  inH.load(Hin + chunk * N * P);
  chunk_decays(vec, dt, d, b, h, t0, A[h]);
  inX.store(sm + Ly::oX, Ly::XS);
  inB.store(sm + Ly::oB, Ly::BS);
  inC.store(sm + Ly::oC, Ly::BS);
  inH.store(sm + Ly::oH);
  __syncthreads();
  const float* Xs = sm + Ly::oX;
  const float* Bs = sm + Ly::oB;
  const float* Cs = sm + Ly::oC;
  const float* HT = sm + Ly::oH;
  float* M1 = sm + Ly::oM1;
  const float* vdt = vec + vDT * Lc;
  const float* vcs = vec + vCS * Lc;
  const float* ein = vec + vEIN * Lc;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int i0 = ty * 4;
  {
    float cb[4][4] = {};
    rows_dot<N>(cb, Cs, Bs, Ly::BS, i0, tx);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + a, j = tx + 16 * q;
        M1[i * Ly::MS + j] = j <= i ? cb[a][q] * __expf(vcs[i] - vcs[j]) * vdt[j] : 0.f;
      }
  }
  __syncthreads();
  // rows i = 4 rb + a, channels p = tx + 16 e.  The triangle is longest for
  // the last row blocks: warp w takes blocks 2w, 2w + 1 and warp w + 4 (on the
  // same SM sub-partition) blocks 14 - 2w, 15 - 2w, which evens the
  // sub-partitions' shares.
  const int warp_id = threadIdx.x >> 5;
  const int rb = 2 * (warp_id < 4 ? warp_id : 11 - warp_id) + (ty & 1);
  const int i1 = rb * 4;
  float in[4][4] = {}, out[4][4] = {};
  for (int j = 0; j <= i1 + 3; j += 4) {  // M1[i][j] = 0 for j > i
    float4 mv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) mv[a] = ld4(M1 + (i1 + a) * Ly::MS + j);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      float xv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) xv[e] = Xs[(j + kk) * Ly::XS + tx + 16 * e];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) in[a][e] = fmaf(get(mv[a], kk), xv[e], in[a][e]);
    }
  }
  rows_dot<N>(out, Cs, HT, Ly::BS, i1, tx);  // sum_n C_i[n] H^T[p][n], p = tx + 16 e
  const float Dh = D[h];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = i1 + a, t = t0 + i;
    if (t >= d.T) continue;
    float* row = y + ((size_t(b) * d.T + t) * d.H + h) * P;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = tx + 16 * e;
      row[p] = in[a][e] + ein[i] * out[a][e] + Dh * Xs[i * Ly::XS + p];
    }
  }
}

template <int N, int P>
static cudaError_t set_limits() {
  cudaError_t e =
      set_smem_limit_once<ssd_chunk_state_kernel<N, P, true>>(SLayoutState<N, P>::kBytes);
  if (e == cudaSuccess)
    e = set_smem_limit_once<ssd_chunk_state_kernel<N, P, false>>(SLayoutState<N, P>::kBytes);
  if (e == cudaSuccess) e = set_smem_limit_once<ssd_chunk_bwd_kernel<N, P>>(SLayout<N, P>::kBytes);
  if (e == cudaSuccess) e = set_smem_limit_once<ssd_chunk_fwd_kernel<N, P>>(SLayout<N, P>::kBytes);
  return e;
}

template <int N, int P>
static cudaError_t run(const SsdArgs& a, cudaStream_t st) {
  cudaError_t e = set_limits<N, P>();
  if (e != cudaSuccess) return e;
  const Dims d{a.Bt, a.T, a.H, a.G, (a.T + Lc - 1) / Lc};
  const dim3 grid(unsigned(d.nc), unsigned(a.H), unsigned(a.Bt));
  const size_t smem = SLayout<N, P>::kBytes;
  auto x = static_cast<const uint16_t*>(a.x);
  auto Bm = static_cast<const uint16_t*>(a.B);
  auto Cm = static_cast<const uint16_t*>(a.C);
  auto dy = static_cast<const uint16_t*>(a.dy);
  const bool bwd = a.dy != nullptr;
  const size_t smem_state = SLayoutState<N, P>::kBytes;
  if (bwd)
    e = launch_kernel(ssd_chunk_state_kernel<N, P, true>, grid, dim3(kThreads), smem_state, st,
                      x, a.dt, a.A, Bm, Cm, dy, a.ws_S, a.ws_R, a.ws_dec, d);
  else
    e = launch_kernel(ssd_chunk_state_kernel<N, P, false>, grid, dim3(kThreads), smem_state, st,
                      x, a.dt, a.A, Bm, Cm, dy, a.ws_S, a.ws_R, a.ws_dec, d);
  if (e != cudaSuccess) return e;
  const int NP = N * P;
  static_assert(N * P % (4 * kThreads) == 0, "the scan takes four state elements a thread");
  e = launch_kernel(ssd_state_scan_kernel, dim3(unsigned(NP / (4 * kThreads)), a.H, a.Bt),
                    dim3(kThreads), 0, st, a.ws_S, a.ws_R, static_cast<const float*>(a.ws_dec),
                    NP, d, bwd ? 1 : 0);
  if (e != cudaSuccess) return e;
  if (!bwd)
    return launch_kernel(ssd_chunk_fwd_kernel<N, P>, grid, dim3(kThreads), smem, st, x, a.dt,
                         a.A, Bm, Cm, a.D, static_cast<const float*>(a.ws_S), a.y, d);
  e = launch_kernel(ssd_chunk_bwd_kernel<N, P>, grid, dim3(kThreads), smem, st, x, a.dt, a.A,
                    Bm, Cm, a.D, dy, static_cast<const float*>(a.ws_S),
                    static_cast<const float*>(a.ws_R), a.dx, a.ddt, a.ws_dBh, a.ws_dCh,
                    a.ws_dA, a.ws_dD, d);
  if (e != cudaSuccess) return e;
  const size_t n_out = size_t(a.Bt) * a.T * a.G * N / 4;
  size_t bc = (n_out + kThreads - 1) / kThreads;
  if (bc > 152 * 8) bc = 152 * 8;
  if (bc == 0) bc = 1;
  return launch_kernel(ssd_reduce_kernel<N>, dim3(unsigned(bc) + unsigned(a.H)), dim3(kThreads),
                       0, st, static_cast<const float*>(a.ws_dBh),
                       static_cast<const float*>(a.ws_dCh), static_cast<const float*>(a.ws_dA),
                       static_cast<const float*>(a.ws_dD), a.dB, a.dC, a.dA, a.dD, d,
                       unsigned(bc));
}

}  // namespace ssd

cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t stream) {
  if (a.P != 64) return cudaErrorInvalidValue;
  if (a.N == 128) return ssd::run<128, 64>(a, stream);
  if (a.N == 64) return ssd::run<64, 64>(a, stream);
  return cudaErrorInvalidValue;
}

// Workspace, in floats: the states S and R ([Bt][H][chunks][P][N] each), the
// per-head dB and dC ([Bt][T][H][N] each), and the per-chunk decays and dA,
// dD shares ([Bt][H][chunks] each); every section a multiple of 64 floats.
size_t ssd_workspace_floats(int Bt, int T, int H, int N, int P) {
  auto r64 = [](size_t v) { return (v + 63) / 64 * 64; };
  const size_t nc = (size_t(T) + ssd::Lc - 1) / ssd::Lc;
  const size_t chunks = size_t(Bt) * H * nc;
  return 2 * r64(chunks * size_t(N) * P) + 2 * r64(size_t(Bt) * T * H * N) + 3 * r64(chunks);
}

}  // namespace attn
