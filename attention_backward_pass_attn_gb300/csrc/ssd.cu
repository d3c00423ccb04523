// ssd.cu -- the Mamba-2 state-space layer (scalar-decay selective scan) and
// its backward pass on sm_103a.
//
// "Training Transformers and Hybrid models on AMD Instinct MI300X
// Accelerators" (section "Mamba-2") trains hybrid models whose second hot
// kernel, beside the attention backward, is the Mamba-2 backward: a prefix
// scan over the sequence, a reverse scan of the state gradient, and block
// reductions of dA and dB/dC finished with atomic adds.  Per batch element b
// and head h (group g of B and C), with state h_t in R^{N x P}:
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
//      contribution R = sum_i e_in[i] C_i dy_i^T, and its decay exp(cs_end).
//   2. ssd_state_scan_kernel, per (b, h, state element): the prefix scan
//      H_in[c] = exp(cs_end[c-1]) H_in[c-1] + S[c-1] and the reverse scan
//      dH_out[c] = exp(cs_end[c+1]) dH_out[c+1] + R[c+1], in place.
//   3. ssd_chunk_bwd_kernel, per (b, h, chunk): with H_in and dH_out known,
//      every gradient of the chunk -- dx, dB, dC, ddt (through the chunk's
//      decays, cs) and the chunk's share of dA and dD -- from the masked,
//      decayed 64 x 64 matrices C B^T and dy x^T.  dB and dC are summed over
//      the heads of a group, and dA, dD over chunks, by atomic adds.
//   (ssd_chunk_fwd_kernel: y from H_in and the chunk, for the forward.)
//
// The arithmetic is fp32 on the CUDA cores (inputs x, B, C, dy in bf16);
// the tiles are small (64 x 64 x 128 contractions), so this first version
// keeps them in shared memory rather than on the tensor core.

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace ssd {

constexpr int Lc = 64;           // chunk length
constexpr int kThreads = 256;
constexpr int kVecs = 10;

// Shared-memory layout of the chunk kernels, in floats; each row padded by
// one float so that column walks across rows hit distinct banks.
template <int N, int P>
struct SLayout {
  static constexpr int XS = P + 1;  // Xs, DYs rows (per time step)
  static constexpr int BS = N + 1;  // Bs, Cs rows (per time step)
  static constexpr int HS = P + 1;  // Hs, dHs rows (per state row n)
  static constexpr int MS = Lc + 1;
  static constexpr int oX = 0;
  static constexpr int oDY = oX + Lc * XS;
  static constexpr int oB = oDY + Lc * XS;
  static constexpr int oC = oB + Lc * BS;
  static constexpr int oH = oC + Lc * BS;
  static constexpr int odH = oH + N * HS;
  static constexpr int oM1 = odH + N * HS;
  static constexpr int oM2 = oM1 + Lc * MS;
  static constexpr int oVec = oM2 + Lc * MS;  // kVecs vectors of Lc
  static constexpr int oColPart = oVec + kVecs * Lc;  // [16][Lc] partial column sums
  static constexpr int oRed = oColPart + 16 * Lc;
  static constexpr int kFloats = oRed + 8;
  static constexpr int kBytes = kFloats * 4;
};
// vectors
constexpr int vDT = 0, vCS = 1, vEIN = 2, vEOUT = 3, vROW = 4, vCOL = 5, vE = 6, vF = 7;

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(uint32_t(v) << 16);
}

struct Dims {
  int Bt, T, H, G, nc;
};

// Loads the chunk's rows of a [Bt][T][X][W] bf16 tensor (index xi along X)
// into shared memory as fp32 rows of stride `ld`; rows past T are zero.
template <int W>
__device__ __forceinline__ void load_rows(float* dst, int ld, const uint16_t* src, const Dims& d,
                                          int X, int b, int t0, int xi) {
  for (int idx = threadIdx.x; idx < Lc * W; idx += kThreads) {
    const int i = idx / W, w = idx - i * W;
    const int t = t0 + i;
    dst[i * ld + w] =
        t < d.T ? bf16_to_f32(src[((size_t(b) * d.T + t) * X + xi) * W + w]) : 0.f;
  }
}

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

// ------------------------------------------------------------------ step 1
// S[n][p] = sum_j e_out[j] dt_j B_j[n] x_j[p] (and, for the backward,
// R[n][p] = sum_i e_in[i] C_i[n] dy_i[p]); dec = exp(cs_end).
template <int N, int P, bool BWD>
__global__ void __launch_bounds__(kThreads)
    ssd_chunk_state_kernel(const uint16_t* __restrict__ x, const float* __restrict__ dt,
                           const float* __restrict__ A, const uint16_t* __restrict__ Bm,
                           const uint16_t* __restrict__ Cm, const uint16_t* __restrict__ dy,
                           float* __restrict__ S, float* __restrict__ R,
                           float* __restrict__ dec, Dims d) {
  using Ly = SLayout<N, P>;
  extern __shared__ float sm[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int t0 = c * Lc;
  float* vec = sm + Ly::oVec;
  grid_dep_wait();
  grid_dep_launch();
  chunk_decays(vec, dt, d, b, h, t0, A[h]);
  load_rows<P>(sm + Ly::oX, Ly::XS, x, d, d.H, b, t0, h);
  load_rows<N>(sm + Ly::oB, Ly::BS, Bm, d, d.G, b, t0, g);
  if (BWD) {
    load_rows<P>(sm + Ly::oDY, Ly::XS, dy, d, d.H, b, t0, h);
    load_rows<N>(sm + Ly::oC, Ly::BS, Cm, d, d.G, b, t0, g);
  }
  __syncthreads();
  const size_t chunk = (size_t(b) * d.H + h) * d.nc + c;
  if (threadIdx.x == 0) dec[chunk] = __expf(vec[vCS * Lc + Lc - 1]);
  // thread tile: NR state rows x 4 channels
  constexpr int NR = N / 16;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int n0 = ty * NR, p0 = tx * 4;
  const float* Xs = sm + Ly::oX;
  const float* Bs = sm + Ly::oB;
  float acc[NR][4] = {};
  for (int j = 0; j < Lc; ++j) {
    const float w = vec[vEOUT * Lc + j] * vec[vDT * Lc + j];
    float xv[4], bv[NR];
#pragma unroll
    for (int q = 0; q < 4; ++q) xv[q] = Xs[j * Ly::XS + p0 + q] * w;
#pragma unroll
    for (int r = 0; r < NR; ++r) bv[r] = Bs[j * Ly::BS + n0 + r];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(bv[r], xv[q], acc[r][q]);
  }
  float* Sc = S + chunk * N * P;
#pragma unroll
  for (int r = 0; r < NR; ++r)
    *reinterpret_cast<float4*>(Sc + (n0 + r) * P + p0) =
        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  if (BWD) {
    const float* DYs = sm + Ly::oDY;
    const float* Cs = sm + Ly::oC;
    float acr[NR][4] = {};
    for (int i = 0; i < Lc; ++i) {
      const float w = vec[vEIN * Lc + i];
      float yv[4], cv[NR];
#pragma unroll
      for (int q = 0; q < 4; ++q) yv[q] = DYs[i * Ly::XS + p0 + q] * w;
#pragma unroll
      for (int r = 0; r < NR; ++r) cv[r] = Cs[i * Ly::BS + n0 + r];
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acr[r][q] = fmaf(cv[r], yv[q], acr[r][q]);
    }
    float* Rc = R + chunk * N * P;
#pragma unroll
    for (int r = 0; r < NR; ++r)
      *reinterpret_cast<float4*>(Rc + (n0 + r) * P + p0) =
          make_float4(acr[r][0], acr[r][1], acr[r][2], acr[r][3]);
  }
}

// ------------------------------------------------------------------ step 2
// One thread per (b, h, state element): the prefix scan of the states over
// chunks (S becomes H_in, the state entering each chunk) and, for the
// backward, the reverse scan of the state gradient (R becomes dH_out, the
// gradient of the state leaving each chunk from the chunks after it).
__global__ void __launch_bounds__(kThreads)
    ssd_state_scan_kernel(float* __restrict__ S, float* __restrict__ R,
                          const float* __restrict__ dec, int NP, Dims d, int bwd) {
  const int e = blockIdx.x * kThreads + threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  grid_dep_wait();
  grid_dep_launch();
  if (e >= NP) return;
  const size_t base = (size_t(b) * d.H + h) * d.nc;
  float carry = 0.f;
  for (int c = 0; c < d.nc; ++c) {
    float* p = S + (base + c) * NP + e;
    const float s = *p;
    *p = carry;
    carry = fmaf(dec[base + c], carry, s);
  }
  if (!bwd) return;
  carry = 0.f;
  for (int c = d.nc - 1; c >= 0; --c) {
    float* p = R + (base + c) * NP + e;
    const float r = *p;
    *p = carry;
    carry = fmaf(dec[base + c], carry, r);
  }
}

// Loads an N x P fp32 state of a chunk into shared memory (row stride HS).
template <int N, int P>
__device__ __forceinline__ void load_state(float* dst, const float* __restrict__ src) {
  for (int idx = threadIdx.x; idx < N * P / 4; idx += kThreads) {
    const int n = (idx * 4) / P, p = (idx * 4) % P;
    const float4 v = *reinterpret_cast<const float4*>(src + n * P + p);
    float* r = dst + n * (P + 1) + p;
    r[0] = v.x;
    r[1] = v.y;
    r[2] = v.z;
    r[3] = v.w;
  }
}

// Sum over the 16 threads of a half-warp that share ty (lanes tx = 0..15).
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ step 3
template <int N, int P>
__global__ void __launch_bounds__(kThreads)
    ssd_chunk_bwd_kernel(const uint16_t* __restrict__ x, const float* __restrict__ dt,
                         const float* __restrict__ A, const uint16_t* __restrict__ Bm,
                         const uint16_t* __restrict__ Cm, const float* __restrict__ D,
                         const uint16_t* __restrict__ dy, const float* __restrict__ Hin,
                         const float* __restrict__ dHout, float* __restrict__ dx,
                         float* __restrict__ ddt, float* __restrict__ dA,
                         float* __restrict__ dB, float* __restrict__ dC,
                         float* __restrict__ dD, Dims d) {
  using Ly = SLayout<N, P>;
  extern __shared__ float sm[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int t0 = c * Lc;
  float* vec = sm + Ly::oVec;
  float* red = sm + Ly::oRed;
  const float Ah = A[h], Dh = D[h];
  const size_t chunk = (size_t(b) * d.H + h) * d.nc + c;
  grid_dep_wait();
  grid_dep_launch();
  for (int i = threadIdx.x; i < 4 * Lc; i += kThreads) vec[vROW * Lc + i] = 0.f;  // ROW..F
  if (threadIdx.x < 8) red[threadIdx.x] = 0.f;
  chunk_decays(vec, dt, d, b, h, t0, Ah);
  load_rows<P>(sm + Ly::oX, Ly::XS, x, d, d.H, b, t0, h);
  load_rows<P>(sm + Ly::oDY, Ly::XS, dy, d, d.H, b, t0, h);
  load_rows<N>(sm + Ly::oB, Ly::BS, Bm, d, d.G, b, t0, g);
  load_rows<N>(sm + Ly::oC, Ly::BS, Cm, d, d.G, b, t0, g);
  load_state<N, P>(sm + Ly::oH, Hin + chunk * N * P);
  load_state<N, P>(sm + Ly::odH, dHout + chunk * N * P);
  __syncthreads();
  const float* Xs = sm + Ly::oX;
  const float* DYs = sm + Ly::oDY;
  const float* Bs = sm + Ly::oB;
  const float* Cs = sm + Ly::oC;
  const float* Hs = sm + Ly::oH;
  const float* dHs = sm + Ly::odH;
  float* M1 = sm + Ly::oM1;  // C B^T o W  (M1[i][j], j <= i)
  float* M2 = sm + Ly::oM2;  // dy x^T o W
  const float* vdt = vec + vDT * Lc;
  const float* vcs = vec + vCS * Lc;
  const float* ein = vec + vEIN * Lc;
  const float* eout = vec + vEOUT * Lc;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;

  // ---- A: C B^T and dy x^T, masked and decayed; the pair sums for ddt
  {
    const int i0 = ty * 4, j0 = tx * 4;
    float cb[4][4] = {}, yx[4][4] = {};
    for (int n = 0; n < N; ++n) {
      float cv[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) cv[a] = Cs[(i0 + a) * Ly::BS + n];
#pragma unroll
      for (int q = 0; q < 4; ++q) bv[q] = Bs[(j0 + q) * Ly::BS + n];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) cb[a][q] = fmaf(cv[a], bv[q], cb[a][q]);
    }
    for (int p = 0; p < P; ++p) {
      float yv[4], xv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) yv[a] = DYs[(i0 + a) * Ly::XS + p];
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = Xs[(j0 + q) * Ly::XS + p];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) yx[a][q] = fmaf(yv[a], xv[q], yx[a][q]);
    }
    float row[4] = {0.f, 0.f, 0.f, 0.f}, col[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + a, j = j0 + q;
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
    for (int q = 0; q < 4; ++q) colpart[ty * Lc + j0 + q] = col[q];
  }
  __syncthreads();
  if (threadIdx.x < Lc) {
    const float* colpart = sm + Ly::oColPart;
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) s += colpart[r * Lc + threadIdx.x];
    vec[vCOL * Lc + threadIdx.x] = s;
  }

  // ---- B: dx_j = dt_j (sum_i M1[i][j] dy_i + e_out[j] dH^T B_j) + D dy_j
  {
    const int j0 = ty * 4, p0 = tx * 4;
    float in[4][4] = {}, out[4][4] = {};
    for (int i = j0; i < Lc; ++i) {  // M1[i][j] = 0 for i < j
      float mv[4], yv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) mv[a] = M1[i * Ly::MS + j0 + a];
#pragma unroll
      for (int q = 0; q < 4; ++q) yv[q] = DYs[i * Ly::XS + p0 + q];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) in[a][q] = fmaf(mv[a], yv[q], in[a][q]);
    }
    for (int n = 0; n < N; ++n) {
      float bv[4], hv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) bv[a] = Bs[(j0 + a) * Ly::BS + n];
#pragma unroll
      for (int q = 0; q < 4; ++q) hv[q] = dHs[n * Ly::HS + p0 + q];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) out[a][q] = fmaf(bv[a], hv[q], out[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = j0 + a, t = t0 + j;
      if (t >= d.T) continue;
      float4 o;
      float* ov = &o.x;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        ov[q] = vdt[j] * (in[a][q] + eout[j] * out[a][q]) + Dh * DYs[j * Ly::XS + p0 + q];
      *reinterpret_cast<float4*>(dx + ((size_t(b) * d.T + t) * d.H + h) * P + p0) = o;
    }
  }

  // ---- C: dB_j = dt_j (sum_i M2[i][j] C_i + e_out[j] dH x_j),
  //         F_j / dt_j = B_j . (e_out[j] dH x_j)
  constexpr int NC = N / 16;  // state columns per thread
  {
    const int j0 = ty * 4, n0 = tx * NC;
    float in[4][NC] = {}, out[4][NC] = {};
    for (int i = j0; i < Lc; ++i) {
      float mv[4], cv[NC];
#pragma unroll
      for (int a = 0; a < 4; ++a) mv[a] = M2[i * Ly::MS + j0 + a];
#pragma unroll
      for (int q = 0; q < NC; ++q) cv[q] = Cs[i * Ly::BS + n0 + q];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NC; ++q) in[a][q] = fmaf(mv[a], cv[q], in[a][q]);
    }
    for (int p = 0; p < P; ++p) {
      float xv[4], hv[NC];
#pragma unroll
      for (int a = 0; a < 4; ++a) xv[a] = Xs[(j0 + a) * Ly::XS + p];
#pragma unroll
      for (int q = 0; q < NC; ++q) hv[q] = dHs[(n0 + q) * Ly::HS + p];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NC; ++q) out[a][q] = fmaf(xv[a], hv[q], out[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = j0 + a, t = t0 + j;
      float f = 0.f;
#pragma unroll
      for (int q = 0; q < NC; ++q) {
        const float inter = eout[j] * out[a][q];
        f = fmaf(Bs[j * Ly::BS + n0 + q], inter, f);
        if (t < d.T)
          atomicAdd(dB + ((size_t(b) * d.T + t) * d.G + g) * N + n0 + q,
                    vdt[j] * (in[a][q] + inter));
      }
      f = sum16(f);
      if (tx == 0) vec[vF * Lc + j] = f;
    }
  }

  // ---- D: dC_i = sum_j M2[i][j] dt_j B_j + e_in[i] H dy_i,
  //         E_i = C_i . (e_in[i] H dy_i)
  {
    const int i0 = ty * 4, n0 = tx * NC;
    float in[4][NC] = {}, out[4][NC] = {};
    for (int j = 0; j <= i0 + 3; ++j) {  // M2[i][j] = 0 for j > i
      float mv[4], bv[NC];
#pragma unroll
      for (int a = 0; a < 4; ++a) mv[a] = M2[(i0 + a) * Ly::MS + j] * vdt[j];
#pragma unroll
      for (int q = 0; q < NC; ++q) bv[q] = Bs[j * Ly::BS + n0 + q];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NC; ++q) in[a][q] = fmaf(mv[a], bv[q], in[a][q]);
    }
    for (int p = 0; p < P; ++p) {
      float yv[4], hv[NC];
#pragma unroll
      for (int a = 0; a < 4; ++a) yv[a] = DYs[(i0 + a) * Ly::XS + p];
#pragma unroll
      for (int q = 0; q < NC; ++q) hv[q] = Hs[(n0 + q) * Ly::HS + p];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NC; ++q) out[a][q] = fmaf(yv[a], hv[q], out[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + a, t = t0 + i;
      float e = 0.f;
#pragma unroll
      for (int q = 0; q < NC; ++q) {
        const float inter = ein[i] * out[a][q];
        e = fmaf(Cs[i * Ly::BS + n0 + q], inter, e);
        if (t < d.T)
          atomicAdd(dC + ((size_t(b) * d.T + t) * d.G + g) * N + n0 + q, in[a][q] + inter);
      }
      e = sum16(e);
      if (tx == 0) vec[vE * Lc + i] = e;
    }
  }

  // ---- E: <dH, H> (the entering state carried through the whole chunk)
  // and this chunk's share of dD = sum dy . x
  {
    float fh = 0.f, dd = 0.f;
    for (int idx = threadIdx.x; idx < N * P; idx += kThreads) {
      const int n = idx / P, p = idx - n * P;
      fh = fmaf(dHs[n * Ly::HS + p], Hs[n * Ly::HS + p], fh);
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
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&red[0], fh);
      atomicAdd(&red[1], dd);
    }
  }
  __syncthreads();

  // ---- F: d(cs_k), its suffix sums d(l_r) = sum_{k >= r} d(cs_k), ddt, dA
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    const float fh = red[0] * __expf(vcs[Lc - 1]);
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
    const float dl1 = s - dcs[0];  // d(l) at k = 2l + 1
    const float dl0 = s;           // d(l) at k = 2l
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
      atomicAdd(dA + h, da);
      atomicAdd(dD + h, red[1]);
    }
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
  extern __shared__ float sm[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int t0 = c * Lc;
  float* vec = sm + Ly::oVec;
  const size_t chunk = (size_t(b) * d.H + h) * d.nc + c;
  grid_dep_wait();
  grid_dep_launch();
  chunk_decays(vec, dt, d, b, h, t0, A[h]);
  load_rows<P>(sm + Ly::oX, Ly::XS, x, d, d.H, b, t0, h);
  load_rows<N>(sm + Ly::oB, Ly::BS, Bm, d, d.G, b, t0, g);
  load_rows<N>(sm + Ly::oC, Ly::BS, Cm, d, d.G, b, t0, g);
  load_state<N, P>(sm + Ly::oH, Hin + chunk * N * P);
  __syncthreads();
  const float* Xs = sm + Ly::oX;
  const float* Bs = sm + Ly::oB;
  const float* Cs = sm + Ly::oC;
  const float* Hs = sm + Ly::oH;
  float* M1 = sm + Ly::oM1;
  const float* vdt = vec + vDT * Lc;
  const float* vcs = vec + vCS * Lc;
  const float* ein = vec + vEIN * Lc;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  {
    const int i0 = ty * 4, j0 = tx * 4;
    float cb[4][4] = {};
    for (int n = 0; n < N; ++n) {
      float cv[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) cv[a] = Cs[(i0 + a) * Ly::BS + n];
#pragma unroll
      for (int q = 0; q < 4; ++q) bv[q] = Bs[(j0 + q) * Ly::BS + n];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) cb[a][q] = fmaf(cv[a], bv[q], cb[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + a, j = j0 + q;
        M1[i * Ly::MS + j] = j <= i ? cb[a][q] * __expf(vcs[i] - vcs[j]) * vdt[j] : 0.f;
      }
  }
  __syncthreads();
  {
    const int i0 = ty * 4, p0 = tx * 4;
    float in[4][4] = {}, out[4][4] = {};
    for (int j = 0; j <= i0 + 3; ++j) {
      float mv[4], xv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) mv[a] = M1[(i0 + a) * Ly::MS + j];
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = Xs[j * Ly::XS + p0 + q];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) in[a][q] = fmaf(mv[a], xv[q], in[a][q]);
    }
    for (int n = 0; n < N; ++n) {
      float cv[4], hv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) cv[a] = Cs[(i0 + a) * Ly::BS + n];
#pragma unroll
      for (int q = 0; q < 4; ++q) hv[q] = Hs[n * Ly::HS + p0 + q];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) out[a][q] = fmaf(cv[a], hv[q], out[a][q]);
    }
    const float Dh = D[h];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + a, t = t0 + i;
      if (t >= d.T) continue;
      float4 o;
      float* ov = &o.x;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        ov[q] = in[a][q] + ein[i] * out[a][q] + Dh * Xs[i * Ly::XS + p0 + q];
      *reinterpret_cast<float4*>(y + ((size_t(b) * d.T + t) * d.H + h) * P + p0) = o;
    }
  }
}

__global__ void __launch_bounds__(kThreads) ssd_zero_kernel(float* a, size_t na, float* b,
                                                            size_t nb, float* c, size_t nc_,
                                                            float* e, size_t ne) {
  grid_dep_wait();
  grid_dep_launch();
  const size_t stride = size_t(gridDim.x) * kThreads;
  for (size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x; i < na + nb + nc_ + ne;
       i += stride) {
    if (i < na) a[i] = 0.f;
    else if (i < na + nb) b[i - na] = 0.f;
    else if (i < na + nb + nc_) c[i - na - nb] = 0.f;
    else e[i - na - nb - nc_] = 0.f;
  }
}

template <int N, int P>
static cudaError_t set_limits() {
  cudaError_t e = set_smem_limit_once<ssd_chunk_state_kernel<N, P, true>>(SLayout<N, P>::kBytes);
  if (e == cudaSuccess)
    e = set_smem_limit_once<ssd_chunk_state_kernel<N, P, false>>(SLayout<N, P>::kBytes);
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
  if (bwd) {
    const size_t nbc = size_t(a.Bt) * a.T * a.G * N;
    e = launch_kernel(ssd_zero_kernel, dim3(152 * 4), dim3(kThreads), 0, st, a.dB, nbc, a.dC,
                      nbc, a.dA, size_t(a.H), a.dD, size_t(a.H));
    if (e != cudaSuccess) return e;
    e = launch_kernel(ssd_chunk_state_kernel<N, P, true>, grid, dim3(kThreads), smem, st, x, a.dt,
                      a.A, Bm, Cm, dy, a.ws_S, a.ws_R, a.ws_dec, d);
  } else {
    e = launch_kernel(ssd_chunk_state_kernel<N, P, false>, grid, dim3(kThreads), smem, st, x,
                      a.dt, a.A, Bm, Cm, dy, a.ws_S, a.ws_R, a.ws_dec, d);
  }
  if (e != cudaSuccess) return e;
  const int NP = N * P;
  e = launch_kernel(ssd_state_scan_kernel, dim3(unsigned(NP / kThreads), a.H, a.Bt),
                    dim3(kThreads), 0, st, a.ws_S, a.ws_R, static_cast<const float*>(a.ws_dec),
                    NP, d, bwd ? 1 : 0);
  if (e != cudaSuccess) return e;
  if (!bwd)
    return launch_kernel(ssd_chunk_fwd_kernel<N, P>, grid, dim3(kThreads), smem, st, x, a.dt,
                         a.A, Bm, Cm, a.D, static_cast<const float*>(a.ws_S), a.y, d);
  return launch_kernel(ssd_chunk_bwd_kernel<N, P>, grid, dim3(kThreads), smem, st, x, a.dt, a.A,
                       Bm, Cm, a.D, dy, static_cast<const float*>(a.ws_S),
                       static_cast<const float*>(a.ws_R), a.dx, a.ddt, a.dA, a.dB, a.dC, a.dD, d);
}

}  // namespace ssd

cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t stream) {
  if (a.P != 64) return cudaErrorInvalidValue;
  if (a.N == 128) return ssd::run<128, 64>(a, stream);
  if (a.N == 64) return ssd::run<64, 64>(a, stream);
  return cudaErrorInvalidValue;
}

size_t ssd_workspace_floats(int Bt, int T, int H, int N, int P) {
  const size_t nc = (size_t(T) + ssd::Lc - 1) / ssd::Lc;
  const size_t chunks = size_t(Bt) * H * nc;
  return 2 * chunks * size_t(N) * P + ((chunks + 63) / 64) * 64;
}

}  // namespace attn
