// kernels.h -- host-side launchers shared between the kernel translation units
// and the C ABI in attn_api.cu.  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace attn {

// One attention problem: BH = B*H independent heads of N rows, head dim d.
struct Shape {
  int BH;
  int N;
  int d;
  int causal;
  int n_tiles;  // ceil(N / 128): 128-row tiles per head
  int Npad;     // n_tiles * 128
  int window;   // causal sliding window: key j visible to query i iff i - window < j <= i;
                // 0 = no window (also used for window >= N)
  int H;        // heads per batch element (BH = B * H)
  const int* doc;  // causal documents: doc[b * N + i] = first position of i's document,
                   // device memory; null = none
};

// Workspace carve-up (256-byte aligned sections):
//   L2    [BH][Npad]     fp32  L * log2(e); +inf on padded rows
//   D     [BH][Npad]     fp32  rowsum(dO o O); 0 on padded rows
//   acc   [BH][Npad][d]  fp32  dQ accumulator (unscaled), row-major
//   items [BH][n_tiles]  int2  with documents: per key/value tile, the last
//                              query tile that sees it and the first query
//                              tile that needs element-wise masking
//   qend  [BH][Npad]     int32 with documents: per key, one past the last
//                              query of its document
//   order [BH*n_tiles]   int32 with documents: work items (bh * n_tiles + jt)
//                              sorted by query-tile count, most first
struct Workspace {
  float* L2;
  float* D;
  float* acc;
  int2* items;
  int* qend;
  int* order;
};

// Streaming multiprocessors of the current device (cached per device).
inline int device_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Grid of the forward kernels over n_tasks tasks (query-tile pairs of one
// head).  Without the causal mask every task costs the same: a persistent
// grid, one CTA per SM taking its share of the tasks in turn, overlaps each
// task's loads and first contraction with the previous one's tail.  Under
// the mask tasks differ up to N/256-fold; with more than four per SM, one CTA
// per task lets the hardware hand the next task to whichever SM frees first,
// which balances the unequal tasks better than a fixed split (measured).
inline long long fwd_grid(long long n_tasks, bool causal) {
  const int sms = device_sm_count();
  if (causal && n_tasks > 4LL * sms) return n_tasks;
  return n_tasks < sms ? n_tasks : sms;
}

// Launches a kernel of this library with programmatic dependent launch
// allowed: the kernel may start while the previous kernel in the stream is
// finishing.  Every kernel of the library executes griddepcontrol.wait before
// it reads global memory that earlier work wrote, so results are the same as
// with plain stream order; what overlaps is the launch latency and the
// prologue (barrier set-up, tensor-memory allocation).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises kernel Kern's dynamic shared-memory limit to `bytes`, once per device:
// later launches make no CUDA call for it, which keeps them legal inside a
// CUDA graph capture.
template <auto Kern>
cudaError_t set_smem_limit_once(int bytes) {
  static std::atomic<unsigned long long> done{0};  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

size_t workspace_bytes(const Shape& s);
Workspace carve_workspace(void* base, const Shape& s);

// Encodes a 3-D bf16 tensor map over a contiguous [BH][N][d] tensor with a
// 64 x 128 x 1 box and 128-byte swizzle.  Returns 0 on success.
int make_tile_map(CUtensorMap* map, const void* ptr, const Shape& s);

// Encodes a 3-D 8-bit tensor map over a contiguous [BH][N][d] e4m3 tensor
// (d = 128: one 128-byte row per position) with a 128 x 128 x 1 box and
// 128-byte swizzle.  Returns 0 on success.
int make_tile_map_u8(CUtensorMap* map, const void* ptr, const Shape& s);

// Encodes a 2-D fp32 tensor map over the dQ accumulator [BH*Npad][d] with a
// 32 x 128 box (128-byte rows) and 128-byte swizzle, for TMA reduce-add.
int make_acc_map(CUtensorMap* map, const float* acc, const Shape& s);

cudaError_t launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       void* O, float* L, const Shape& s, float scale, int* err,
                       cudaStream_t stream);

// D, L log2(e) (and the document tables); zeroes the dQ accumulator only if
// zero_acc (the fused main kernel reduces into it; the separate dQ pass does
// not use it).
// The e4m3 forward (head dim 128): score_log2 = scale * q_descale *
// k_descale * log2(e); O is scaled by v_descale.
cudaError_t launch_fwd_fp8(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, void* O, float* L, const Shape& s,
                           float score_log2, float v_descale, int* err, cudaStream_t stream);

// Factors of the e4m3 backward (attn_bwd_fp8.cu): the score scale
// s qd kd log2(e), dP's scale vd dod, the caller's dS quantisation scale,
// and the output factors of dK (s qd / ds_scale) and dV (dod / 256).
struct Fp8BwdScales {
  float score_log2, dp_mult, ds_scale, dk_mult, dv_mult;
};
cudaError_t launch_bwd_fp8_preprocess(const void* O, const void* dO8, const float* L,
                                      const Workspace& ws, const Shape& s, float do_descale,
                                      float* ds_amax, cudaStream_t stream);
cudaError_t launch_bwd_fp8_main(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                const CUtensorMap& tmAcc, void* dK, void* dV, const Workspace& ws,
                                const Shape& s, const Fp8BwdScales& sc, float* ds_amax, int* err,
                                cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const void* O, const void* dO, const float* L,
                                  const Workspace& ws, const Shape& s, bool zero_acc,
                                  cudaStream_t stream);

cudaError_t launch_bwd_main(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO,
                            const CUtensorMap& tmAcc, void* dK, void* dV, const Workspace& ws,
                            const Shape& s, float scale, int* err, cudaStream_t stream);

// The main kernel without the dQ contraction (dK and dV only), for use with
// the separate dQ pass below.
cudaError_t launch_bwd_main_dkdv(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO, void* dK,
                                 void* dV, const Workspace& ws, const Shape& s, float scale,
                                 int* err, cudaStream_t stream);

// The separate query-stationary dQ pass: recomputes S and dP per key/value
// tile, keeps dQ in tensor memory and writes bf16(scale * dQ).  Needs the
// preprocessing step's L log2(e) and D (and, with documents, nothing more).
cudaError_t launch_bwd_dq(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, void* dQ, const Workspace& ws, const Shape& s,
                          float scale, int* err, cudaStream_t stream);

// With documents: sorts the work items by their query-tile count (from the
// preprocessing step's table) so that the main kernel deals them out heaviest
// first.
cudaError_t launch_bwd_order(const Workspace& ws, const Shape& s, cudaStream_t stream);

cudaError_t launch_bwd_dq_convert(void* dQ, const Workspace& ws, const Shape& s, float scale,
                                  cudaStream_t stream);

cudaError_t launch_watchdog_selftest(int* err, uint64_t limit_ns, cudaStream_t stream);

// The Mamba-2 state-space layer (ssd.cu).  Layouts: x, dy [Bt][T][H][P] bf16;
// dt [Bt][T][H], A, D [H] fp32; B, C [Bt][T][G][N] bf16; outputs fp32 with
// the same layouts (dA, dD [H]).  dy == null selects the forward (y).
struct SsdArgs {
  const void* x;
  const float* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* dy;
  float* y;
  float* dx;
  float* ddt;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  int Bt, T, H, G, N, P;
  float* ws_S;    // [Bt][H][chunks][P][N]: chunk states, then the entering states
  float* ws_R;    // [Bt][H][chunks][P][N]: chunk state gradients, then the leaving ones
  float* ws_dBh;  // [Bt][T][H][N]: each head's dB, summed over a group's heads after
  float* ws_dCh;  // [Bt][T][H][N]: each head's dC
  float* ws_dec;  // [Bt][H][chunks]: each chunk's total decay
  float* ws_dA;   // [Bt][H][chunks]: each chunk's share of dA
  float* ws_dD;   // [Bt][H][chunks]: each chunk's share of dD
};
cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t stream);
// Floats of workspace the layer needs (both scans' states plus the decays).
size_t ssd_workspace_floats(int Bt, int T, int H, int N, int P);

}  // namespace attn
