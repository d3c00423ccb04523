// attn_api.cu -- the library's C ABI (declared in include/attn.h): argument
// validation, TMA tensor-map encoding, workspace carve-up, the per-device
// error word, and the calls into the kernel launchers.

#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

// The device error word the kernels report failures into.  Host code never
// dereferences the symbol: it asks the runtime for its device address.
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;

int* error_word_ptr() {
  static std::mutex mu;
  static int* ptrs[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Validate sizes and flags; fill `s`.  Returns ATTN_OK, or an error, or
// (through *empty) that the problem has no rows.
int make_shape(int B, int H, int N, int d, int causal, Shape* s, bool* empty) {
  if (B < 0 || H < 0 || N < 0 || d < 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  *empty = (B == 0 || H == 0 || N == 0);
  if (*empty) return ATTN_OK;
  const long long BH = (long long)B * H;
  const long long n_tiles = (N + 127LL) / 128;
  // Keep every row index (and the grid size) inside 31 bits.
  if (BH > INT_MAX || BH * n_tiles * 128 > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  s->BH = int(BH);
  s->N = N;
  s->d = d;
  s->causal = causal;
  s->n_tiles = int(n_tiles);
  s->Npad = int(n_tiles * 128);
  s->window = 0;
  s->H = H;
  s->doc = nullptr;
  return ATTN_OK;
}

// The sliding window and the document map: only with the causal mask; a
// window of N or more keys is the causal mask itself.  The map is read by
// the kernels as int32 and must be 4-byte aligned.
int check_mask(int causal, int window, const int* doc) {
  if (window < 0 || (window > 0 && !causal)) return ATTN_ERR_INVALID_ARG;
  if (doc && (!causal || (reinterpret_cast<uintptr_t>(doc) & 3u) != 0))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}
void set_mask(Shape* s, int window, const int* doc) {
  s->window = window >= s->N ? 0 : window;
  s->doc = doc;
}

bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

int check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

int check_workspace(const void* ws, size_t bytes, const Shape& s) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return ATTN_ERR_WORKSPACE;
  if (bytes < workspace_bytes(s)) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

}  // namespace

size_t workspace_bytes(const Shape& s) {
  const size_t vec = round256(sizeof(float) * size_t(s.BH) * s.Npad);
  const size_t acc = round256(sizeof(float) * size_t(s.BH) * s.Npad * s.d);
  const size_t items = round256(sizeof(int2) * size_t(s.BH) * s.n_tiles);
  const size_t order = round256(sizeof(int) * size_t(s.BH) * s.n_tiles);
  return 3 * vec + acc + items + order;  // qend: one int32 per row, the size of a vec section
}

Workspace carve_workspace(void* base, const Shape& s) {
  const size_t vec = round256(sizeof(float) * size_t(s.BH) * s.Npad);
  char* p = static_cast<char*>(base);
  Workspace w;
  w.L2 = reinterpret_cast<float*>(p);
  w.D = reinterpret_cast<float*>(p + vec);
  w.acc = reinterpret_cast<float*>(p + 2 * vec);
  char* q = p + 2 * vec + round256(sizeof(float) * size_t(s.BH) * s.Npad * s.d);
  w.items = reinterpret_cast<int2*>(q);
  w.qend = reinterpret_cast<int*>(q + round256(sizeof(int2) * size_t(s.BH) * s.n_tiles));
  w.order = reinterpret_cast<int*>(reinterpret_cast<char*>(w.qend) +
                                   round256(sizeof(int) * size_t(s.BH) * s.Npad));
  return w;
}

int make_tile_map(CUtensorMap* map, const void* ptr, const Shape& s) {
  auto encode = encode_fn();
  if (!encode) return -1;
  const cuuint64_t dims[3] = {cuuint64_t(s.d), cuuint64_t(s.N), cuuint64_t(s.BH)};
  const cuuint64_t strides[2] = {cuuint64_t(s.d) * 2, cuuint64_t(s.N) * s.d * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_tile_map_u8(CUtensorMap* map, const void* ptr, const Shape& s) {
  auto encode = encode_fn();
  if (!encode) return -1;
  const cuuint64_t dims[3] = {cuuint64_t(s.d), cuuint64_t(s.N), cuuint64_t(s.BH)};
  const cuuint64_t strides[2] = {cuuint64_t(s.d), cuuint64_t(s.N) * s.d};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_acc_map(CUtensorMap* map, const float* acc, const Shape& s) {
  auto encode = encode_fn();
  if (!encode) return -1;
  const cuuint64_t dims[2] = {cuuint64_t(s.d), cuuint64_t(s.BH) * cuuint64_t(s.Npad)};
  const cuuint64_t strides[1] = {cuuint64_t(s.d) * 4};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(acc), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

// The main kernel for a validated, non-empty shape (mask included): with
// `fused_dq` the instantiation that also adds dQ partials into the
// workspace's accumulator, else the one that forms dK and dV only.
int bwd_main_launch(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                    void* dV, const Shape& s, float scale, void* workspace, bool fused_dq,
                    void* stream) {
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  const Workspace ws = carve_workspace(workspace, s);
  CUtensorMap mq, mk, mv, mdo, macc;
  if (make_tile_map(&mq, Q, s) || make_tile_map(&mk, K, s) || make_tile_map(&mv, V, s) ||
      make_tile_map(&mdo, dO, s))
    return ATTN_ERR_CUDA;
  if (!fused_dq)
    return cuda_status(
        launch_bwd_main_dkdv(mq, mk, mv, mdo, dK, dV, ws, s, scale, err, (cudaStream_t)stream));
  if (make_acc_map(&macc, ws.acc, s)) return ATTN_ERR_CUDA;
  return cuda_status(launch_bwd_main(mq, mk, mv, mdo, macc, dK, dV, ws, s, scale, err,
                                     (cudaStream_t)stream));
}

// The separate dQ pass for a validated, non-empty shape (mask included).
int bwd_dq_launch(const void* Q, const void* K, const void* V, const void* dO, void* dQ,
                  const Shape& s, float scale, void* workspace, void* stream) {
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv, mdo;
  if (make_tile_map(&mq, Q, s) || make_tile_map(&mk, K, s) || make_tile_map(&mv, V, s) ||
      make_tile_map(&mdo, dO, s))
    return ATTN_ERR_CUDA;
  return cuda_status(launch_bwd_dq(mq, mk, mv, mdo, dQ, carve_workspace(workspace, s), s, scale,
                                   err, (cudaStream_t)stream));
}

// The dQ method attn_bwd uses when the caller leaves the choice to the
// library.
int auto_dq_method(const Shape& s) {
  (void)s;
  return ATTN_DQ_REDUCE;
}

}  // namespace attn

namespace attn {
namespace {
// Validates the SSD layer's sizes; fills `empty` for a problem with no work.
int ssd_shape(int Bt, int T, int H, int G, int N, int P, bool* empty) {
  if (Bt < 0 || T < 0 || H < 0 || G <= 0 || N < 0 || P < 0) return ATTN_ERR_INVALID_ARG;
  if (H % G != 0) return ATTN_ERR_INVALID_ARG;
  if (P != 64 || (N != 64 && N != 128)) return ATTN_ERR_UNSUPPORTED;
  const long long nc = (T + 63LL) / 64;
  if ((long long)Bt * T * H * P > INT_MAX * 64LL || nc > INT_MAX || H > 65535 || Bt > 65535)
    return ATTN_ERR_UNSUPPORTED;
  *empty = (Bt == 0 || T == 0 || H == 0);
  return ATTN_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int ssd_carve(SsdArgs* a, void* workspace, size_t bytes) {
  const size_t need = ssd_workspace_size(a->Bt, a->T, a->H, a->G, a->N, a->P);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || bytes < need)
    return ATTN_ERR_WORKSPACE;
  auto r64 = [](size_t v) { return (v + 63) / 64 * 64; };
  const size_t nc = (size_t(a->T) + 63) / 64;
  const size_t chunks = size_t(a->Bt) * a->H * nc;
  const size_t states = r64(chunks * a->N * a->P);
  const size_t heads = r64(size_t(a->Bt) * a->T * a->H * a->N);
  float* p = static_cast<float*>(workspace);
  a->ws_S = p;
  a->ws_R = p += states;
  a->ws_dBh = p += states;
  a->ws_dCh = p += heads;
  a->ws_dec = p += heads;
  a->ws_dA = p += r64(chunks);
  a->ws_dD = p += r64(chunks);
  return ATTN_OK;
}
}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int attn_version(void) { return 100; }

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128)";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_ERR_DEVICE: return "device-side check failed";
    case ATTN_ERR_TOO_LARGE: return "problem too large for the built-in 32 MiB scratch";
    default: return "unknown status";
  }
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
  Shape s;
  bool empty = false;
  if (make_shape(B, H, N, d, 0, &s, &empty) != ATTN_OK || empty) return 0;
  return workspace_bytes(s);
}

int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int N,
             int d, int causal, float scale, void* stream) {
  return attn_fwd_ex(Q, K, V, O, L, B, H, N, d, causal, 0, nullptr, scale, stream);
}

int attn_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                int N, int d, int causal, int window, const int* doc_start, float scale,
                void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if ((st = check_mask(causal, window, doc_start)) != ATTN_OK) return st;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  set_mask(&s, window, doc_start);
  if ((st = check_ptrs({Q, K, V, O, L})) != ATTN_OK) return st;
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  if (make_tile_map(&mq, Q, s) || make_tile_map(&mk, K, s) || make_tile_map(&mv, V, s))
    return ATTN_ERR_CUDA;
  return cuda_status(launch_fwd(mq, mk, mv, O, L, s, scale, err, (cudaStream_t)stream));
}

int attn_fwd_fp8(const void* Q8, const void* K8, const void* V8, float q_descale,
                 float k_descale, float v_descale, void* O, float* L, int B, int H, int N, int d,
                 int causal, float scale, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!scale_ok(scale) || !scale_ok(q_descale) || !scale_ok(k_descale) || !scale_ok(v_descale))
    return ATTN_ERR_INVALID_ARG;
  const float score_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
  if (!scale_ok(score_log2)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({Q8, K8, V8, O, L})) != ATTN_OK) return st;
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  if (make_tile_map_u8(&mq, Q8, s) || make_tile_map_u8(&mk, K8, s) ||
      make_tile_map_u8(&mv, V8, s))
    return ATTN_ERR_CUDA;
  return cuda_status(
      launch_fwd_fp8(mq, mk, mv, O, L, s, score_log2, v_descale, err, (cudaStream_t)stream));
}

int attn_bwd_fp8(const void* Q8, const void* K8, const void* V8, const void* O, const void* dO8,
                 const float* L, float q_descale, float k_descale, float v_descale,
                 float do_descale, float ds_scale, void* dQ, void* dK, void* dV, float* ds_amax,
                 int B, int H, int N, int d, int causal, float scale, void* workspace,
                 size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  for (float f : {scale, q_descale, k_descale, v_descale, do_descale, ds_scale})
    if (!scale_ok(f)) return ATTN_ERR_INVALID_ARG;
  Fp8BwdScales sc;
  sc.score_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
  sc.dp_mult = v_descale * do_descale;
  sc.ds_scale = ds_scale;
  sc.dk_mult = scale * q_descale / ds_scale;
  sc.dv_mult = do_descale / 256.f;
  const float dq_mult = scale * k_descale / ds_scale;
  for (float f : {sc.score_log2, sc.dp_mult, sc.dk_mult, sc.dv_mult, dq_mult})
    if (!scale_ok(f)) return ATTN_ERR_INVALID_ARG;
  if (ds_amax && (reinterpret_cast<uintptr_t>(ds_amax) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({Q8, K8, V8, O, dO8, L, dQ, dK, dV})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  const Workspace ws = carve_workspace(workspace, s);
  CUtensorMap mq, mk, mv, mdo, macc;
  if (make_tile_map_u8(&mq, Q8, s) || make_tile_map_u8(&mk, K8, s) ||
      make_tile_map_u8(&mv, V8, s) || make_tile_map_u8(&mdo, dO8, s) ||
      make_acc_map(&macc, ws.acc, s))
    return ATTN_ERR_CUDA;
  cudaStream_t strm = (cudaStream_t)stream;
  if ((st = cuda_status(launch_bwd_fp8_preprocess(O, dO8, L, ws, s, do_descale, ds_amax,
                                                  strm))) != ATTN_OK)
    return st;
  if ((st = cuda_status(launch_bwd_fp8_main(mq, mk, mv, mdo, macc, dK, dV, ws, s, sc, ds_amax,
                                            err, strm))) != ATTN_OK)
    return st;
  return cuda_status(launch_bwd_dq_convert(dQ, ws, s, dq_mult, strm));
}

int attn_bwd_preprocess(const void* O, const void* dO, const float* L, int B, int H, int N, int d,
                        void* workspace, size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, 0, &s, &empty);
  if (st != ATTN_OK) return st;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({O, dO, L})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  return cuda_status(launch_bwd_preprocess(O, dO, L, carve_workspace(workspace, s), s, true,
                                           (cudaStream_t)stream));
}

int attn_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dK, void* dV,
                  int B, int H, int N, int d, int causal, float scale, void* workspace,
                  size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({Q, K, V, dO, dK, dV})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  return bwd_main_launch(Q, K, V, dO, dK, dV, s, scale, workspace, true, stream);
}

int attn_bwd_main_dkdv(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                       void* dV, int B, int H, int N, int d, int causal, float scale,
                       void* workspace, size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({Q, K, V, dO, dK, dV})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  return bwd_main_launch(Q, K, V, dO, dK, dV, s, scale, workspace, false, stream);
}

int attn_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, void* dQ, int B,
                int H, int N, int d, int causal, float scale, const void* workspace,
                size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({Q, K, V, dO, dQ})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  return bwd_dq_launch(Q, K, V, dO, dQ, s, scale, const_cast<void*>(workspace), stream);
}

int attn_bwd_dq_convert(void* dQ, int B, int H, int N, int d, float scale, const void* workspace,
                        size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, 0, &s, &empty);
  if (st != ATTN_OK) return st;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({dQ})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  return cuda_status(launch_bwd_dq_convert(dQ, carve_workspace(const_cast<void*>(workspace), s),
                                           s, scale, (cudaStream_t)stream));
}

int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
             const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d, int causal,
             float scale, void* workspace, size_t workspace_bytes_, void* stream) {
  return attn_bwd_ex(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, causal, 0, nullptr, scale,
                     workspace, workspace_bytes_, stream);
}

int attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                int causal, int window, const int* doc_start, float scale, void* workspace,
                size_t workspace_bytes_, void* stream) {
  return attn_bwd_opts(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, causal, window, doc_start,
                       scale, ATTN_DQ_AUTO, workspace, workspace_bytes_, stream);
}

int attn_bwd_opts(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                  int causal, int window, const int* doc_start, float scale, int dq_method,
                  void* workspace, size_t workspace_bytes_, void* stream) {
  Shape s;
  bool empty = false;
  int st = make_shape(B, H, N, d, causal, &s, &empty);
  if (st != ATTN_OK) return st;
  if ((st = check_mask(causal, window, doc_start)) != ATTN_OK) return st;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (dq_method != ATTN_DQ_AUTO && dq_method != ATTN_DQ_REDUCE && dq_method != ATTN_DQ_SEPARATE)
    return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  set_mask(&s, window, doc_start);
  if ((st = check_ptrs({Q, K, V, O, dO, L, dQ, dK, dV})) != ATTN_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes_, s)) != ATTN_OK) return st;
  const bool fused = (dq_method == ATTN_DQ_AUTO ? auto_dq_method(s) : dq_method) == ATTN_DQ_REDUCE;
  const Workspace ws = carve_workspace(workspace, s);
  if ((st = cuda_status(launch_bwd_preprocess(O, dO, L, ws, s, fused, (cudaStream_t)stream))) !=
      ATTN_OK)
    return st;
  if (s.doc && (st = cuda_status(launch_bwd_order(ws, s, (cudaStream_t)stream))) != ATTN_OK)
    return st;
  if ((st = bwd_main_launch(Q, K, V, dO, dK, dV, s, scale, workspace, fused, stream)) != ATTN_OK)
    return st;
  if (!fused) return bwd_dq_launch(Q, K, V, dO, dQ, s, scale, workspace, stream);
  return cuda_status(launch_bwd_dq_convert(dQ, ws, s, scale, (cudaStream_t)stream));
}


size_t ssd_workspace_size(int Bt, int T, int H, int G, int N, int P) {
  bool empty = false;
  if (ssd_shape(Bt, T, H, G, N, P, &empty) != ATTN_OK || empty) return 0;
  return sizeof(float) * ssd_workspace_floats(Bt, T, H, N, P);
}

int ssd_fwd(const void* x, const float* dt, const float* A, const void* B, const void* C,
            const float* D, float* y, int Bt, int T, int H, int G, int N, int P,
            void* workspace, size_t workspace_bytes_, void* stream) {
  bool empty = false;
  int st = ssd_shape(Bt, T, H, G, N, P, &empty);
  if (st != ATTN_OK || empty) return st;
  if ((st = check_ptrs({x, B, C, y})) != ATTN_OK) return st;
  if (!dt || !A || !D || !aligned4(dt) || !aligned4(A) || !aligned4(D))
    return ATTN_ERR_INVALID_ARG;
  SsdArgs a = {};
  a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.y = y;
  a.Bt = Bt; a.T = T; a.H = H; a.G = G; a.N = N; a.P = P;
  if ((st = ssd_carve(&a, workspace, workspace_bytes_)) != ATTN_OK) return st;
  return cuda_status(launch_ssd(a, (cudaStream_t)stream));
}

int ssd_bwd(const void* x, const float* dt, const float* A, const void* B, const void* C,
            const float* D, const void* dy, float* dx, float* ddt, float* dA, float* dB,
            float* dC, float* dD, int Bt, int T, int H, int G, int N, int P, void* workspace,
            size_t workspace_bytes_, void* stream) {
  bool empty = false;
  int st = ssd_shape(Bt, T, H, G, N, P, &empty);
  if (st != ATTN_OK) return st;
  if (empty) return ATTN_OK;
  if ((st = check_ptrs({x, B, C, dy, dx, dB, dC})) != ATTN_OK) return st;
  for (const void* p : {static_cast<const void*>(dt), static_cast<const void*>(A),
                        static_cast<const void*>(D), static_cast<const void*>(ddt),
                        static_cast<const void*>(dA), static_cast<const void*>(dD)})
    if (!p || !aligned4(p)) return ATTN_ERR_INVALID_ARG;
  SsdArgs a = {};
  a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.dy = dy;
  a.dx = dx; a.ddt = ddt; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD;
  a.Bt = Bt; a.T = T; a.H = H; a.G = G; a.N = N; a.P = P;
  if ((st = ssd_carve(&a, workspace, workspace_bytes_)) != ATTN_OK) return st;
  return cuda_status(launch_ssd(a, (cudaStream_t)stream));
}

int attn_device_error_word(void* stream, int* word) {
  if (word) *word = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  int host = 0;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (host != 0 && cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (word) *word = host;
  if (host == 0) return ATTN_OK;
  return (host >> 24) == kDevTimeout ? ATTN_ERR_TIMEOUT : ATTN_ERR_DEVICE;
}

int attn_last_device_error(void* stream) { return attn_device_error_word(stream, nullptr); }

int attn_watchdog_selftest(uint64_t limit_ns, void* stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
  int* err = error_word_ptr();
  if (!err) return ATTN_ERR_CUDA;
  return cuda_status(launch_watchdog_selftest(err, limit_ns, (cudaStream_t)stream));
}

}  // extern "C"
