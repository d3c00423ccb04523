// attn_noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework whose allocator owns
// all device memory and hands a plug-in only its tensors, or a latency-bound
// loop that cannot afford cudaMalloc's implicit device synchronisation.
// attn_bwd needs a workspace from its caller; this entry point instead uses a
// scratch array that the library itself places in device memory when it is
// loaded, so the caller passes only inputs and outputs.
//
// Set-up: the first call on each device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it.  Make that
// first call before any stream capture on that device.
//
// The scratch is the file-scope array below, of fixed size kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads the library holds it until the process
// exits.  Problems whose workspace (attn_bwd_workspace_size) exceeds it are
// rejected with ATTN_ERR_TOO_LARGE.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the preprocessing step rewrites every part of it that the main
// kernel reads (it zeroes the dQ accumulator), so stale contents never leak
// into a result.  Because it is shared, calls that overlap on the GPU (for
// example on two streams) race with each other and give wrong results: order
// them on one stream or synchronise between them.

#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"

namespace attn {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

// Device scratch of attn_bwd_noalloc.  In host code this name is only a
// host-side stand-in: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// The scratch's device address on the current device, looked up once per
// device (the first attn_bwd_noalloc call on that device does it).
void* noalloc_scratch_ptr() {
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                     int causal, float scale, void* stream) {
  // attn_bwd without a workspace validates every other argument and launches
  // nothing: any answer but "workspace missing" (an argument error, or OK for
  // an empty problem) is this call's answer too.
  const int st = attn_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, causal, scale, nullptr, 0,
                          stream);
  if (st != ATTN_ERR_WORKSPACE) return st;
  if (attn_bwd_workspace_size(B, H, N, d) > attn::kNoAllocScratchBytes) return ATTN_ERR_TOO_LARGE;
  void* scratch = attn::noalloc_scratch_ptr();
  if (!scratch) return ATTN_ERR_CUDA;
  return attn_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, causal, scale, scratch,
                  attn::kNoAllocScratchBytes, stream);
}

}  // extern "C"
