// mask.cuh -- the key range a query row may attend to under the causal mask,
// a sliding window and documents (packed sequences).
#pragma once

#include <cuda_runtime.h>

namespace attn {

// Masks beyond the plain (causal or full) one; a template argument of the
// kernels, so the plain kernels carry none of this code.
constexpr int kMaskPlain = 0;
constexpr int kMaskWindow = 1;    // causal sliding window
constexpr int kMaskDocument = 2;  // causal documents, optionally with a window

// First key row that query row q may see: q - window + 1 under a window, and
// no earlier than the start of q's document, docb[q] (the document map of q's
// batch element, or null).  A map entry outside [0, q] is clamped into it, so
// a malformed map gives wrong values but never an out-of-range tile.
__device__ __forceinline__ int first_visible_key(int q, const int* docb, int window, int N) {
  int lo = window > 0 && q - window + 1 > 0 ? q - window + 1 : 0;
  if (docb && q < N) {
    int ds = __ldg(docb + q);
    ds = ds < 0 ? 0 : (ds > q ? q : ds);
    lo = ds > lo ? ds : lo;
  }
  return lo;
}

}  // namespace attn
