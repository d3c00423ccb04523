// attn_bwd_split.cu -- the backward main kernel's instantiations that leave
// dQ to the separate query-stationary pass (attn_bwd_dq.cu): per key/value
// tile they form dK and dV only, so four contractions per tile pair instead
// of five, no dQ drain, no fp32 accumulator and no TMA reduce-adds.  The
// kernel template is in attn_bwd_main.cuh; this file exists so the two
// instantiation families compile in parallel.

#include "attn_bwd_main.cuh"

namespace attn {

cudaError_t launch_bwd_main_dkdv(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO, void* dK,
                                 void* dV, const Workspace& ws, const Shape& s, float scale,
                                 int* err, cudaStream_t stream) {
  // The dQ accumulator map is never used by these instantiations; the
  // kernel's signature takes one, so the Q map stands in for it.
  return bwd::launch_main_any<false>(tmQ, tmK, tmV, tmdO, tmQ, dK, dV, ws, s, scale, err, stream);
}

}  // namespace attn
