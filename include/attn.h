/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * What it computes.  Exact softmax attention and its fused backward pass, the
 * "Flash Attention v2" forward and backward kernels named by "Training
 * Transformers and Hybrid models on AMD Instinct MI300X Accelerators"
 * (section "Flash Attention"; section "Harnessing the MI300 Hardware Specs"
 * adds that the backward recomputes the forward's activations).  Per head,
 * with s = scale and the causal mask keeping key j <= query i:
 *
 *   S = s Q K^T (+ mask),  L_i = logsumexp_j S_ij,  P = exp(S - L),  O = P V
 *   D_i = <dO_i, O_i>,  dP = dO V^T,  dS = P o (dP - D)
 *   dQ = s dS K,  dK = s dS^T Q,  dV = P^T dO
 *
 * The N x N matrices S, P, dP, dS are never stored: each kernel recomputes
 * them tile by tile on the tensor cores.
 *
 * Layout and types (every entry point).
 *   Q, K, V, O, dO, dQ, dK, dV : bf16 (raw uint16 bits), contiguous
 *                                [B][H][N][d], 16-byte aligned.
 *   L                          : fp32 [B][H][N], natural-log log-sum-exp.
 *   d                          : 64 or 128.   N: any value >= 0.
 *   causal                     : 0 or 1 (square, top-left aligned mask).
 *   scale                      : finite and > 0 (usually 1/sqrt(d)).
 *   stream                     : a cudaStream_t (NULL = legacy default).
 * All pointers are DEVICE pointers on the current CUDA device.  The caller
 * allocates and owns every buffer, the backward's workspace included; the
 * library allocates no device memory.
 *
 * Behaviour.  Arguments are validated on the host before anything is
 * launched; a bad argument returns an error status and launches nothing.  A
 * zero B, H or N is a valid empty problem: the call returns ATTN_OK and
 * launches nothing (pointers may then be NULL).  Otherwise the work is
 * enqueued on `stream` and the call returns without waiting: inputs must stay
 * alive and unmodified, and outputs untouched, until the stream reaches the
 * call.  Kernels never trap: a device-side failure (a bounded wait that ran
 * out) is recorded in a per-device error word that attn_last_device_error()
 * reads.  Every kernel is launched with programmatic dependent launch
 * allowed: it may start its set-up while the previous kernel in the stream
 * is finishing, and waits for that kernel to complete (griddepcontrol.wait)
 * before it reads global memory, so stream order is kept for all data.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale, misaligned pointer */
  ATTN_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, or a size beyond the 32-bit index range */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_TIMEOUT = 4,     /* a kernel's bounded wait ran out (reported by attn_last_device_error) */
  ATTN_ERR_WORKSPACE = 5,   /* workspace NULL, misaligned or smaller than attn_bwd_workspace_size */
  ATTN_ERR_DEVICE = 6,      /* another device-side check failed (see attn_device_error_word) */
  ATTN_ERR_TOO_LARGE = 7    /* attn_bwd_noalloc: workspace need exceeds its built-in scratch */
} attn_status_t;

/*
 * Forward.  O = softmax(scale Q K^T + mask) V and L = row log-sum-exp of the
 * scaled, masked scores (natural log), as in the forward of the page section
 * "Flash Attention" (FlashAttention-2).  Writes O [B][H][N][d] bf16 and L
 * [B][H][N] fp32.  Q, K, V must not alias O.
 */
int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
             int N, int d, int causal, float scale, void* stream);

/*
 * Forward with the mask variants of "Training - CUDA Moat Still Alive",
 * section on attention variants, on top of the causal mask; otherwise as
 * attn_fwd.
 *
 *   window     sliding window (Mistral 7B): key j is visible to query i
 *              when i - window < j <= i.  0 = none; window >= N is the
 *              causal mask.
 *   doc_start  document mask for packed sequences (FlexAttention's document
 *              mask): DEVICE int32 [B][N], doc_start[b*N + i] = the first
 *              position of the document holding position i, so query i sees
 *              keys doc_start[i] <= j <= i.  NULL = one document.  Entries
 *              must be i (a document starts) or doc_start[i - 1]; other
 *              values give unspecified results (no fault).  4-byte aligned.
 *
 * Both need causal = 1 (else ATTN_ERR_INVALID_ARG, as for a negative window)
 * and combine: j >= max(doc_start[i], i - window + 1).  Key/value tiles that
 * no query of a tile can see are skipped, so the cost follows the visible
 * area (N * window, or the sum of squared document lengths), not N^2.
 */
int attn_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                int N, int d, int causal, int window, const int* doc_start, float scale,
                void* stream);

/*
 * Forward with 8-bit floating-point inputs, the extension to fp8 precision
 * that "Training Transformers and Hybrid models on AMD Instinct MI300X
 * Accelerators" (section "Summary") names as its attention kernel's next
 * step.  Q8, K8, V8 are OCP FP8 E4M3 bytes (torch.float8_e4m3fn), contiguous
 * [B][H][N][d], 16-byte aligned; the values they stand for are byte value x
 * q_descale (k_descale, v_descale), each finite and > 0.  Computes, with both
 * contractions on the tensor core in fp8 and fp32 accumulation,
 *
 *   S = scale q_descale k_descale Q8 K8^T (+ mask),  L = logsumexp(S),
 *   O = softmax(S) (v_descale V8)
 *
 * and writes O (bf16) and L (fp32) as attn_fwd does.  The probabilities are
 * rounded to e4m3 (relative error up to 2^-4) for P V; the row sums and L use
 * the unrounded fp32 values.  d must be 128 (ATTN_ERR_UNSUPPORTED otherwise);
 * the causal mask is supported, the window and document masks are not.
 */
int attn_fwd_fp8(const void* Q8, const void* K8, const void* V8, float q_descale,
                 float k_descale, float v_descale, void* O, float* L, int B, int H, int N, int d,
                 int causal, float scale, void* stream);

/*
 * Backward with 8-bit floating-point operands, the fp8 extension of the same
 * page section "Summary" applied to the backward: all five contractions per
 * tile pair (S^T, dP^T, dV, dK, dQ) run on e4m3 operands on the tensor core
 * with fp32 accumulation.  Q8, K8, V8, dO8: E4M3 bytes [B][H][N][d] standing
 * for byte x q_descale (k_descale, v_descale, do_descale); O: the forward's
 * output, bf16; L: its log-sum-exp.  Writes dQ, dK, dV (bf16) as attn_bwd
 * does, with the same workspace (attn_bwd_workspace_size).
 *
 * The probabilities are rounded to e4m3 as 256 P (P <= 1); dS = P o (dP - D)
 * is rounded as ds_scale x dS, where ds_scale is the caller's: the largest
 * |dS| the call met is stored in *ds_amax (a device float; NULL = not
 * reported), so the caller can pick the next call's scale with
 * ds_scale x amax <= 448 (delayed scaling).  Values of ds_scale x dS beyond
 * 448 saturate.  d must be 128 (ATTN_ERR_UNSUPPORTED otherwise); the causal
 * mask or none; every factor finite and > 0.
 */
int attn_bwd_fp8(const void* Q8, const void* K8, const void* V8, const void* O, const void* dO8,
                 const float* L, float q_descale, float k_descale, float v_descale,
                 float do_descale, float ds_scale, void* dQ, void* dK, void* dV, float* ds_amax,
                 int B, int H, int N, int d, int causal, float scale, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * Interface utility of this library's boundary; the paper has no counterpart.
 * Bytes of device workspace attn_bwd needs for this shape (0 for an empty
 * problem).  Holds, per head, D = rowsum(dO o O) and L scaled to base 2, each
 * [roundup(N,128)] fp32, an fp32 dQ accumulator of roundup(N,128) x d,
 * three int32 per 128-row tile and one per row (query ranges and the order
 * of work under a document mask); each section starts on a 256-byte
 * boundary.
 * The workspace must be 256-byte aligned; its contents on entry do not matter.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward.  Given the forward's inputs, its outputs O and L, and the
 * upstream gradient dO, writes dQ, dK, dV (bf16, [B][H][N][d]) -- the
 * FlashAttention-2 backward of the page section "Flash Attention", with the
 * probabilities P recomputed from Q, K and L ("activation recomputation",
 * section "Harnessing the MI300 Hardware Specs").  Runs three kernels on
 * `stream`: attn_bwd_preprocess, attn_bwd_main and attn_bwd_dq_convert
 * (below), in that order.  Outputs must not alias inputs or the workspace.
 */
int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
             const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
             int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward with the mask variants of attn_fwd_ex (window, doc_start; L must
 * come from attn_fwd_ex with the same mask).  Same workspace and steps as
 * attn_bwd; window = 0 and doc_start = NULL is attn_bwd.
 */
int attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                int causal, int window, const int* doc_start, float scale, void* workspace,
                size_t workspace_bytes, void* stream);

/*
 * How the backward forms dQ_i = s sum_j dS_ij k_j, a sum over key tiles while
 * the main kernel walks key tiles (the backward of the page section "Flash
 * Attention"):
 *
 *   ATTN_DQ_REDUCE    the main kernel also forms each key tile's partial
 *                     dS K and adds it into an fp32 accumulator in the
 *                     workspace (TMA reduce-add); a last kernel converts it
 *                     to bf16.  Five contractions per tile pair.  The fp32
 *                     summation order varies between runs (dQ repeats to
 *                     about 1e-3 relative; dK, dV bitwise).
 *   ATTN_DQ_SEPARATE  the main kernel forms dK and dV only; a separate
 *                     query-stationary pass recomputes S and dP per key tile
 *                     (the activation recomputation of section "Harnessing
 *                     the MI300 Hardware Specs") and keeps dQ in tensor
 *                     memory.  Seven contractions per tile pair, no
 *                     accumulator traffic, every output bitwise repeatable.
 *   ATTN_DQ_AUTO      the library's choice for the shape (measured on GB300).
 */
typedef enum { ATTN_DQ_AUTO = 0, ATTN_DQ_REDUCE = 1, ATTN_DQ_SEPARATE = 2 } attn_dq_method_t;

/*
 * attn_bwd_ex with the dQ method chosen by the caller (attn_dq_method_t;
 * another value is ATTN_ERR_INVALID_ARG).  Same workspace, results (within
 * rounding) and errors as attn_bwd_ex, which is this call with ATTN_DQ_AUTO.
 */
int attn_bwd_opts(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                  int causal, int window, const int* doc_start, float scale, int dq_method,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Step 1 of attn_bwd: D_i = <dO_i, O_i> in fp32 and L_i * log2(e) into the
 * workspace, and zero the workspace's dQ accumulator.  Bound by HBM
 * bandwidth.
 */
int attn_bwd_preprocess(const void* O, const void* dO, const float* L, int B, int H, int N, int d,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Step 2 of attn_bwd: the fused main kernel.  For each 128-row key/value
 * tile it recomputes S^T = K Q^T and P^T tile by tile, accumulates
 * dV += P^T dO and dK += dS^T Q in tensor memory, and adds each dQ tile
 * partial dS K into the workspace's fp32 accumulator.  Writes dK and dV.
 * Requires attn_bwd_preprocess to have run on the same workspace.
 */
int attn_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                  void* dV, int B, int H, int N, int d, int causal, float scale, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * Step 3 of attn_bwd: dQ = bf16(scale * accumulator).  Bound by HBM
 * bandwidth.  Requires attn_bwd_main to have run on the same workspace.
 */
int attn_bwd_dq_convert(void* dQ, int B, int H, int N, int d, float scale, const void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Step 2 of the ATTN_DQ_SEPARATE backward: the main kernel without the dQ
 * contraction -- dV += P^T dO and dK += dS^T Q per key/value tile, written
 * as bf16 dK, dV.  Requires attn_bwd_preprocess on the same workspace (whose
 * dQ accumulator it does not use).
 */
int attn_bwd_main_dkdv(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                       void* dV, int B, int H, int N, int d, int causal, float scale,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Step 3 of the ATTN_DQ_SEPARATE backward: the query-stationary dQ pass.  Per
 * pair of 128-row query tiles it recomputes S = s Q K^T, P = exp(S - L),
 * dP = dO V^T and dS = P o (dP - D) for every key/value tile the mask lets it
 * see, accumulates dQ += dS K in tensor memory, and writes dQ (bf16).
 * Requires attn_bwd_preprocess (L and D) on the same workspace; it does not
 * depend on step 2, and writes nothing step 2 reads.
 */
int attn_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, void* dQ, int B,
                int H, int N, int d, int causal, float scale, const void* workspace,
                size_t workspace_bytes, void* stream);

/*
 * Backward without any device allocation, for callers that cannot call
 * cudaMalloc (a host framework whose allocator owns all device memory and
 * hands a plug-in only its tensors, or a latency-bound loop that cannot
 * afford cudaMalloc's implicit synchronisation).  The paper has no
 * counterpart: this is an interface variant of attn_bwd, not part of the
 * method.  Same arguments, results and errors as attn_bwd, without the
 * workspace: the library uses a 32 MiB scratch array of its own in device
 * memory, held by every GPU that loads the library until the process exits.
 * Problems whose attn_bwd_workspace_size exceeds 32 MiB return
 * ATTN_ERR_TOO_LARGE and launch nothing.  The first call on each device looks
 * up the scratch's device address; make it before any stream capture on that
 * device.  All calls share the scratch (it keeps the last call's contents,
 * and every call rewrites what it reads), so calls that overlap on the GPU,
 * e.g. on two streams, race: order them on one stream.  The address is
 * looked up once per device and kept for the life of the process, so a
 * cudaDeviceReset after the first call on a device is not supported (the
 * same holds for the error word every entry point reports into).
 */
int attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                     int causal, float scale, void* stream);

/*
 * The Mamba-2 state-space layer, the hybrid model's second hot kernel beside
 * attention ("Training Transformers and Hybrid models on AMD Instinct MI300X
 * Accelerators", section "Mamba-2": its backward by a prefix scan, a reverse
 * scan, and block reductions finished with atomic adds).  Per batch element b
 * and head h, with B and C from group g = h / (H / G) and a state h_t of
 * N x P values:
 *
 *   h_t = exp(dt_t A_h) h_{t-1} + dt_t B_t x_t^T,  h_{-1} = 0
 *   y_t = h_t^T C_t + D_h x_t
 *
 * Layouts (contiguous): x, dy [Bt][T][H][P] bf16; dt [Bt][T][H] fp32 (the
 * step sizes, already positive); A, D [H] fp32; B, C [Bt][T][G][N] bf16.
 * Outputs fp32: y, dx [Bt][T][H][P]; ddt [Bt][T][H]; dA, dD [H];
 * dB, dC [Bt][T][G][N].  P must be 64 and N 64 or 128 (else
 * ATTN_ERR_UNSUPPORTED); H a multiple of G; bf16 and fp32 arrays 16- and
 * 4-byte aligned.  All pointers are device pointers; the workspace
 * (ssd_workspace_size bytes, 256-byte aligned) is the caller's.  Sums over
 * heads (dB, dC of a group) and over time (dA, dD) run in a fixed order, so
 * every output is bitwise repeatable.
 */
size_t ssd_workspace_size(int Bt, int T, int H, int G, int N, int P);

/* Forward: y of the layer above. */
int ssd_fwd(const void* x, const float* dt, const float* A, const void* B, const void* C,
            const float* D, float* y, int Bt, int T, int H, int G, int N, int P,
            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward for the loss <dy, y>: dx, ddt, dA, dB, dC, dD (overwritten, not
 * accumulated into).  Recomputes the states from the inputs; y is not needed.
 */
int ssd_bwd(const void* x, const float* dt, const float* A, const void* B, const void* C,
            const float* D, const void* dy, float* dx, float* ddt, float* dA, float* dB,
            float* dC, float* dD, int Bt, int T, int H, int G, int N, int P, void* workspace,
            size_t workspace_bytes, void* stream);

/*
 * Interface utility of this library's boundary (failure detection); the paper
 * has no counterpart.
 * Synchronise `stream`, then read and clear the current device's error word.
 * Returns ATTN_OK if no kernel reported a failure since the last call,
 * ATTN_ERR_TIMEOUT if a bounded wait ran out, ATTN_ERR_DEVICE for another
 * device-side check, ATTN_ERR_CUDA if the synchronisation itself failed.
 */
int attn_last_device_error(void* stream);

/*
 * Interface utility; the paper has no counterpart.
 * Like attn_last_device_error, but also stores the raw error word
 * ((code << 24) | site, 0 if none) in *word before clearing it.
 */
int attn_device_error_word(void* stream, int* word);

/*
 * Interface utility; the paper has no counterpart.
 * Failure-detection self-test: launches one tiny kernel whose bounded
 * mbarrier wait can never be satisfied (nothing arrives), with a limit of
 * `limit_ns` nanoseconds (1e3 .. 1e10).  The kernel gives up, records
 * ATTN_ERR_TIMEOUT in the error word and exits normally; it never traps or
 * hangs.  Returns the launch status.
 */
int attn_watchdog_selftest(uint64_t limit_ns, void* stream);

/* Interface utility; the paper has no counterpart.  Static text for a status
 * code. */
const char* attn_status_string(int status);

/* Interface utility; the paper has no counterpart.  Library version,
 * major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
