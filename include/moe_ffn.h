/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) batched routed-MoE FFN library.
 *
 * The layer (one call, moe_ffn_prefill) follows the SharpInference issue pages:
 *   router matvec over all N tokens, softmax + top-k (norm_topk_prob on/off)
 *   and shared-expert gate   -- "Carnice prefill toward llama.cpp 676 t/s"
 *                               (#388), breakdown table "router" row and
 *                               "Remaining levers" item 1;
 *   GPU-side expert bucketing into the expStart/expTokI/expTokK CSR
 *                             -- #388 "Remaining levers" item 1 ("Hard part");
 *   gather tokens per expert -> grouped expert GEMM -> scatter
 *                             -- "batched int8-MMQ trunk prefill gated off for
 *                               MoE" (#406), "The work" item 2; #388 lever 3;
 *   Q8_0 weights x Q8_1 activations (int8 block dot products)
 *                             -- #406 references (Q8_0 MMQ), "full-offload MoE
 *                               decode" (#408) lever 2 (Q8_1 / dp4a);
 *   weighted scatter-reduce in top-k slot order k = 0..na-1, then the shared
 *   expert row             -- issue #129, "Scope".
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers (CUDA global memory of the
 *     current device) unless a comment says otherwise.  Arrays are dense,
 *     row-major, C order.  The caller owns every buffer it passes; the library
 *     owns only what moe_weights_create allocates.
 *   - Calls are asynchronous on `stream`: they enqueue kernels and return.
 *     Only moe_weights_create/destroy and moe_workspace_status synchronise.
 *     No call on the hot path allocates memory or copies to/from the host.
 *   - Return value: MOE_OK (0) or a negative moe_status code for an error the
 *     host can see before launching (bad argument, unsupported shape, small
 *     workspace, launch failure).  Errors found by the kernels (an expert
 *     index out of range, a token that selects an expert twice, a malformed
 *     CSR, a device wait that timed out) are OR-ed into the status word at the
 *     start of the workspace; read them with moe_workspace_status.  A kernel
 *     that finds such an error writes a safe result (empty segments, zero
 *     rows) instead of reading out of bounds.
 *   - Shapes: D (hidden), F (routed expert intermediate) and Fs (shared
 *     expert intermediate) are multiples of 32 (the Q8 block).  The tensor-
 *     core path also needs D % 128 == 0, F % 64 == 0 and Fs % 64 == 0; other
 *     shapes run on the matvec path.  1 <= top_k <= min(E, 32), E <= 1024, N >= 1.
 *
 * Block formats
 *   Q8_0 (weights, GGUF): per 32 values one 34-byte block: fp16 scale d
 *     (little-endian) followed by 32 int8 quants q; value = d * q.
 *   Q8_1 (activations, produced on the device): per 32 values
 *     d = amax/127 (fp32), q = roundf(x * (1/d)) (int8), stored scale fp16(d).
 *     This library stores the quants as int8 and the stored scale widened to
 *     fp32 (exactly the fp16 value); the Q8_1 sum field d*sum(q) is only
 *     consumed by weight formats with an offset, so it is not produced.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_FFN_ABI_VERSION 1

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,        /* null required pointer, N < 1, top_k > E, ... */
    MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* D/F/Fs not a multiple of 32, E > 1024, sizes overflow */
    MOE_ERR_WORKSPACE_TOO_SMALL = -3,
    MOE_ERR_CUDA = -4,               /* a CUDA call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = -5,     /* a bounded device-side wait gave up */
    MOE_ERR_UNSUPPORTED_DEVICE = -6, /* not compute capability 10.3 */
    MOE_ERR_BAD_ROUTING = -7,        /* expert index out of range / selected twice */
    MOE_ERR_BAD_CSR = -8             /* CSR offsets or token indices out of range */
};

/* Device status word bits (moe_workspace_status returns the word; a nonzero
 * word maps to the first matching moe_status in this order). */
#define MOE_DEV_BAD_ROUTING 0x1u
#define MOE_DEV_BAD_CSR 0x2u
#define MOE_DEV_TIMEOUT 0x4u

/* Human-readable name of a moe_status code (static string, never NULL). */
const char *moe_status_string(int status);

/* MOE_FFN_ABI_VERSION of the loaded library. */
int moe_abi_version(void);

/* Path selection for moe_grouped_ffn_ex / moe_ffn_prefill_ex. */
enum moe_path {
    MOE_PATH_AUTO = 0,   /* tensor-core grouped GEMM for prefill batches, matvec for small N */
    MOE_PATH_MATVEC = 1, /* fused gather-matvec (dp4a int8 dots), any N */
    MOE_PATH_TENSOR = 2  /* tcgen05 grouped GEMM (needs the shapes above) */
};

/* ---------------------------------------------------------------------------
 * Expert weights.  moe_weights_create copies the caller's Q8_0 tensors into a
 * library-owned device copy laid out for the kernels (int8 quants and fp32
 * scales split apart; a second copy of the quants as exact fp16 integers in
 * 128-row tiles for the tensor cores).  It allocates device memory and
 * synchronises `stream`.  The caller's buffers may be freed afterwards.
 *   gate_q8_0, up_q8_0 : device, Q8_0 blocks [E][F][D/32]  (row f reduces over D)
 *   down_q8_0          : device, Q8_0 blocks [E][D][F/32]
 *   sh_gate, sh_up     : device, Q8_0 blocks [Fs][D/32], or NULL when Fs == 0
 *   sh_down            : device, Q8_0 blocks [D][Fs/32], or NULL when Fs == 0
 * Returns MOE_ERR_UNSUPPORTED_DEVICE on anything but compute capability 10.3.
 * ------------------------------------------------------------------------- */
typedef struct moe_weights_s *moe_weights_t;

int moe_weights_create(moe_weights_t *out, int E, int D, int F,
                       const void *gate_q8_0, const void *up_q8_0, const void *down_q8_0,
                       int Fs, const void *sh_gate_q8_0, const void *sh_up_q8_0,
                       const void *sh_down_q8_0, cudaStream_t stream);

/* Block format of the caller's expert weights. */
enum moe_weight_format {
    MOE_WFMT_Q8_0 = 0, /* GGUF Q8_0: 34-byte blocks of 32 (fp16 d, 32 int8) */
    MOE_WFMT_Q4_K = 1, /* GGUF Q4_K: 144-byte super-blocks of 256 (fp16 d, fp16 dmin, 12 bytes
                          of 6-bit sub-block scales sc_j and mins m_j, 128 bytes of 4-bit
                          quants q): value = d*sc_j*q - dmin*m_j ("Q8_0/Q4_K MMQ", #406
                          references).  Needs D, F, Fs multiples of 256. */
    MOE_WFMT_Q3_K = 2  /* GGUF Q3_K: 110-byte super-blocks of 256 (32 bytes of high bits, 64
                          bytes of 2-bit low parts, 12 bytes of sixteen 6-bit scales s_j + 32,
                          fp16 d): value = d*s_j*q, q in [-4, 3], one s_j per 16 values (the
                          routed experts' format on the Carnice prefill page, #388 "Key
                          references").  Needs D, F, Fs multiples of 256. */
};
/* moe_weights_create for either format: the same arrays, rows in `format`'s
 * blocks ([E][F][D/256] super-blocks for Q4_K gate/up, [E][D][F/256] down,
 * and likewise for the shared expert).  A Q4_K layer computes, per 32-wide
 * sub-block b, the exact int32 dot of the quants (0..15) with the Q8_1
 * activation codes and the code sum of the activation block:
 *   sum_b d_x[b] * (d*sc_b * isum_b - dmin*m_b * xsum_b).
 * A Q3_K layer folds the 16-wide sub-block scales into the integer codes at
 * load time: per 32-wide block b it stores c_i = -s_j*q_i (always in
 * [-128, 124], one int8) with the block scale -d, and computes
 *   sum_b d_x[b] * (-d) * (sum_i c_i * x_i) = sum_b d_x[b] * d * (s_2b*isum_2b + s_2b+1*isum_2b+1),
 * the same exact block integer as the format's own definition (the signs
 * cancel in every product).
 * MOE_ERR_UNSUPPORTED_SHAPE for shapes the format cannot hold; an unknown
 * format is MOE_ERR_INVALID_ARG. */
int moe_weights_create_ex(moe_weights_t *out, int format, int E, int D, int F,
                          const void *gate, const void *up, const void *down, int Fs,
                          const void *sh_gate, const void *sh_up, const void *sh_down,
                          cudaStream_t stream);
/* MOE_WFMT_* of a weights handle, or MOE_ERR_INVALID_ARG for NULL. */
int moe_weights_format(moe_weights_t w);
int moe_weights_destroy(moe_weights_t w);
/* Shape of a weights handle (any output pointer may be NULL; host pointers). */
int moe_weights_shape(moe_weights_t w, int *E, int *D, int *F, int *Fs);
/* Library-owned device bytes held by the handle. */
size_t moe_weights_device_bytes(moe_weights_t w);
/* 1 when the tensor-core path can run on these weights (shapes and build), else 0. */
int moe_weights_tensor_path(moe_weights_t w);

/* ---------------------------------------------------------------------------
 * Workspace: one caller-owned device buffer per concurrent call chain.  The
 * first 256 bytes hold the device status word (and the bucketing kernel's
 * grid-barrier words and the small-batch routing's arrival counter, all zero
 * between calls).  moe_workspace_init zeroes those 256 bytes
 * (asynchronously); moe_workspace_status synchronises the
 * stream, returns the status word (host int, MOE_DEV_* bits) and, when
 * clear != 0, zeroes it.  Two call chains must not share a workspace.
 * moe_ffn_workspace_size covers every entry point below for that shape.
 * ------------------------------------------------------------------------- */
size_t moe_ffn_workspace_size(int N, int D, int E, int F, int top_k, int Fs);
int moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);
int moe_workspace_status(void *ws, int clear, cudaStream_t stream);
/* Map a status word to the moe_status code of its first error (MOE_OK if 0). */
int moe_status_from_word(int word);

/* ---------------------------------------------------------------------------
 * moe_router_topk -- router, softmax, top-k, shared gate, Q8_1 of x (#388
 * breakdown table "router" row: matvec + softmax + top-k + shexp-gate;
 * levers item 1: norm[N x embDim] x routerW[numExperts x embDim]).
 *   hidden     [N][D] fp32          routerW [E][D] fp32
 *   shexp_gate [D] fp32 or NULL     (shared-expert gate vector)
 *   topk_idx   [N][top_k] int32 out: experts by decreasing logit, ties to
 *              the lower index (slot 0 = largest)
 *   topk_w     [N][top_k] fp32 out: softmax over all E experts at the
 *              selected experts; divided by their sum when norm_topk_prob
 *   shexp_scale [N] fp32 out, sigmoid(hidden[t] . shexp_gate); NULL iff
 *              shexp_gate is NULL
 *   x_q [N][D] int8 out, x_d [N][D/32] fp32 out: Q8_1 of hidden
 *   logits_out [N][E] fp32 out or NULL (the router logits)
 *   ws: workspace (split-K partial logits).
 * ------------------------------------------------------------------------- */
int moe_router_topk(const float *hidden, const float *routerW, const float *shexp_gate,
                    int N, int D, int E, int top_k, int norm_topk_prob,
                    int32_t *topk_idx, float *topk_w, float *shexp_scale,
                    int8_t *x_q, float *x_d, float *logits_out,
                    void *ws, size_t ws_bytes, cudaStream_t stream);

/* moe_router_topk for callers that cannot allocate device memory (no
 * counterpart on the pages: it exists only for hosts whose device memory is
 * owned by another allocator, or that forbid cudaMalloc after start-up).  Same
 * arguments and results as moe_router_topk, without the workspace: the router's
 * split-K partial logits go to a 16 MiB array inside the library (2^22 floats,
 * held on every GPU that loads the library until exit).  The problem must fit:
 * nsplit * N * (E + 1) <= 2^22 floats, nsplit being the router's split-K factor:
 * 1 when N <= 8 and D % 4 == 0; otherwise, with tiles = ceil(N/64)*ceil(E/64)
 * and SMs the current device's multiprocessor count, the largest s that
 * divides D/32 with s <= min(ceil(4*SMs/tiles), D/depth), depth = 32 when
 * tiles <= 4 and 128 otherwise (so at most min(4*SMs, D/32)).  A problem that
 * does not fit returns MOE_ERR_WORKSPACE_TOO_SMALL and nothing runs.  The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress, which may load the library's kernels onto that device)
 * and should therefore come before any stream capture.  All calls on a device
 * share the array, so calls that may overlap on the GPU race and must be
 * ordered by the caller.  Allocates nothing. */
int moe_router_topk_noalloc(const float *hidden, const float *routerW, const float *shexp_gate,
                            int N, int D, int E, int top_k, int norm_topk_prob,
                            int32_t *topk_idx, float *topk_w, float *shexp_scale,
                            int8_t *x_q, float *x_d, float *logits_out, cudaStream_t stream);

/* Softmax + top-k alone, from given logits [N][E] (same outputs as above).
 * Lets a caller check routing against logits computed elsewhere. */
int moe_topk_from_logits(const float *logits, int N, int E, int top_k, int norm_topk_prob,
                         int32_t *topk_idx, float *topk_w, cudaStream_t stream);

/* Q8_1 quantisation of n_blocks consecutive 32-value blocks: q [n_blocks*32]
 * int8, d [n_blocks] fp32 (the fp16 stored scale, widened).  The same rule
 * moe_router_topk applies to hidden. */
int moe_quantize_q8_1(const float *x, int64_t n_blocks, int8_t *q, float *d, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * moe_bucket -- expert bucketing into a CSR on the device (#388 levers item 1:
 * expStart/expTokI/expTokK).  A counting sort of the N*top_k (token, slot)
 * pairs by expert, stable in token order:
 *   expStart [E+1] int32 out: segment offsets, expStart[0] = 0,
 *            expStart[E] = N*top_k
 *   expTokI  [N*top_k] int32 out: token of each entry (ascending per segment)
 *   expTokK  [N*top_k] int32 out: top-k slot of that token for this expert
 * A bad index or a repeated expert within a token sets MOE_DEV_BAD_ROUTING
 * and leaves every segment empty.  One cooperative kernel: each CTA counts a
 * token range, a grid barrier, then every CTA scans the count table and
 * scatters its range (histogram, scan and scatter in one launch).
 * ws: 256-byte aligned, at least moe_bucket_workspace_size(N, top_k, E)
 * bytes (a moe_ffn_workspace_size workspace of the same N, E, top_k always
 * is), initialised once by moe_workspace_init; the barrier keeps its words at
 * zero between calls.  If the barrier times out (MOE_DEV_TIMEOUT) the outputs
 * are undefined; run moe_workspace_init before the next call.
 * ------------------------------------------------------------------------- */
size_t moe_bucket_workspace_size(int N, int top_k, int E);
int moe_bucket(const int32_t *topk_idx, int N, int top_k, int E,
               int32_t *expStart, int32_t *expTokI, int32_t *expTokK,
               void *ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * moe_grouped_ffn -- every routed expert over its CSR segment, plus the shared
 * expert over all tokens (#406 "The work" item 2: gather -> grouped GEMM ->
 * scatter; #129 intro: gate/up/down grouped by expert; #129 "Scope": the
 * optionally batched shared expert):
 *   for entry j of expert e (t = expTokI[j], s = expTokK[j]):
 *     h_j = Q8_1( SiLU(W_g[e] x_t) * (W_u[e] x_t) )      (x_t = Q8_1 row t)
 *     partials[t*top_k + s][0..D) = W_d[e] h_j            (fp32, unweighted)
 *   shared (when the weights have Fs > 0 and shared_out != NULL):
 *     shared_out[t][0..D) = shexp_scale[t] * W_sd Q8_1(SiLU(W_sg x_t) * (W_su x_t))
 *   x_q [N][D] int8, x_d [N][D/32] fp32: Q8_1 rows (moe_router_topk output)
 *   partials [N*top_k][D] fp32 out; shared_out [N][D] fp32 out or NULL.
 * Every dot product is a sum over 32-blocks of fp16(d_w)*d_x*isum with isum
 * the exact int32 dot of the block's quants.
 * ------------------------------------------------------------------------- */
int moe_grouped_ffn(moe_weights_t w, const int8_t *x_q, const float *x_d,
                    const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                    int N, int top_k, const float *shexp_scale, float *partials, float *shared_out,
                    void *ws, size_t ws_bytes, cudaStream_t stream);

/* As moe_grouped_ffn with an explicit path (enum moe_path). */
int moe_grouped_ffn_ex(moe_weights_t w, const int8_t *x_q, const float *x_d,
                       const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                       int N, int top_k, const float *shexp_scale, float *partials, float *shared_out,
                       int path, void *ws, size_t ws_bytes, cudaStream_t stream);

/* The two halves of moe_grouped_ffn, for checking each on its own.
 * moe_expert_gate_up writes the requantised activations of every entry in
 * segment order: h_q [N*top_k][F] int8, h_d [N*top_k][F/32] fp32.
 * moe_expert_down consumes them (from any source) and writes partials. */
int moe_expert_gate_up(moe_weights_t w, const int8_t *x_q, const float *x_d,
                       const int32_t *expStart, const int32_t *expTokI, int N, int top_k,
                       int8_t *h_q, float *h_d, int path, void *ws, size_t ws_bytes,
                       cudaStream_t stream);
int moe_expert_down(moe_weights_t w, const int8_t *h_q, const float *h_d,
                    const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                    int N, int top_k, float *partials, int path, void *ws, size_t ws_bytes,
                    cudaStream_t stream);

/* Raw int32 block dot products of the gate/up GEMM for one 32-block `block`
 * of the reduction dimension: dots [N*top_k][2][F] int32, entry j in segment
 * order, [.][0][f] = isum(W_g[e][f], x_t), [.][1][f] = isum(W_u[e][f], x_t),
 * as computed inside the selected path's kernel.  The weight codes are the
 * stored ones: Q8_0 quants, Q4_K quants 0..15, and for Q3_K c_i = -s_j*q_i,
 * so a Q3_K dot is -(s_2b*isum_2b + s_2b+1*isum_2b+1). */
int moe_debug_gate_up_block_dots(moe_weights_t w, const int8_t *x_q, const float *x_d,
                                 const int32_t *expStart, const int32_t *expTokI, int N, int top_k,
                                 int block, int32_t *dots, int path, void *ws, size_t ws_bytes,
                                 cudaStream_t stream);

/* Raw int32 block dot products of the down GEMM for one 32-block `block` of
 * its reduction dimension (the intermediate size F), given requantised
 * activations h_q [N*top_k][F] int8 and h_d [N*top_k][F/32] fp32 in segment
 * order (as moe_expert_gate_up writes them): dots [N*top_k][D] int32, entry j
 * in segment order, [j][c] = isum(W_d[e][c], h_j) over block `block`, as
 * computed inside the selected path's kernel (stored weight codes, as for
 * moe_debug_gate_up_block_dots).  expTokK is needed because the tensor path's
 * plan (and its partial rows, written to the workspace) uses it.  Same errors
 * as moe_expert_down; block outside [0, F/32) is MOE_ERR_UNSUPPORTED_SHAPE. */
int moe_debug_down_block_dots(moe_weights_t w, const int8_t *h_q, const float *h_d,
                              const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                              int N, int top_k, int block, int32_t *dots, int path, void *ws,
                              size_t ws_bytes, cudaStream_t stream);

/* Failure-detection check of the bucketing kernel's grid barrier: runs
 * moe_bucket with the barrier waiting for one more arrival than there are
 * CTAs, so it can never complete, and a wait limit of limit_ms (1..2000)
 * instead of the normal 1 s.  Every CTA gives up after the limit, sets
 * MOE_DEV_TIMEOUT in the workspace status word and returns without writing
 * the CSR; the context stays usable.  The barrier's words are left mid-count:
 * call moe_workspace_init before the workspace serves another call.  Needs a
 * batch large enough for more than one token range (otherwise there is no
 * barrier): MOE_ERR_UNSUPPORTED_SHAPE.  Same arguments as moe_bucket. */
int moe_debug_bucket_barrier_timeout(const int32_t *topk_idx, int N, int top_k, int E,
                                     int32_t *expStart, int32_t *expTokI, int32_t *expTokK,
                                     int limit_ms, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Failure-detection check of the tensor path: runs the gate/up grouped GEMM with
 * its TMA producer told to issue nothing, so the MMA's first wait can never be
 * satisfied.  Every device wait is bounded; after limit_ms (1..2000) the kernel
 * gives up, sets MOE_DEV_TIMEOUT in the workspace status word, lets in-flight
 * work drain, frees its tensor memory and returns, leaving the context usable.
 * Returns the launch status; read the outcome with moe_workspace_status. */
int moe_debug_expert_wait_timeout(moe_weights_t w, const int8_t *x_q, const float *x_d,
                                  const int32_t *expStart, const int32_t *expTokI, int N, int top_k,
                                  int limit_ms, void *ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * moe_combine -- batched weighted scatter-reduce (#129 "Scope"), one launch
 * over N x D: for every token t and column c
 *   acc = +0.0f;
 *   for s = 0..top_k-1: acc = fmaf(topk_w[t][s], partials[t*top_k+s][c], acc);
 *   if (shared) acc = acc + shared[t][c];
 *   out[t][c] = acc;
 * in exactly this order and rounding (bit-reproducible).
 *   partials [N*top_k][D] fp32, topk_w [N][top_k] fp32, shared [N][D] or NULL,
 *   out [N][D] fp32 (may not alias the inputs).
 * ------------------------------------------------------------------------- */
int moe_combine(const float *partials, const float *topk_w, const float *shared,
                int N, int top_k, int D, float *out, cudaStream_t stream);
/* moe_combine followed by the residual add of the pages' per-layer combine,
 * (routed + shared) + resid ("Carnice prefill toward llama.cpp 676 t/s", #388,
 * "Dead ends"): after the shared row, acc = acc + residual[t][c] (one fp32
 * add), out[t][c] = acc.  residual [N][D] fp32, 16-byte aligned; it may be
 * `out` itself (an in-place residual update), otherwise it may not overlap
 * out.  residual == NULL is moe_combine. */
int moe_combine_residual(const float *partials, const float *topk_w, const float *shared,
                         const float *residual, int N, int top_k, int D, float *out,
                         cudaStream_t stream);
/* moe_combine_residual, then the next layer's input norm of every output row.
 * The pages feed the router a normalised activation ("Carnice prefill toward
 * llama.cpp 676 t/s", #388, "Remaining levers" item 1: norm[N x embDim] x
 * routerW) and chain the layers through this residual stream (item 2); the
 * norm is read as RMSNorm with a per-column weight:
 *   out[t][c]    = moe_combine_residual's value (bit for bit);
 *   normed[t][c] = (out[t][c] * r_t) * gamma[c],
 *   r_t          = 1 / sqrt(sum_c out[t][c]^2 / D + eps)   (fp32; the row sum in a
 *                  fixed order: each thread's columns, then a warp butterfly,
 *                  then the warps in order; 128 threads per row, or 512 when N
 *                  is below 8 times the SM count, so its grouping, and the last
 *                  bits of normed, depend on N).
 * residual [N][D] fp32, non-NULL (it may be `out`); gamma [D] fp32, device;
 * eps > 0 and finite; normed [N][D] fp32, overlapping neither out nor any
 * input; gamma and normed 16-byte aligned.  MOE_ERR_INVALID_ARG otherwise. */
int moe_combine_residual_rmsnorm(const float *partials, const float *topk_w, const float *shared,
                                 const float *residual, const float *gamma, float eps, int N,
                                 int top_k, int D, float *out, float *normed, cudaStream_t stream);
/* The same norm of rows x alone: normed[t][c] = (x[t][c] * r_t) * gamma[c],
 * r_t = 1 / sqrt(sum_c x[t][c]^2 / D + eps), summed as above (the input norm of
 * a stack's first layer).  x [N][D], gamma [D], normed [N][D] (not x): fp32,
 * device, 16-byte aligned; eps > 0 and finite. */
int moe_rmsnorm(const float *x, const float *gamma, float eps, int N, int D, float *normed,
                cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * moe_ffn_prefill -- the whole layer in one call (all of the above, on one
 * stream, with no host round trip): the pages' batched routed-MoE FFN over
 * N prompt tokens.
 *   hidden [N][D] fp32, routerW [E][D] fp32, shexp_gate [D] fp32 or NULL
 *   (NULL: no shared expert even if the weights carry one; non-NULL needs
 *   weights with Fs > 0), out [N][D] fp32 (the FFN output; no residual).
 * ------------------------------------------------------------------------- */
int moe_ffn_prefill(moe_weights_t w, const float *hidden, const float *routerW,
                    const float *shexp_gate, int N, int top_k, int norm_topk_prob, float *out,
                    void *ws, size_t ws_bytes, cudaStream_t stream);
int moe_ffn_prefill_ex(moe_weights_t w, const float *hidden, const float *routerW,
                       const float *shexp_gate, int N, int top_k, int norm_topk_prob, float *out,
                       int path, void *ws, size_t ws_bytes, cudaStream_t stream);
/* moe_ffn_prefill_ex whose combine also adds the residual row (moe_combine_residual):
 * out = residual + FFN(hidden).  residual [N][D] fp32, non-NULL, 16-byte aligned;
 * it may be `out` itself (the residual stream updated in place). */
int moe_ffn_prefill_residual(moe_weights_t w, const float *hidden, const float *routerW,
                             const float *shexp_gate, const float *residual, int N, int top_k,
                             int norm_topk_prob, float *out, int path, void *ws, size_t ws_bytes,
                             cudaStream_t stream);
/* moe_ffn_prefill_residual whose combine also writes the next layer's normalised
 * input (moe_combine_residual_rmsnorm): out = residual + FFN(hidden), normed =
 * RMSNorm(out) * gamma.  Arguments as there and as moe_combine_residual_rmsnorm;
 * normed may be `hidden` itself (the router has read it before the combine writes). */
int moe_ffn_prefill_residual_rmsnorm(moe_weights_t w, const float *hidden, const float *routerW,
                                     const float *shexp_gate, const float *residual,
                                     const float *gamma, float eps, int N, int top_k,
                                     int norm_topk_prob, float *out, float *normed, int path,
                                     void *ws, size_t ws_bytes, cudaStream_t stream);

/* moe_ffn_prefill_ex with hidden and out in HOST memory (the layer as a host
 * program calls it).  No staging copies: the router reads the hidden rows and
 * the combine writes the output rows in place over the host link (NVLink-C2C
 * on Grace-Blackwell), so that traffic overlaps the two kernels' own work.
 *   hidden_host [N][D] fp32, out_host [N][D] fp32: host memory the device can
 *   address -- pinned (cudaHostAlloc, cudaHostRegister) on any system, or any
 *   host allocation where the device reports pageable access through the host
 *   page tables.  Device (or managed) memory, or unreachable host memory:
 *   MOE_ERR_INVALID_ARG and nothing is launched.  out_host may not alias
 *   hidden_host.  routerW, shexp_gate, ws as for moe_ffn_prefill (device
 *   memory).  The call is asynchronous like the others: out_host holds the
 *   result once `stream` has reached the end of it. */
int moe_ffn_prefill_host(moe_weights_t w, const float *hidden_host, const float *routerW,
                         const float *shexp_gate, int N, int top_k, int norm_topk_prob,
                         float *out_host, int path, void *ws, size_t ws_bytes, cudaStream_t stream);
/* 1 when `p` is host memory the current device can address (what
 * moe_ffn_prefill_host accepts), 0 otherwise (device or managed memory,
 * NULL, or pageable memory on a system without host page-table access). */
int moe_host_memory_addressable(const void *p);
/* The host NUMA node closest to the current device (where the host buffers of
 * moe_ffn_prefill_host cross the fewest links: on a multi-socket host, memory
 * of another socket is reached through the inter-socket link as well), or -1
 * when the system reports no NUMA placement.  *node: host pointer.  Returns 0,
 * MOE_ERR_INVALID_ARG for NULL, MOE_ERR_CUDA if the query fails. */
int moe_device_host_numa_node(int *node);

/* A stack of routed-MoE FFN layers applied in place, one after another on
 * `stream`: for l = 0..n_layers-1, hidden <- hidden + FFN_l(hidden), each
 * layer exactly as moe_ffn_prefill_residual computes it with the residual
 * and output both `hidden` (so the results equal n_layers such calls bit for
 * bit).  Layer l uses weights w[l], routerW[l] and shexp_gate[l] (the array
 * itself may be NULL when no layer has a shared expert; entries may be NULL
 * per layer).  w, routerW and shexp_gate are HOST arrays of n_layers handles
 * / device pointers.  Every layer shares N, top_k, norm_topk_prob, path and
 * the workspace, which must be large enough for each layer's shapes (same D
 * in every layer).  From the second layer on, the router is launched so that
 * it may start while the previous layer's combine is still running
 * (cross-layer overlap, #388 "Remaining levers" 2): it first pulls its own
 * router weights into L2, then waits on the device for the previous layer's
 * output before reading it.  Errors as moe_ffn_prefill; nothing is launched
 * when an argument check fails. */
int moe_ffn_prefill_stack(const moe_weights_t *w, const float *const *routerW,
                          const float *const *shexp_gate, int n_layers, float *hidden, int N,
                          int top_k, int norm_topk_prob, int path, void *ws, size_t ws_bytes,
                          cudaStream_t stream);
/* moe_ffn_prefill_stack with an input norm before every layer (the pre-norm
 * chain the pages' router input implies, #388 "Remaining levers" items 1-2):
 *   normed = RMSNorm_0(hidden);  for l: hidden = hidden + FFN_l(normed),
 *   normed = RMSNorm_{l+1}(hidden) (fused into layer l's combine; after the last
 *   layer only when gamma[n_layers] is not NULL).
 * gamma: host array of n_layers + 1 device pointers to [D] fp32 weights (the
 * last may be NULL); normed [N][D] fp32 device (not hidden), holds the last
 * norm on return; eps > 0 and finite.  Every router after the first norm is
 * launched behind the kernel that writes its input.  Errors as
 * moe_ffn_prefill_stack. */
int moe_ffn_prefill_stack_rmsnorm(const moe_weights_t *w, const float *const *routerW,
                                  const float *const *shexp_gate, const float *const *gamma,
                                  float eps, int n_layers, float *hidden, float *normed, int N,
                                  int top_k, int norm_topk_prob, int path, void *ws,
                                  size_t ws_bytes, cudaStream_t stream);

/* moe_ffn_prefill_ex that also records seven caller-created CUDA events on
 * `stream` around its stages, for measuring each kernel in place:
 *   [0] start, [1] after the router (+softmax/top-k/Q8_1), [2] after bucketing
 *   (which on the tensor path also writes the GEMM plan), [3] after the gather
 *   (tensor path; nothing on the matvec path), [4] after gate/up, [5] after
 *   down (both incl. the shared expert), [6] after the combine.
 * stage_events: host array of 7 cudaEvent_t (created by the caller). */
int moe_ffn_prefill_timed(moe_weights_t w, const float *hidden, const float *routerW,
                          const float *shexp_gate, int N, int top_k, int norm_topk_prob, float *out,
                          int path, void *ws, size_t ws_bytes, cudaStream_t stream,
                          cudaEvent_t *stage_events);

/* Device pointers to the intermediates moe_ffn_prefill leaves in `ws`
 * (valid after it ran on that workspace with the same shape); any output
 * pointer may be NULL.  Host pointers to receive device addresses. */
int moe_workspace_views(void *ws, int N, int D, int E, int F, int top_k, int Fs,
                        int32_t **topk_idx, float **topk_w, float **shexp_scale,
                        int8_t **x_q, float **x_d, int32_t **expStart, int32_t **expTokI,
                        int32_t **expTokK, float **partials, float **shared_out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FFN_H */
