// moe_internal.cuh -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_ffn.h"

namespace moe {

constexpr int QK = 32;          // values per Q8 block (and per Q4_K sub-block)
constexpr int QK_K = 256;       // values per K-quant super-block
constexpr int Q4_K_BYTES = 144; // fp16 d, fp16 dmin, 12 bytes of 6-bit scales/mins, 128 bytes of nibbles
constexpr int Q3_K_BYTES = 110; // 32 bytes high bits, 64 bytes 2-bit low parts, 12 bytes 6-bit scales, fp16 d
constexpr int Q8_0_BYTES = 34;  // fp16 scale + 32 int8
constexpr int MAX_E = 1024;
constexpr int SEG_ALIGN = 16;   // padded segment start (rows) in the tensor-core row space
constexpr int TILE_M = 128;     // weight rows per tensor-core tile
constexpr int TILE_N = 96;      // token rows per tensor-core tile (max)

// ---------------------------------------------------------------- weights --
// Library-owned device copy of the expert weights (see moe_weights_create).
struct WeightSet {
    int rows_gu = 0;  // 2*F (gate and up, tile-interleaved for the tensor path)
    int F = 0;        // intermediate size of this set
    // int8 quants + fp32 scales, row-major, for the matvec path
    int8_t *gate_q = nullptr, *up_q = nullptr;  // [nexp][F][D]
    float *gate_d = nullptr, *up_d = nullptr;   // [nexp][F][D/32]
    int8_t *down_q = nullptr;                   // [nexp][D][F]
    float *down_d = nullptr;                    // [nexp][D][F/32]
    // Q4_K only: per-32-block mins dmin*m (the weight is d*sc*q - dmin*m, quants 0..15 above)
    float *gate_m = nullptr, *up_m = nullptr, *down_m = nullptr;  // same shapes as the scales
    // Q4_K only: the quants packed two per byte, 16 bytes per 32-block: byte j of a block holds
    // q[j] in its low and q[j + 16] in its high nibble (the decode ring's stream: half the bytes)
    uint8_t *gate_p = nullptr, *up_p = nullptr;  // [nexp][F][D/2]
    uint8_t *down_p = nullptr;                   // [nexp][D][F/2]
    // tensor path: exact fp16 integers in tile-interleaved order + transposed scales
    __half *gu16 = nullptr;   // [nexp][2F][D]: 128-row tile mt = 64 gate rows then 64 up rows
    float *gu_dT = nullptr;   // [nexp][D/32][2F] (same row order)
    __half *dn16 = nullptr;   // [nexp][D][F]
    float *dn_dT = nullptr;   // [nexp][F/32][D]
    float *gu_mT = nullptr;   // Q4_K: mins, as gu_dT
    float *dn_mT = nullptr;   // Q4_K: mins, as dn_dT
};

}  // namespace moe

struct moe_weights_s {
    int E = 0, D = 0, F = 0, Fs = 0;
    int device = -1;
    int wfmt = MOE_WFMT_Q8_0;  // block format of the caller's expert weights
    bool tensor_ok = false;  // shapes fit the tensor-core path
    moe::WeightSet routed;   // E experts
    moe::WeightSet shared;   // 1 expert (Fs > 0)
    size_t bytes = 0;
    char *routed_arena_ = nullptr;  // one device allocation holding both weight sets
    void *tmaps = nullptr;   // host copy of the TMA descriptors (tensor path), owned
};

namespace moe {

// ------------------------------------------------------------- workspace --
struct WsLayout {
    size_t status, topk_idx, topk_w, shexp_scale, x_q, x_d, expStart, expTokI, expTokK;
    size_t partials, shared_out, part_logits, total;
    // tensor path
    size_t plan, tiles, rowinfo, xg16, xg_dT, h16, h_dT;
    size_t xg_sT, h_sT;  // Q4_K: per-block code sums times scale ([K/32][rows], as the scales)
    // matvec path
    size_t hq8, hd8;
    int nsplit;      // router split-K factor
    int rows_max;    // padded row space of the tensor path
    int tiles_max;   // token tiles of the tensor path
};

WsLayout ws_layout(int N, int D, int E, int F, int top_k, int Fs);
// The shape rules every entry point applies to (N, D, E, top_k) (moe_api.cu).
bool shape_ok(int N, int D, int E, int top_k);
// router.cu: the split-K factor of the router for a batch (workspace layout), and the split its
// launch actually uses (1 for batches of at most 8 tokens with D % 4 == 0, which the one-pass
// small-batch kernel routes); its partial-logit table holds split * N * (E + 1) floats.
int router_nsplit(int N, int D, int E);
int router_split_used(int N, int D, int E);

template <typename T>
inline T *ws_ptr(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(ws) + off); }

// Plan header written by the planning kernel (tensor path), at ws + plan.
struct PlanHeader {
    int n_tiles;        // token tiles (routed + shared)
    int n_rows;         // padded rows used
    int shared_row0;    // first padded row of the shared segment (-1: none)
    int pad;
};
// One token tile: padded row start, valid rows, expert (E = shared), segment entry start.
struct TileDesc {
    int row0, nrows, expert, entry0;
};

// Token rows per tile in the tensor path's plan for these weights (the plan is written by the
// bucketing kernel or plan_kernel and read by the grouped GEMM).
inline int plan_tile_rows(const moe_weights_s *) { return TILE_N; }

// ----------------------------------------------------------- launchers --
// router.cu
// status (nullable): the workspace's status word; with it, batches the tensor-core router can take
// (router_tc_eligible) run there (part_logits unused), without it on the fp32 SIMT router.
// tile_counts (nullable; with status): ask the tensor-core router for the bucketing kernel's count
// table of 128-token ranges; *counted tells whether it wrote it.
int launch_router(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D,
                  int E, int top_k, int norm, int32_t *topk_idx, float *topk_w, float *shexp_scale,
                  int8_t *x_q, float *x_d, float *logits_out, float *part_logits, int nsplit,
                  cudaStream_t s, bool early = false, unsigned *status = nullptr, int *tile_counts = nullptr,
                  bool *counted = nullptr);
// router_tc.cu: logits on the tensor cores (split tf32, three MMAs per K step) with the Q8_1 of x
// and the per-token softmax / top-k in one cluster launch; E % 8 == 0, 8 <= E <= 256, N > 8,
// 16-byte-aligned hidden / routerW / gate.
bool router_tc_eligible(int N, int D, int E, bool has_gate, const float *hidden, const float *routerW,
                        const float *shexp_gate);
int launch_router_tc(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D, int E,
                     int top_k, int norm, int32_t *topk_idx, float *topk_w, float *shexp_scale, int8_t *x_q,
                     float *x_d, float *logits_out, unsigned *status, cudaStream_t s, bool early,
                     int *tile_counts = nullptr);
int launch_topk_from_logits(const float *logits, int N, int E, int top_k, int norm, int32_t *idx,
                            float *w, cudaStream_t s);
// early (both routers): launched to overlap the kernel before it, the previous layer's combine (see
// launch_early); the router kernels wait on the device before reading hidden.
// router + softmax/top-k + bucketing of a batch of at most 8 tokens in one launch (counter: an
// arrival word in the workspace's status block, ROUTE_COUNTER_OFFSET, zero between launches);
// MOE_ERR_UNSUPPORTED_SHAPE when the batch is too large for it.
constexpr size_t ROUTE_COUNTER_OFFSET = 192;
int launch_route_small(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D, int E,
                       int top_k, int norm, int32_t *topk_idx, float *topk_w, float *shexp_scale, int8_t *x_q,
                       float *x_d, float *part_logits, int32_t *expStart, int32_t *expTokI, int32_t *expTokK,
                       unsigned *counter, unsigned *status, cudaStream_t s, bool early = false);
int launch_quantize_q8_1(const float *x, int64_t nblk, int8_t *q, float *d, cudaStream_t s);
// bucket.cu
// ws: the workspace (status word at 0, the grid barrier's two words at BUCKET_BARRIER_OFFSET
// and +64, the small-batch routing's arrival counter at ROUTE_COUNTER_OFFSET, the per-range
// count table at BUCKET_SCRATCH_OFFSET, bucket_scratch_bytes long).
// L non-null: also write the tensor path's plan into ws (layout L).
constexpr size_t BUCKET_BARRIER_OFFSET = 64;
constexpr size_t BUCKET_SCRATCH_OFFSET = 256;
constexpr int BUCKET_TABLE_MAX = 65536;  // ints in the ranges x experts count table
int bucket_grid(int N, int E, int *range_out);
size_t bucket_scratch_bytes(int N, int E);
int launch_bucket(const int32_t *topk_idx, int N, int top_k, int E, int32_t *expStart, int32_t *expTokI,
                  int32_t *expTokK, void *ws, cudaStream_t s, const WsLayout *L = nullptr, bool with_shared = false,
                  int tile_rows = TILE_N, unsigned long long barrier_ns = 0, int extra_arrivals = 0,
                  bool counts_ready = false);
// expert_matvec.cu
int launch_matvec_gate_up(const moe_weights_s *w, const WeightSet &ws, bool is_shared,
                          const int8_t *x_q, const float *x_d, const int32_t *expStart,
                          const int32_t *expTokI, int N, int top_k, int8_t *h_q, float *h_d,
                          int32_t *dbg_dots, int dbg_block, unsigned *status, cudaStream_t s);
// early: launched to overlap the kernel before it (which must be a matvec gate/up launch of the
// same call); the CSR must come from a kernel further back.
int launch_matvec_down(const moe_weights_s *w, const WeightSet &ws, bool is_shared,
                       const int8_t *h_q, const float *h_d, const int32_t *expStart,
                       const int32_t *expTokI, const int32_t *expTokK, int N, int top_k,
                       const float *shexp_scale, float *out, unsigned *status, cudaStream_t s,
                       bool early = false, int32_t *dbg_dots = nullptr, int dbg_block = -1);
// combine.cu
// early: launched to overlap the kernel before it (see launch_early); topk_w must come from a
// kernel further back.
int launch_combine(const float *partials, const float *topk_w, const float *shared, const float *residual, int N,
                   int top_k, int D, float *out, cudaStream_t s, bool early = false);
// launch_combine with a residual, then RMSNorm of each output row into normed (gamma [D], eps > 0).
int launch_combine_rmsnorm(const float *partials, const float *topk_w, const float *shared, const float *residual,
                           const float *gamma, float eps, int N, int top_k, int D, float *out, float *normed,
                           cudaStream_t s, bool early = false);
// normed = RMSNorm(x) * gamma alone (launch_combine_rmsnorm with no slots and no out).
int launch_rmsnorm(const float *x, const float *gamma, float eps, int N, int D, float *normed, cudaStream_t s);
// weights.cu
int repack_weights(moe_weights_s *w, const void *gate, const void *up, const void *down,
                   const void *sh_gate, const void *sh_up, const void *sh_down, cudaStream_t s);
void free_weights(moe_weights_s *w);
// expert_gemm.cu (tensor path)
bool tensor_path_supported(const moe_weights_s *w);
// plan_ready: the plan was already written (by the bucketing kernel); only gather
int launch_plan_and_gather(const moe_weights_s *w, const int8_t *x_q, const float *x_d,
                           const int32_t *expStart, const int32_t *expTokI,
                           const int32_t *expTokK, int N, int top_k, bool with_shared,
                           void *ws, const WsLayout &L, cudaStream_t s, bool plan_ready = false);
int launch_gemm_gate_up(const moe_weights_s *w, int N, int top_k, bool with_shared, void *ws,
                        const WsLayout &L, int32_t *dbg_dots, int dbg_block, cudaStream_t s);
int launch_gemm_gate_up_starved(const moe_weights_s *w, int N, int top_k, void *ws, const WsLayout &L,
                                unsigned long long wait_ns, cudaStream_t s);
int launch_gemm_down(const moe_weights_s *w, int N, int top_k, bool with_shared,
                     const float *shexp_scale, float *partials, float *shared_out, void *ws,
                     const WsLayout &L, cudaStream_t s, int32_t *dbg_dots = nullptr, int dbg_block = -1);
int launch_h16_to_q8(const moe_weights_s *w, int N, int top_k, void *ws, const WsLayout &L,
                     int8_t *h_q, float *h_d, cudaStream_t s);
int launch_q8_to_h16(const moe_weights_s *w, int N, int top_k, void *ws, const WsLayout &L,
                     const int8_t *h_q, const float *h_d, cudaStream_t s);
int prepare_tensor_maps(moe_weights_s *w);
// Tensor map of a row-major fp32 matrix [rows][cols] read in 128-byte-swizzled boxes of 32
// columns x box_rows rows (false when the driver entry point or the encoding fails).
bool encode_fp32_sw128_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// matvec_ring.cu: the matvecs of batches of at most 8 tokens with the weight rows streamed through
// a shared-memory ring; eligible when the batch's activation rows and two stages fit on chip,
// K % 128 == 0 and every operand is 16-byte aligned.  Same arguments and results as launch_matvec_gate_up / launch_matvec_down.
bool matvec_ring_eligible(int N, int K, int rows_e, int n_xrows, int nexp, int entries, bool mins, const void *xq,
                          const void *xd, const WeightSet &set);
int launch_matvec_ring_gate_up(const WeightSet &set, int D, int F, int nexp, bool is_shared, const int8_t *x_q,
                               const float *x_d, const int32_t *expStart, const int32_t *expTokI, int N, int top_k,
                               int8_t *h_q, float *h_d, int32_t *dbg_dots, int dbg_block, unsigned *status,
                               cudaStream_t s);
int launch_matvec_ring_down(const WeightSet &set, int D, int F, int nexp, bool is_shared, const int8_t *h_q,
                            const float *h_d, const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                            int N, int top_k, const float *shexp_scale, float *out, unsigned *status, cudaStream_t s,
                            bool early, int32_t *dbg_dots, int dbg_block);

void free_tensor_maps(moe_weights_s *w);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

constexpr int MAX_DEVICES = 64;  // device ordinals the per-device caches below cover

// The current device's ordinal, or -1 when none can be queried.
inline int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return -1;
    return dev;
}
// The current device's multiprocessor count, queried once per device; 0 when there is no device.
int device_sm_count();

// Per-device record of the largest dynamic shared-memory size a kernel was opted into.
struct SmemOptIn {
    int bytes[MAX_DEVICES] = {};
};
// Raise a kernel's dynamic shared-memory limit to what a launch needs on the current device (the
// 48 KB that needs no opt-in counts static shared memory too, so every size is set explicitly);
// the attribute is per device, so the largest value set is remembered per kernel and device, and
// repeated launches -- also launches under stream capture -- make no further call.
inline int ensure_dynamic_smem(const void *kernel, size_t bytes, SmemOptIn *done) {
    const int dev = current_device();
    if (dev < 0) return MOE_ERR_CUDA;
    if ((int)bytes <= done->bytes[dev]) return MOE_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
    done->bytes[dev] = (int)bytes;
    return MOE_OK;
}
inline int launch_status() { return cuda_status(cudaGetLastError()); }

// Launches `kernel` so that it may start while the previous kernel on the stream is still
// running (programmatic dependent launch: it is scheduled once every CTA of that kernel has
// executed griddepcontrol.launch_dependents or exited).  The kernel must execute
// griddepcontrol.wait before it reads anything that kernel writes; without this launch
// attribute that wait returns at once.
template <typename... KArgs, typename... Args>
inline int launch_early(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...));
}

// ----------------------------------------------------- device helpers --
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Q8_1 quantisation of one 32-value block held one value per lane:
//   d = amax/127 (IEEE fp32 division), q = roundf(x * (1/d)), stored scale fp16(d).
// Returns q; *d16f receives the stored scale widened to fp32.
__device__ __forceinline__ int q8_quantize_lane(float x, float *d16f) {
    float a = fabsf(x);
    // |x| bit patterns order like the values for non-negative floats
    unsigned amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(a));
    float amax = __uint_as_float(amax_bits);
    float d = __fdiv_rn(amax, 127.0f);
    float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    *d16f = __half2float(__float2half_rn(d));
    return (int)roundf(__fmul_rn(x, id));
}

}  // namespace moe
