// moe_api.cu -- the C ABI (include/moe_ffn.h): argument checks, workspace
// layout and the launch sequence of each entry point.  No entry point on the
// hot path allocates or synchronises; only moe_ffn_prefill_host's kernels touch
// host memory (the caller's hidden and output rows, in place).
#include <algorithm>
#include <atomic>
#include <new>

#include "moe_internal.cuh"

using namespace moe;

namespace moe {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int device_sm_count() {
    static std::atomic<int> cached[MAX_DEVICES];
    const int dev = current_device();
    if (dev < 0) return 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

static bool tensor_shapes(int D, int F, int Fs) {
    return D % TILE_M == 0 && F % 64 == 0 && (Fs == 0 || Fs % 64 == 0);
}

WsLayout ws_layout(int N, int D, int E, int F, int top_k, int Fs) {
    WsLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align256(bytes);
        return o;
    };
    const size_t Nk = (size_t)N * top_k;
    const int Fmax = std::max(F, Fs);
    L.status = take(256);
    // the router's split-K scratch comes first: moe_router_topk, which knows only (N, D, E),
    // finds it at the same offset as every other entry point
    L.nsplit = router_nsplit(N, D, E);
    // ... and the bucketing's count table reuses it once the router is done with it
    L.part_logits = take(std::max((size_t)L.nsplit * N * (E + 1) * 4, bucket_scratch_bytes(N, E)));
    L.topk_idx = take(Nk * 4);
    L.topk_w = take(Nk * 4);
    L.shexp_scale = take((size_t)N * 4);
    L.x_q = take((size_t)N * D);
    L.x_d = take((size_t)N * (D / QK) * 4);
    L.expStart = take((size_t)(E + 1) * 4);
    L.expTokI = take(Nk * 4);
    L.expTokK = take(Nk * 4);
    L.partials = take(Nk * D * 4);
    L.shared_out = take(Fs ? (size_t)N * D * 4 : 0);
    L.hq8 = take((Nk + N) * Fmax);
    L.hd8 = take((Nk + N) * (Fmax / QK) * 4);
    if (tensor_shapes(D, F, Fs)) {
        // every segment start is 16-aligned; the row count is a multiple of 16 as well, so the
        // transposed scale arrays have 16-byte-aligned rows (a TMA requirement)
        L.rows_max = (int)((Nk + (size_t)SEG_ALIGN * (E + 2) + N + 15) / 16 * 16);
        L.tiles_max = (int)(Nk / TILE_N + E + 1 + N / TILE_N + 2);
        L.plan = take(sizeof(PlanHeader) + (size_t)(E + 2) * 4);
        L.tiles = take((size_t)L.tiles_max * sizeof(TileDesc));
        L.rowinfo = take((size_t)L.rows_max * 16);
        L.xg16 = take((size_t)L.rows_max * D * 2);
        L.xg_dT = take((size_t)(D / QK) * L.rows_max * 4);
        L.h16 = take((size_t)L.rows_max * Fmax * 2);
        L.h_dT = take((size_t)(Fmax / QK) * L.rows_max * 4);
        L.xg_sT = take((size_t)(D / QK) * L.rows_max * 4);
        L.h_sT = take((size_t)(Fmax / QK) * L.rows_max * 4);
    }
    L.total = off;
    return L;
}

bool shape_ok(int N, int D, int E, int top_k) {
    if (N < 1 || D < QK || D % QK != 0 || E < 1 || E > MAX_E || top_k < 1 || top_k > E || top_k > 32)
        return false;
    if ((int64_t)N * top_k > (int64_t)0x7fffffff / 2) return false;
    return true;
}

}  // namespace moe

namespace {

int check_ws(const void *ws, size_t ws_bytes, const WsLayout &L) {
    if (ws == nullptr) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_INVALID_ARG;
    return ws_bytes >= L.total ? MOE_OK : MOE_ERR_WORKSPACE_TOO_SMALL;
}

unsigned *status_word(void *ws) { return reinterpret_cast<unsigned *>(ws); }

int pick_path(const moe_weights_s *w, int N, int top_k, int path) {
    if (path == MOE_PATH_MATVEC) return MOE_PATH_MATVEC;
    if (path == MOE_PATH_TENSOR) return tensor_path_supported(w) ? MOE_PATH_TENSOR : -1;
    // auto: the tensor cores pay off once the average segment holds a tile's worth of rows
    if (!tensor_path_supported(w)) return MOE_PATH_MATVEC;
    const int64_t avg_rows = ((int64_t)N * top_k) / w->E;
    return (N >= 64 && avg_rows >= 8) ? MOE_PATH_TENSOR : MOE_PATH_MATVEC;
}

int grouped_ffn_impl(moe_weights_s *w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                     const int32_t *expTokI, const int32_t *expTokK, int N, int top_k,
                     const float *shexp_scale, float *partials, float *shared_out, int path, void *ws,
                     const WsLayout &L, cudaStream_t s, bool plan_ready = false) {
    unsigned *st = status_word(ws);
    const bool with_shared = shared_out != nullptr;
    if (path == MOE_PATH_TENSOR) {
        int rc = launch_plan_and_gather(w, x_q, x_d, expStart, expTokI, expTokK, N, top_k, with_shared, ws, L, s,
                                        plan_ready);
        if (!rc) rc = launch_gemm_gate_up(w, N, top_k, with_shared, ws, L, nullptr, -1, s);
        if (!rc) rc = launch_gemm_down(w, N, top_k, with_shared, shexp_scale, partials, shared_out, ws, L, s);
        return rc;
    }
    int8_t *hq = ws_ptr<int8_t>(ws, L.hq8);
    float *hd = ws_ptr<float>(ws, L.hd8);
    int rc = launch_matvec_gate_up(w, w->routed, false, x_q, x_d, expStart, expTokI, N, top_k, hq, hd, nullptr, -1,
                                   st, s);
    if (!rc)
        rc = launch_matvec_down(w, w->routed, false, hq, hd, expStart, expTokI, expTokK, N, top_k, nullptr, partials,
                                st, s);
    if (!rc && with_shared) {
        const size_t Nk = (size_t)N * top_k;
        int8_t *shq = hq + Nk * std::max(w->F, w->Fs);
        float *shd = hd + Nk * (std::max(w->F, w->Fs) / QK);
        rc = launch_matvec_gate_up(w, w->shared, true, x_q, x_d, nullptr, nullptr, N, top_k, shq, shd, nullptr, -1,
                                   st, s);
        if (!rc)
            rc = launch_matvec_down(w, w->shared, true, shq, shd, nullptr, nullptr, nullptr, N, top_k, shexp_scale,
                                    shared_out, st, s);
    }
    return rc;
}

}  // namespace

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
        case MOE_ERR_BAD_ROUTING: return "bad routing (expert index out of range or repeated)";
        case MOE_ERR_BAD_CSR: return "malformed CSR";
        default: return "unknown status";
    }
}

int moe_abi_version(void) { return MOE_FFN_ABI_VERSION; }

int moe_status_from_word(int word) {
    unsigned u = (unsigned)word;
    if (u & MOE_DEV_BAD_ROUTING) return MOE_ERR_BAD_ROUTING;
    if (u & MOE_DEV_BAD_CSR) return MOE_ERR_BAD_CSR;
    if (u & MOE_DEV_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
    return MOE_OK;
}

int moe_weights_create(moe_weights_t *out, int E, int D, int F, const void *gate, const void *up, const void *down,
                       int Fs, const void *sh_gate, const void *sh_up, const void *sh_down, cudaStream_t stream) {
    return moe_weights_create_ex(out, MOE_WFMT_Q8_0, E, D, F, gate, up, down, Fs, sh_gate, sh_up, sh_down, stream);
}

int moe_weights_format(moe_weights_t w) { return w ? w->wfmt : MOE_ERR_INVALID_ARG; }

int moe_weights_create_ex(moe_weights_t *out, int format, int E, int D, int F, const void *gate, const void *up,
                          const void *down, int Fs, const void *sh_gate, const void *sh_up, const void *sh_down,
                          cudaStream_t stream) {
    if (out == nullptr) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!gate || !up || !down) return MOE_ERR_INVALID_ARG;
    if (format != MOE_WFMT_Q8_0 && format != MOE_WFMT_Q4_K && format != MOE_WFMT_Q3_K) return MOE_ERR_INVALID_ARG;
    if (Fs < 0 || (Fs > 0 && (!sh_gate || !sh_up || !sh_down))) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > MAX_E || D < QK || D % QK || F < QK || F % QK || Fs % QK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (format != MOE_WFMT_Q8_0 && (D % QK_K || F % QK_K || Fs % QK_K)) return MOE_ERR_UNSUPPORTED_SHAPE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED_DEVICE;
    moe_weights_s *w = new (std::nothrow) moe_weights_s();
    if (!w) return MOE_ERR_CUDA;
    w->E = E;
    w->D = D;
    w->F = F;
    w->Fs = Fs;
    w->device = dev;
    w->wfmt = format;
    w->tensor_ok = tensor_shapes(D, F, Fs);
    int rc = repack_weights(w, gate, up, down, sh_gate, sh_up, sh_down, stream);
    if (!rc && w->tensor_ok) rc = prepare_tensor_maps(w);
    if (rc) {
        free_tensor_maps(w);
        free_weights(w);
        delete w;
        return rc;
    }
    *out = w;
    return MOE_OK;
}

int moe_weights_destroy(moe_weights_t w) {
    if (!w) return MOE_ERR_INVALID_ARG;
    free_tensor_maps(w);
    free_weights(w);
    delete w;
    return MOE_OK;
}

int moe_weights_shape(moe_weights_t w, int *E, int *D, int *F, int *Fs) {
    if (!w) return MOE_ERR_INVALID_ARG;
    if (E) *E = w->E;
    if (D) *D = w->D;
    if (F) *F = w->F;
    if (Fs) *Fs = w->Fs;
    return MOE_OK;
}

size_t moe_weights_device_bytes(moe_weights_t w) { return w ? w->bytes : 0; }

int moe_weights_tensor_path(moe_weights_t w) { return (w && tensor_path_supported(w)) ? 1 : 0; }

size_t moe_ffn_workspace_size(int N, int D, int E, int F, int top_k, int Fs) {
    if (!shape_ok(N, D, E, top_k) || F < QK || F % QK || Fs < 0 || Fs % QK) return 0;
    return ws_layout(N, D, E, F, top_k, Fs).total;
}

int moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(ws, 0, 256, stream));
}

int moe_workspace_status(void *ws, int clear, cudaStream_t stream) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (clear && word) {
        if (cudaMemsetAsync(ws, 0, sizeof(word), stream) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return (int)word;
}

int moe_router_topk(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D, int E,
                    int top_k, int norm_topk_prob, int32_t *topk_idx, float *topk_w, float *shexp_scale,
                    int8_t *x_q, float *x_d, float *logits_out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!hidden || !routerW || !topk_idx || !topk_w || !x_q || !x_d) return MOE_ERR_INVALID_ARG;
    if ((shexp_gate == nullptr) != (shexp_scale == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, D, E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    // only the router's own scratch is needed: status + partial logits
    const int nsplit = router_nsplit(N, D, E);
    const size_t need = 256 + align256((size_t)nsplit * N * (E + 1) * 4);
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    float *part = ws_ptr<float>(ws, 256);
    return launch_router(hidden, routerW, shexp_gate, N, D, E, top_k, norm_topk_prob ? 1 : 0, topk_idx, topk_w,
                         shexp_scale, x_q, x_d, logits_out, part, nsplit, stream, false, status_word(ws));
}

int moe_topk_from_logits(const float *logits, int N, int E, int top_k, int norm_topk_prob, int32_t *topk_idx,
                         float *topk_w, cudaStream_t stream) {
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, QK, E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return launch_topk_from_logits(logits, N, E, top_k, norm_topk_prob ? 1 : 0, topk_idx, topk_w, stream);
}

int moe_quantize_q8_1(const float *x, int64_t n_blocks, int8_t *q, float *d, cudaStream_t stream) {
    if (n_blocks < 0) return MOE_ERR_INVALID_ARG;
    if (n_blocks > 0 && (!x || !q || !d)) return MOE_ERR_INVALID_ARG;
    return launch_quantize_q8_1(x, n_blocks, q, d, stream);
}

size_t moe_bucket_workspace_size(int N, int top_k, int E) {
    if (!shape_ok(N, QK, E, top_k)) return 0;
    return moe::BUCKET_SCRATCH_OFFSET + moe::bucket_scratch_bytes(N, E);
}

int moe_bucket(const int32_t *topk_idx, int N, int top_k, int E, int32_t *expStart, int32_t *expTokI,
               int32_t *expTokK, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!topk_idx || !expStart || !expTokI || !expTokK || !ws) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, QK, E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_bucket_workspace_size(N, top_k, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return launch_bucket(topk_idx, N, top_k, E, expStart, expTokI, expTokK, ws, stream);
}

int moe_debug_bucket_barrier_timeout(const int32_t *topk_idx, int N, int top_k, int E, int32_t *expStart,
                                     int32_t *expTokI, int32_t *expTokK, int limit_ms, void *ws, size_t ws_bytes,
                                     cudaStream_t stream) {
    if (!topk_idx || !expStart || !expTokI || !expTokK || !ws || limit_ms < 1 || limit_ms > 2000)
        return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, QK, E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_bucket_workspace_size(N, top_k, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return launch_bucket(topk_idx, N, top_k, E, expStart, expTokI, expTokK, ws, stream, nullptr, false, TILE_N,
                         (unsigned long long)limit_ms * 1000000ull, 1);
}

int moe_grouped_ffn_ex(moe_weights_t w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                       const int32_t *expTokI, const int32_t *expTokK, int N, int top_k, const float *shexp_scale,
                       float *partials, float *shared_out, int path, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!w || !x_q || !x_d || !expStart || !expTokI || !expTokK || !partials) return MOE_ERR_INVALID_ARG;
    if (shared_out && (!shexp_scale || w->Fs == 0)) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, w->D, w->E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, w->D, w->E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    int p = pick_path(w, N, top_k, path);
    if (p < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    return grouped_ffn_impl(w, x_q, x_d, expStart, expTokI, expTokK, N, top_k, shexp_scale, partials, shared_out, p,
                            ws, L, stream);
}

int moe_grouped_ffn(moe_weights_t w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                    const int32_t *expTokI, const int32_t *expTokK, int N, int top_k, const float *shexp_scale,
                    float *partials, float *shared_out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return moe_grouped_ffn_ex(w, x_q, x_d, expStart, expTokI, expTokK, N, top_k, shexp_scale, partials, shared_out,
                              MOE_PATH_AUTO, ws, ws_bytes, stream);
}

int moe_expert_gate_up(moe_weights_t w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                       const int32_t *expTokI, int N, int top_k, int8_t *h_q, float *h_d, int path, void *ws,
                       size_t ws_bytes, cudaStream_t stream) {
    if (!w || !x_q || !x_d || !expStart || !expTokI || !h_q || !h_d) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, w->D, w->E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, w->D, w->E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    int p = pick_path(w, N, top_k, path);
    if (p < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (p == MOE_PATH_TENSOR) {
        // expTokK is not needed for gate/up; the plan only uses it for the down scatter
        rc = launch_plan_and_gather(w, x_q, x_d, expStart, expTokI, nullptr, N, top_k, false, ws, L, stream);
        if (!rc) rc = launch_gemm_gate_up(w, N, top_k, false, ws, L, nullptr, -1, stream);
        if (!rc) rc = launch_h16_to_q8(w, N, top_k, ws, L, h_q, h_d, stream);
        return rc;
    }
    return launch_matvec_gate_up(w, w->routed, false, x_q, x_d, expStart, expTokI, N, top_k, h_q, h_d, nullptr, -1,
                                 status_word(ws), stream);
}

int moe_expert_down(moe_weights_t w, const int8_t *h_q, const float *h_d, const int32_t *expStart,
                    const int32_t *expTokI, const int32_t *expTokK, int N, int top_k, float *partials, int path,
                    void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!w || !h_q || !h_d || !expStart || !expTokI || !expTokK || !partials) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, w->D, w->E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, w->D, w->E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    int p = pick_path(w, N, top_k, path);
    if (p < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (p == MOE_PATH_TENSOR) {
        rc = launch_plan_and_gather(w, nullptr, nullptr, expStart, expTokI, expTokK, N, top_k, false, ws, L, stream);
        if (!rc) rc = launch_q8_to_h16(w, N, top_k, ws, L, h_q, h_d, stream);
        if (!rc) rc = launch_gemm_down(w, N, top_k, false, nullptr, partials, nullptr, ws, L, stream);
        return rc;
    }
    return launch_matvec_down(w, w->routed, false, h_q, h_d, expStart, expTokI, expTokK, N, top_k, nullptr, partials,
                              status_word(ws), stream);
}

int moe_debug_gate_up_block_dots(moe_weights_t w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                                 const int32_t *expTokI, int N, int top_k, int block, int32_t *dots, int path,
                                 void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!w || !x_q || !x_d || !expStart || !expTokI || !dots) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, w->D, w->E, top_k) || block < 0 || block >= w->D / QK) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, w->D, w->E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    int p = pick_path(w, N, top_k, path);
    if (p < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (p == MOE_PATH_TENSOR) {
        rc = launch_plan_and_gather(w, x_q, x_d, expStart, expTokI, nullptr, N, top_k, false, ws, L, stream);
        if (!rc) rc = launch_gemm_gate_up(w, N, top_k, false, ws, L, dots, block, stream);
        return rc;
    }
    return launch_matvec_gate_up(w, w->routed, false, x_q, x_d, expStart, expTokI, N, top_k,
                                 ws_ptr<int8_t>(ws, L.hq8), ws_ptr<float>(ws, L.hd8), dots, block, status_word(ws),
                                 stream);
}

int moe_debug_down_block_dots(moe_weights_t w, const int8_t *h_q, const float *h_d, const int32_t *expStart,
                              const int32_t *expTokI, const int32_t *expTokK, int N, int top_k, int block,
                              int32_t *dots, int path, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!w || !h_q || !h_d || !expStart || !expTokI || !expTokK || !dots) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, w->D, w->E, top_k) || block < 0 || block >= w->F / QK) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, w->D, w->E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    int p = pick_path(w, N, top_k, path);
    if (p < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    float *part = ws_ptr<float>(ws, L.partials);
    if (p == MOE_PATH_TENSOR) {
        rc = launch_plan_and_gather(w, nullptr, nullptr, expStart, expTokI, expTokK, N, top_k, false, ws, L, stream);
        if (!rc) rc = launch_q8_to_h16(w, N, top_k, ws, L, h_q, h_d, stream);
        if (!rc) rc = launch_gemm_down(w, N, top_k, false, nullptr, part, nullptr, ws, L, stream, dots, block);
        return rc;
    }
    return launch_matvec_down(w, w->routed, false, h_q, h_d, expStart, expTokI, expTokK, N, top_k, nullptr, part,
                              status_word(ws), stream, false, dots, block);
}

int moe_debug_expert_wait_timeout(moe_weights_t w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                                  const int32_t *expTokI, int N, int top_k, int limit_ms, void *ws, size_t ws_bytes,
                                  cudaStream_t stream) {
    if (!w || !x_q || !x_d || !expStart || !expTokI || limit_ms < 1 || limit_ms > 2000) return MOE_ERR_INVALID_ARG;
    if (!tensor_path_supported(w)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!shape_ok(N, w->D, w->E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, w->D, w->E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    rc = launch_plan_and_gather(w, x_q, x_d, expStart, expTokI, nullptr, N, top_k, false, ws, L, stream);
    if (!rc) rc = launch_gemm_gate_up_starved(w, N, top_k, ws, L, (unsigned long long)limit_ms * 1000000ull, stream);
    return rc;
}

int moe_combine_residual(const float *partials, const float *topk_w, const float *shared, const float *residual,
                         int N, int top_k, int D, float *out, cudaStream_t stream) {
    if (!partials || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (N < 1 || top_k < 1 || D < 4 || D % 4) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (((uintptr_t)partials | (uintptr_t)out | (uintptr_t)shared | (uintptr_t)residual) % 16)
        return MOE_ERR_INVALID_ARG;
    return launch_combine(partials, topk_w, shared, residual, N, top_k, D, out, stream);
}

// eps of the fused norm: positive and finite
static bool norm_args_ok(const float *gamma, float eps, const float *normed, const float *out, const float *residual) {
    return gamma && normed && eps > 0.0f && eps <= 3.0e38f && normed != out && normed != residual &&
           ((uintptr_t)gamma | (uintptr_t)normed) % 16 == 0;
}

int moe_combine_residual_rmsnorm(const float *partials, const float *topk_w, const float *shared,
                                 const float *residual, const float *gamma, float eps, int N, int top_k, int D,
                                 float *out, float *normed, cudaStream_t stream) {
    if (!partials || !topk_w || !out || !residual) return MOE_ERR_INVALID_ARG;
    if (!norm_args_ok(gamma, eps, normed, out, residual)) return MOE_ERR_INVALID_ARG;
    if (N < 1 || top_k < 1 || D < 4 || D % 4) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (((uintptr_t)partials | (uintptr_t)out | (uintptr_t)shared | (uintptr_t)residual) % 16)
        return MOE_ERR_INVALID_ARG;
    return launch_combine_rmsnorm(partials, topk_w, shared, residual, gamma, eps, N, top_k, D, out, normed, stream);
}

int moe_rmsnorm(const float *x, const float *gamma, float eps, int N, int D, float *normed, cudaStream_t stream) {
    if (!x || !norm_args_ok(gamma, eps, normed, nullptr, x) || (uintptr_t)x % 16) return MOE_ERR_INVALID_ARG;
    if (N < 1 || D < 4 || D % 4) return MOE_ERR_UNSUPPORTED_SHAPE;
    return launch_rmsnorm(x, gamma, eps, N, D, normed, stream);
}

int moe_combine(const float *partials, const float *topk_w, const float *shared, int N, int top_k, int D, float *out,
                cudaStream_t stream) {
    return moe_combine_residual(partials, topk_w, shared, nullptr, N, top_k, D, out, stream);
}

static int prefill_impl(moe_weights_t w, const float *hidden, const float *routerW, const float *shexp_gate, int N,
                        int top_k, int norm_topk_prob, float *out, int path, void *ws, size_t ws_bytes,
                        cudaStream_t stream, cudaEvent_t *ev, const float *residual = nullptr,
                        bool early_router = false, const float *gamma = nullptr, float eps = 0.0f,
                        float *normed = nullptr) {
    if (!w || !hidden || !routerW || !out) return MOE_ERR_INVALID_ARG;
    if (residual && ((uintptr_t)residual % 16 || w->D % 4)) return MOE_ERR_INVALID_ARG;
    if (shexp_gate && w->Fs == 0) return MOE_ERR_INVALID_ARG;
    const int D = w->D, E = w->E;
    if (!shape_ok(N, D, E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout L = ws_layout(N, D, E, w->F, top_k, w->Fs);
    int rc = check_ws(ws, ws_bytes, L);
    if (rc) return rc;
    int p = pick_path(w, N, top_k, path);
    if (p < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    auto mark = [&](int i) {
        if (ev != nullptr && rc == MOE_OK) rc = cuda_status(cudaEventRecord(ev[i], stream));
    };
    int32_t *idx = ws_ptr<int32_t>(ws, L.topk_idx);
    float *tw = ws_ptr<float>(ws, L.topk_w);
    float *sh = shexp_gate ? ws_ptr<float>(ws, L.shexp_scale) : nullptr;
    int8_t *xq = ws_ptr<int8_t>(ws, L.x_q);
    float *xd = ws_ptr<float>(ws, L.x_d);
    int32_t *es = ws_ptr<int32_t>(ws, L.expStart);
    int32_t *ti = ws_ptr<int32_t>(ws, L.expTokI);
    int32_t *tk = ws_ptr<int32_t>(ws, L.expTokK);
    float *part = ws_ptr<float>(ws, L.partials);
    float *shout = shexp_gate ? ws_ptr<float>(ws, L.shared_out) : nullptr;
    mark(0);
    // on the tensor path the bucketing kernel also writes the GEMMs' plan
    const bool tensor = (p == MOE_PATH_TENSOR);
    // decode batches on the matvec path: routing and bucketing in one launch
    int small = MOE_ERR_UNSUPPORTED_SHAPE;
    if (!tensor)
        small = launch_route_small(hidden, routerW, shexp_gate, N, D, E, top_k, norm_topk_prob ? 1 : 0, idx, tw, sh,
                                   xq, xd, ws_ptr<float>(ws, L.part_logits), es, ti, tk,
                                   reinterpret_cast<unsigned *>(static_cast<char *>(ws) + ROUTE_COUNTER_OFFSET),
                                   status_word(ws), stream, early_router && ev == nullptr);
    if (small != MOE_ERR_UNSUPPORTED_SHAPE) {
        rc = small;
        mark(1);
        mark(2);
    } else {
        // when the bucketing's token ranges are the tensor-core router's 128-token tiles, the
        // router also writes the bucketing's count table (its scratch, unused by that router)
        int range = 0;
        const int G = bucket_grid(N, E, &range);
        int *tile_counts = (range == 128 && (size_t)G * (E + 1) * 4 <= bucket_scratch_bytes(N, E))
                               ? reinterpret_cast<int *>(static_cast<char *>(ws) + BUCKET_SCRATCH_OFFSET)
                               : nullptr;
        bool counted = false;
        rc = launch_router(hidden, routerW, shexp_gate, N, D, E, top_k, norm_topk_prob ? 1 : 0, idx, tw, sh, xq,
                           xd, nullptr, ws_ptr<float>(ws, L.part_logits), L.nsplit, stream, early_router && ev == nullptr,
                           status_word(ws), tile_counts, &counted);
        mark(1);
        if (!rc)
            rc = launch_bucket(idx, N, top_k, E, es, ti, tk, ws, stream, tensor ? &L : nullptr, shout != nullptr,
                               plan_tile_rows(w), 0, 0, counted);
        mark(2);
    }
    if (tensor) {
        const bool with_shared = shout != nullptr;
        if (!rc) rc = launch_plan_and_gather(w, xq, xd, es, ti, tk, N, top_k, with_shared, ws, L, stream, true);
        mark(3);
        if (!rc) rc = launch_gemm_gate_up(w, N, top_k, with_shared, ws, L, nullptr, -1, stream);
        mark(4);
        if (!rc) rc = launch_gemm_down(w, N, top_k, with_shared, sh, part, shout, ws, L, stream);
        mark(5);
    } else {
        unsigned *st = status_word(ws);
        int8_t *hq = ws_ptr<int8_t>(ws, L.hq8);
        float *hd = ws_ptr<float>(ws, L.hd8);
        const size_t Nk = (size_t)N * top_k;
        const int Fmax = std::max(w->F, w->Fs);
        mark(3);
        if (!rc)
            rc = launch_matvec_gate_up(w, w->routed, false, xq, xd, es, ti, N, top_k, hq, hd, nullptr, -1, st, stream);
        if (!rc && shout)
            rc = launch_matvec_gate_up(w, w->shared, true, xq, xd, nullptr, nullptr, N, top_k, hq + Nk * Fmax,
                                       hd + Nk * (Fmax / QK), nullptr, -1, st, stream);
        mark(4);
        // without the stage events the down kernels and the combine start early, each behind the
        // launch before it, and wait on the device for that launch's output
        const bool early = ev == nullptr;
        if (!rc)
            rc = launch_matvec_down(w, w->routed, false, hq, hd, es, ti, tk, N, top_k, nullptr, part, st, stream,
                                    early);
        if (!rc && shout)
            rc = launch_matvec_down(w, w->shared, true, hq + Nk * Fmax, hd + Nk * (Fmax / QK), nullptr, nullptr,
                                    nullptr, N, top_k, sh, shout, st, stream, early);
        mark(5);
    }
    if (!rc)
        rc = gamma ? launch_combine_rmsnorm(part, tw, shout, residual, gamma, eps, N, top_k, D, out, normed, stream,
                                            !tensor && ev == nullptr)
                   : launch_combine(part, tw, shout, residual, N, top_k, D, out, stream, !tensor && ev == nullptr);
    mark(6);
    return rc;
}

int moe_ffn_prefill_ex(moe_weights_t w, const float *hidden, const float *routerW, const float *shexp_gate, int N,
                       int top_k, int norm_topk_prob, float *out, int path, void *ws, size_t ws_bytes,
                       cudaStream_t stream) {
    return prefill_impl(w, hidden, routerW, shexp_gate, N, top_k, norm_topk_prob, out, path, ws, ws_bytes, stream,
                        nullptr);
}

// The device address of host memory the GPU can reach (pinned: its mapped address; unregistered:
// itself, where the device walks the host page tables), or nullptr.
static const void *host_view(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    if (a.type != cudaMemoryTypeUnregistered) return nullptr;
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) != cudaSuccess)
        return nullptr;
    return pageable ? p : nullptr;
}

int moe_host_memory_addressable(const void *p) { return p != nullptr && host_view(p) != nullptr ? 1 : 0; }

int moe_device_host_numa_node(int *node) {
    if (node == nullptr) return MOE_ERR_INVALID_ARG;
    *node = -1;
    int dev = 0, v = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrHostNumaId, dev) != cudaSuccess) return MOE_ERR_CUDA;
    *node = v < 0 ? -1 : v;
    return MOE_OK;
}

int moe_ffn_prefill_host(moe_weights_t w, const float *hidden_host, const float *routerW, const float *shexp_gate,
                         int N, int top_k, int norm_topk_prob, float *out_host, int path, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    if (!hidden_host || !out_host) return MOE_ERR_INVALID_ARG;
    const float *hidden = static_cast<const float *>(host_view(hidden_host));
    float *out = static_cast<float *>(const_cast<void *>(host_view(out_host)));
    if (!hidden || !out) return MOE_ERR_INVALID_ARG;
    return prefill_impl(w, hidden, routerW, shexp_gate, N, top_k, norm_topk_prob, out, path, ws, ws_bytes, stream,
                        nullptr);
}

int moe_ffn_prefill_residual(moe_weights_t w, const float *hidden, const float *routerW, const float *shexp_gate,
                             const float *residual, int N, int top_k, int norm_topk_prob, float *out, int path,
                             void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!residual) return MOE_ERR_INVALID_ARG;
    return prefill_impl(w, hidden, routerW, shexp_gate, N, top_k, norm_topk_prob, out, path, ws, ws_bytes, stream,
                        nullptr, residual);
}

int moe_ffn_prefill_residual_rmsnorm(moe_weights_t w, const float *hidden, const float *routerW,
                                     const float *shexp_gate, const float *residual, const float *gamma, float eps,
                                     int N, int top_k, int norm_topk_prob, float *out, float *normed, int path,
                                     void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!residual || !out) return MOE_ERR_INVALID_ARG;
    if (!norm_args_ok(gamma, eps, normed, out, residual)) return MOE_ERR_INVALID_ARG;
    return prefill_impl(w, hidden, routerW, shexp_gate, N, top_k, norm_topk_prob, out, path, ws, ws_bytes, stream,
                        nullptr, residual, false, gamma, eps, normed);
}

int moe_ffn_prefill_stack_rmsnorm(const moe_weights_t *w, const float *const *routerW,
                                  const float *const *shexp_gate, const float *const *gamma, float eps, int n_layers,
                                  float *hidden, float *normed, int N, int top_k, int norm_topk_prob, int path,
                                  void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!w || !routerW || !hidden || !gamma || n_layers < 1) return MOE_ERR_INVALID_ARG;
    if (!norm_args_ok(gamma[0], eps, normed, hidden, hidden)) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        if (!w[l] || !routerW[l] || !gamma[l] || (uintptr_t)gamma[l] % 16) return MOE_ERR_INVALID_ARG;
        if (w[l]->D != w[0]->D || (reinterpret_cast<uintptr_t>(hidden) % 16) || w[0]->D % 4) return MOE_ERR_INVALID_ARG;
        const WsLayout L = ws_layout(N, w[l]->D, w[l]->E, w[l]->F, top_k, w[l]->Fs);
        if (!shape_ok(N, w[l]->D, w[l]->E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (int rc = check_ws(ws, ws_bytes, L)) return rc;
    }
    if (gamma[n_layers] && (uintptr_t)gamma[n_layers] % 16) return MOE_ERR_INVALID_ARG;
    // the first layer's input norm; afterwards every layer's combine writes both the residual stream
    // and the next layer's normalised input, and the next router is launched behind that combine
    if (int rc = launch_rmsnorm(hidden, gamma[0], eps, N, w[0]->D, normed, stream)) return rc;
    for (int l = 0; l < n_layers; ++l) {
        const float *g = shexp_gate ? shexp_gate[l] : nullptr;
        const float *gn = gamma[l + 1];  // NULL after the last layer: no final norm
        if (int rc = prefill_impl(w[l], normed, routerW[l], g, N, top_k, norm_topk_prob, hidden, path, ws, ws_bytes,
                                  stream, nullptr, hidden, true, gn, eps, gn ? normed : nullptr))
            return rc;
    }
    return MOE_OK;
}

int moe_ffn_prefill_stack(const moe_weights_t *w, const float *const *routerW, const float *const *shexp_gate,
                          int n_layers, float *hidden, int N, int top_k, int norm_topk_prob, int path, void *ws,
                          size_t ws_bytes, cudaStream_t stream) {
    if (!w || !routerW || !hidden || n_layers < 1) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        if (!w[l] || !routerW[l]) return MOE_ERR_INVALID_ARG;
        if (w[l]->D != w[0]->D || (reinterpret_cast<uintptr_t>(hidden) % 16) || w[0]->D % 4) return MOE_ERR_INVALID_ARG;
        const WsLayout L = ws_layout(N, w[l]->D, w[l]->E, w[l]->F, top_k, w[l]->Fs);
        if (!shape_ok(N, w[l]->D, w[l]->E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (int rc = check_ws(ws, ws_bytes, L)) return rc;
    }
    for (int l = 0; l < n_layers; ++l) {
        // hidden <- hidden + FFN_l(hidden), in place; from the second layer on the router is
        // launched behind the previous layer's combine (it waits on the device for its output)
        const float *g = shexp_gate ? shexp_gate[l] : nullptr;
        if (int rc = prefill_impl(w[l], hidden, routerW[l], g, N, top_k, norm_topk_prob, hidden, path, ws, ws_bytes,
                                  stream, nullptr, hidden, l > 0))
            return rc;
    }
    return MOE_OK;
}

int moe_ffn_prefill_timed(moe_weights_t w, const float *hidden, const float *routerW, const float *shexp_gate, int N,
                          int top_k, int norm_topk_prob, float *out, int path, void *ws, size_t ws_bytes,
                          cudaStream_t stream, cudaEvent_t *stage_events) {
    if (!stage_events) return MOE_ERR_INVALID_ARG;
    return prefill_impl(w, hidden, routerW, shexp_gate, N, top_k, norm_topk_prob, out, path, ws, ws_bytes, stream,
                        stage_events);
}

int moe_ffn_prefill(moe_weights_t w, const float *hidden, const float *routerW, const float *shexp_gate, int N,
                    int top_k, int norm_topk_prob, float *out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return moe_ffn_prefill_ex(w, hidden, routerW, shexp_gate, N, top_k, norm_topk_prob, out, MOE_PATH_AUTO, ws,
                              ws_bytes, stream);
}

int moe_workspace_views(void *ws, int N, int D, int E, int F, int top_k, int Fs, int32_t **topk_idx, float **topk_w,
                        float **shexp_scale, int8_t **x_q, float **x_d, int32_t **expStart, int32_t **expTokI,
                        int32_t **expTokK, float **partials, float **shared_out) {
    if (!ws || !shape_ok(N, D, E, top_k)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(N, D, E, F, top_k, Fs);
    if (topk_idx) *topk_idx = ws_ptr<int32_t>(ws, L.topk_idx);
    if (topk_w) *topk_w = ws_ptr<float>(ws, L.topk_w);
    if (shexp_scale) *shexp_scale = ws_ptr<float>(ws, L.shexp_scale);
    if (x_q) *x_q = ws_ptr<int8_t>(ws, L.x_q);
    if (x_d) *x_d = ws_ptr<float>(ws, L.x_d);
    if (expStart) *expStart = ws_ptr<int32_t>(ws, L.expStart);
    if (expTokI) *expTokI = ws_ptr<int32_t>(ws, L.expTokI);
    if (expTokK) *expTokK = ws_ptr<int32_t>(ws, L.expTokK);
    if (partials) *partials = ws_ptr<float>(ws, L.partials);
    if (shared_out) *shared_out = Fs ? ws_ptr<float>(ws, L.shared_out) : nullptr;
    return MOE_OK;
}

}  // extern "C"
