// router_noalloc.cu -- moe_router_topk for callers that cannot allocate device memory.
//
// Some hosts own all device memory themselves (a serving process whose pool
// allocator claimed the GPU at start-up, a plugin that may only use what its
// framework hands it, a runtime that forbids cudaMalloc after initialisation
// because it synchronises the device and can fail under fragmentation).  Such a
// caller cannot provide moe_router_topk's workspace.  This entry point runs the
// same router kernels with their split-K partial logits in a fixed array that
// lives in the library's own device image instead.
//
// The array is g_router_noalloc_scratch below: 2^22 floats (16 MiB), present on
// every GPU that loads the library until the process exits.  Every call on a
// device shares it, so calls that overlap on the GPU (two streams, two host
// threads) race on it: the caller must order them.  The kernels overwrite every
// element they later read, so nothing in it has to start at zero.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(1) << 22;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_router_noalloc_scratch[kNoAllocScratchFloats];

std::mutex g_mu;
float *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, resolved once per
// device.  The host-side name of a __device__ array is not a device address,
// hence the lookup; the first lookup on a device may load the library's module
// onto it.
int scratch_for_current_device(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_router_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

}  // namespace moe

extern "C" int moe_router_topk_noalloc(const float *hidden, const float *routerW, const float *shexp_gate, int N,
                                       int D, int E, int top_k, int norm_topk_prob, int32_t *topk_idx,
                                       float *topk_w, float *shexp_scale, int8_t *x_q, float *x_d,
                                       float *logits_out, cudaStream_t stream) {
    using namespace moe;
    if (!hidden || !routerW || !topk_idx || !topk_w || !x_q || !x_d) return MOE_ERR_INVALID_ARG;
    if ((shexp_gate == nullptr) != (shexp_scale == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(N, D, E, top_k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    // the split the router's launch uses decides how much of the array it writes
    if ((size_t)router_split_used(N, D, E) * (size_t)N * (size_t)(E + 1) > kNoAllocScratchFloats)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    const int nsplit = router_nsplit(N, D, E);
    float *scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    return launch_router(hidden, routerW, shexp_gate, N, D, E, top_k, norm_topk_prob ? 1 : 0, topk_idx, topk_w,
                         shexp_scale, x_q, x_d, logits_out, scratch, nsplit, stream);
}
