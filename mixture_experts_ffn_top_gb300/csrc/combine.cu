// combine.cu -- batched weighted scatter-reduce (issue #129, "Scope"): for each
// token row, sum the top_k unweighted down-partials in slot order k = 0..na-1
// with the per-(token, slot) weights, then add the shared-expert row, in one
// launch over N x D.  The per-element order and rounding are fixed (one fused
// multiply-add per slot, then one add), so the result is bit-reproducible:
//   acc = +0; for s: acc = fma(w[t,s], partial[t*k+s], acc); acc += shared.
// With a residual row (the pages' per-layer combine is (routed + shared) + resid,
// "Carnice prefill toward llama.cpp 676 t/s", #388, "Dead ends") one more add: acc += resid.
// HBM-bound: each thread owns 4 consecutive columns (16-byte loads/stores); for the
// usual top_k the slot loads are all issued before the fma chain; partial rows are
// streamed once (evict-first loads), the output is written once.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

// KMAX > 0: top_k known at compile time (all slot loads issued before the fma chain);
// KMAX == 0: any top_k.
template <int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(const float4 *__restrict__ partials, const float *__restrict__ w,
               const float4 *__restrict__ shared, const float4 *residual, int N, int k, int D4, float4 *out) {
    // the next layer's router may be scheduled now (it waits for this grid before reading out)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // launched early behind the down kernel: its partials are complete past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t total = (int64_t)N * D4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / D4;
        const int64_t c = i - t * D4;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (KMAX > 0) {
            float4 p[KMAX > 0 ? KMAX : 1];
            float ws[KMAX > 0 ? KMAX : 1];
#pragma unroll
            for (int s = 0; s < KMAX; ++s) {
                p[s] = __ldcs(partials + (t * KMAX + s) * D4 + c);
                ws[s] = w[t * KMAX + s];
            }
#pragma unroll
            for (int s = 0; s < KMAX; ++s) {
                acc.x = __fmaf_rn(ws[s], p[s].x, acc.x);
                acc.y = __fmaf_rn(ws[s], p[s].y, acc.y);
                acc.z = __fmaf_rn(ws[s], p[s].z, acc.z);
                acc.w = __fmaf_rn(ws[s], p[s].w, acc.w);
            }
        } else {
            for (int s = 0; s < k; ++s) {
                const float ws = w[t * k + s];
                const float4 p = __ldcs(partials + (t * k + s) * D4 + c);
                acc.x = __fmaf_rn(ws, p.x, acc.x);
                acc.y = __fmaf_rn(ws, p.y, acc.y);
                acc.z = __fmaf_rn(ws, p.z, acc.z);
                acc.w = __fmaf_rn(ws, p.w, acc.w);
            }
        }
        if (shared != nullptr) {
            const float4 sv = __ldcs(shared + t * D4 + c);
            acc.x = __fadd_rn(acc.x, sv.x);
            acc.y = __fadd_rn(acc.y, sv.y);
            acc.z = __fadd_rn(acc.z, sv.z);
            acc.w = __fadd_rn(acc.w, sv.w);
        }
        if (residual != nullptr) {  // may be `out` itself: read before the write of the same element
            const float4 rv = residual[i];
            acc.x = __fadd_rn(acc.x, rv.x);
            acc.y = __fadd_rn(acc.y, rv.y);
            acc.z = __fadd_rn(acc.z, rv.z);
            acc.w = __fadd_rn(acc.w, rv.w);
        }
        out[i] = acc;
    }
}

}  // namespace

int launch_combine(const float *partials, const float *topk_w, const float *shared, const float *residual, int N,
                   int top_k, int D, float *out, cudaStream_t s, bool early) {
    const int D4 = D / 4;
    const int64_t total = (int64_t)N * D4;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)std::max(1, device_sm_count()) * 8;  // 8 resident CTAs of 256 threads per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const float4 *p4 = reinterpret_cast<const float4 *>(partials);
    const float4 *s4 = reinterpret_cast<const float4 *>(shared);
    const float4 *r4 = reinterpret_cast<const float4 *>(residual);
    float4 *o4 = reinterpret_cast<float4 *>(out);
    const unsigned g = (unsigned)blocks;
    auto go = [&](auto kernel) {
        if (early) return launch_early(kernel, dim3(g), dim3(256), 0, s, p4, topk_w, s4, r4, N, top_k, D4, o4);
        kernel<<<g, 256, 0, s>>>(p4, topk_w, s4, r4, N, top_k, D4, o4);
        return launch_status();
    };
    switch (top_k) {
        case 1: return go(combine_kernel<1>);
        case 2: return go(combine_kernel<2>);
        case 4: return go(combine_kernel<4>);
        case 6: return go(combine_kernel<6>);
        case 8: return go(combine_kernel<8>);
        default: return go(combine_kernel<0>);
    }
}

}  // namespace moe
