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
// A second kernel also normalises each output row for the next layer (RMSNorm with a
// per-column weight and epsilon: the pages' router reads a normalised activation,
// #388 "Remaining levers" items 1 and 2), one CTA per row.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

// The combined value of the 4 columns c*4 .. c*4+3 of token row t (element index i = t*D4 + c):
// the slot-order fused multiply-adds, then the shared row, then the residual (which may be the
// output buffer: the caller reads it here, before its write of the same element).
// KMAX > 0: top_k known at compile time (all slot loads issued before the fma chain);
// KMAX == 0: any top_k.
template <int KMAX>
__device__ __forceinline__ float4 combine4(const float4 *__restrict__ partials, const float *__restrict__ w,
                                           const float4 *__restrict__ shared, const float4 *residual, int64_t t,
                                           int64_t c, int k, int D4) {
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
    if (residual != nullptr) {
        const float4 rv = residual[t * D4 + c];
        acc.x = __fadd_rn(acc.x, rv.x);
        acc.y = __fadd_rn(acc.y, rv.y);
        acc.z = __fadd_rn(acc.z, rv.z);
        acc.w = __fadd_rn(acc.w, rv.w);
    }
    return acc;
}

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
        out[i] = combine4<KMAX>(partials, w, shared, residual, t, i - t * D4, k, D4);
    }
}

// The combine with residual, then the next layer's input norm read as RMSNorm: one CTA per token
// row at a time (the grid strides over rows).  With k = 0 and no out it is the norm of the
// residual rows alone (the first layer's input norm of a stack).  Each element is combine4's value (out, bit for bit
// the plain combine's); the row's sum of squares is accumulated in fp32 per thread (its columns in
// order), then over the warp (butterfly) and the warps (in order), and
//   normed = (out * r) * gamma,  r = 1 / sqrt(sum / D + eps)  (IEEE divide and square root).
// CN_THREADS threads per row: 128 when the batch fills the SMs with rows, 512 for small batches
// (decode), where rows are few and each must be spread over more threads.
template <int KMAX, int CN_THREADS>
__global__ void __launch_bounds__(CN_THREADS)
combine_rmsnorm_kernel(const float4 *__restrict__ partials, const float *__restrict__ w,
                       const float4 *__restrict__ shared, const float4 *residual, const float4 *__restrict__ gamma,
                       float eps, int N, int k, int D4, float4 *out, float4 *__restrict__ normed) {
    __shared__ float wsum[CN_THREADS / 32];
    __shared__ float r_row;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t = blockIdx.x; t < N; t += gridDim.x) {
        float ss = 0.0f;
        for (int c = threadIdx.x; c < D4; c += CN_THREADS) {
            const float4 v = combine4<KMAX>(partials, w, shared, residual, t, c, k, D4);
            if (out != nullptr) out[t * D4 + c] = v;
            ss = __fmaf_rn(v.x, v.x, ss);
            ss = __fmaf_rn(v.y, v.y, ss);
            ss = __fmaf_rn(v.z, v.z, ss);
            ss = __fmaf_rn(v.w, v.w, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) wsum[warp] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = wsum[0];
#pragma unroll
            for (int i = 1; i < CN_THREADS / 32; ++i) tot = __fadd_rn(tot, wsum[i]);
            r_row = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)(4 * D4)), eps)));
        }
        __syncthreads();
        const float r = r_row;
        for (int c = threadIdx.x; c < D4; c += CN_THREADS) {
            // this thread's own store above, or (no out: the norm of the residual rows alone) the
            // value again
            const float4 o = out != nullptr ? out[t * D4 + c] : combine4<KMAX>(partials, w, shared, residual, t, c, k, D4);
            const float4 g = gamma[c];
            normed[t * D4 + c] = make_float4(__fmul_rn(__fmul_rn(o.x, r), g.x), __fmul_rn(__fmul_rn(o.y, r), g.y),
                                             __fmul_rn(__fmul_rn(o.z, r), g.z), __fmul_rn(__fmul_rn(o.w, r), g.w));
        }
        __syncthreads();  // wsum and r_row are the next row's
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

int launch_combine_rmsnorm(const float *partials, const float *topk_w, const float *shared, const float *residual,
                           const float *gamma, float eps, int N, int top_k, int D, float *out, float *normed,
                           cudaStream_t s, bool early) {
    const int D4 = D / 4;
    // rows in flight: 16 CTAs of 128 threads per SM, or, for batches too small to fill the SMs that
    // way (fewer than 8 rows per SM), 4 CTAs of 512 threads per SM
    const int sms = std::max(1, device_sm_count());
    const bool wide = N < 8 * sms;
    const int64_t cap = (int64_t)sms * (wide ? 4 : 16);
    const unsigned g = (unsigned)std::max<int64_t>(1, std::min<int64_t>(N, cap));
    const int nt = wide ? 512 : 128;
    const float4 *p4 = reinterpret_cast<const float4 *>(partials);
    const float4 *s4 = reinterpret_cast<const float4 *>(shared);
    const float4 *r4 = reinterpret_cast<const float4 *>(residual);
    const float4 *g4 = reinterpret_cast<const float4 *>(gamma);
    float4 *o4 = reinterpret_cast<float4 *>(out);
    float4 *n4 = reinterpret_cast<float4 *>(normed);
    auto go1 = [&](auto kernel) {
        if (early)
            return launch_early(kernel, dim3(g), dim3(nt), 0, s, p4, topk_w, s4, r4, g4, eps, N, top_k, D4, o4, n4);
        kernel<<<g, nt, 0, s>>>(p4, topk_w, s4, r4, g4, eps, N, top_k, D4, o4, n4);
        return launch_status();
    };
    auto go = [&](auto narrow, auto widek) { return wide ? go1(widek) : go1(narrow); };
    switch (top_k) {
        case 1: return go(combine_rmsnorm_kernel<1, 128>, combine_rmsnorm_kernel<1, 512>);
        case 2: return go(combine_rmsnorm_kernel<2, 128>, combine_rmsnorm_kernel<2, 512>);
        case 4: return go(combine_rmsnorm_kernel<4, 128>, combine_rmsnorm_kernel<4, 512>);
        case 6: return go(combine_rmsnorm_kernel<6, 128>, combine_rmsnorm_kernel<6, 512>);
        case 8: return go(combine_rmsnorm_kernel<8, 128>, combine_rmsnorm_kernel<8, 512>);
        default: return go(combine_rmsnorm_kernel<0, 128>, combine_rmsnorm_kernel<0, 512>);
    }
}

int launch_rmsnorm(const float *x, const float *gamma, float eps, int N, int D, float *normed, cudaStream_t s) {
    return launch_combine_rmsnorm(nullptr, nullptr, nullptr, x, gamma, eps, N, 0, D, nullptr, normed, s, false);
}

}  // namespace moe
