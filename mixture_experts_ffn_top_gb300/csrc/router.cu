// router.cu -- router logits, softmax + top-k, shared-expert gate and the Q8_1
// quantisation of the hidden rows ("Carnice prefill toward llama.cpp 676 t/s",
// #388: breakdown table "router" row -- matvec + softmax + top-k + shexp-gate,
// per token -- and "Remaining levers" item 1, which moves it onto the GPU).
//
// Two kernels (router_small_kernel replaces the first for batches of at most 8 tokens):
//   router_logits_kernel: split-K fp32 SIMT GEMM  logits = hidden . routerW^T
//     (routerW extended by the shared gate vector as row E).  The CTAs of
//     expert tile 0 also quantise the hidden rows they stage (each 32-wide K
//     chunk is exactly one Q8_1 block), so hidden is read from HBM once.
//   softmax_topk_kernel: one warp per token; sums the split-K partials in a
//     fixed order, softmax over all E, top-k by repeated warp argmax (ties to
//     the lower expert index), weights, sigmoid gate.
#include "moe_internal.cuh"
#include "topk_token.cuh"

namespace moe {

namespace {

constexpr int RB_M = 64;   // tokens per tile
constexpr int RB_N = 64;   // experts per tile
constexpr int RB_K = 32;   // K chunk = one Q8 block
constexpr int R_THREADS = 256;

// logits partials for one (token tile, expert tile, K split): 4x4 outputs per
// thread from a double-buffered shared tile; the next K chunk is fetched into
// registers while the current one is multiplied.
__global__ void __launch_bounds__(R_THREADS)
router_logits_kernel(const float *__restrict__ hidden, const float *__restrict__ routerW,
                     const float *__restrict__ shexp_gate, int N, int D, int E, int Eext, int ksplit,
                     float *__restrict__ part, int8_t *__restrict__ x_q, float *__restrict__ x_d) {
    __shared__ __align__(16) float Xs[2][RB_K][RB_M + 4];
    __shared__ __align__(16) float Ws[2][RB_K][RB_N + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * RB_M;
    const int e0 = blockIdx.y * RB_N;
    const int split = blockIdx.z;
    const int k_begin = split * ksplit;
    const int k_end = min(D, k_begin + ksplit);
    const bool quantise = (blockIdx.y == 0);
    const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads, 4x4 outputs each
    // Launched early behind the previous layer's combine (a chain of layers): this CTA's slice of
    // routerW does not depend on it, so ask L2 for it first; hidden is the previous layer's output,
    // read only after the wait (which returns at once without the launch attribute).
    for (int i = tid; i < RB_N * ((k_end - k_begin + 31) / 32); i += R_THREADS) {
        const int e = e0 + i / ((k_end - k_begin + 31) / 32), c = k_begin + 32 * (i % ((k_end - k_begin + 31) / 32));
        const float *src = e < E ? routerW + (size_t)e * D + c : (e == E && shexp_gate ? shexp_gate + c : nullptr);
        if (src != nullptr && c < k_end) asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    // per chunk: 2 float4 of hidden (64 rows x 8 float4) and 2 float4 of W (64 rows x 8 float4)
    float4 xr[2], wr[2];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = tid + r * R_THREADS, row = i >> 3, c4 = (i & 7) * 4;
            const int t = t0 + row;
            xr[r] = t < N ? *reinterpret_cast<const float4 *>(hidden + (size_t)t * D + k0 + c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = tid + r * R_THREADS, row = i >> 3, c4 = (i & 7) * 4;
            const int e = e0 + row;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < E) v = *reinterpret_cast<const float4 *>(routerW + (size_t)e * D + k0 + c4);
            else if (e == E && shexp_gate != nullptr) v = *reinterpret_cast<const float4 *>(shexp_gate + k0 + c4);
            wr[r] = v;
        }
    };
    auto stash = [&](int b) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = tid + r * R_THREADS, row = i >> 3, c4 = (i & 7) * 4;
            Xs[b][c4 + 0][row] = xr[r].x;
            Xs[b][c4 + 1][row] = xr[r].y;
            Xs[b][c4 + 2][row] = xr[r].z;
            Xs[b][c4 + 3][row] = xr[r].w;
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = tid + r * R_THREADS, row = i >> 3, c4 = (i & 7) * 4;
            Ws[b][c4 + 0][row] = wr[r].x;
            Ws[b][c4 + 1][row] = wr[r].y;
            Ws[b][c4 + 2][row] = wr[r].z;
            Ws[b][c4 + 3][row] = wr[r].w;
        }
    };
    int b = 0;
    if (k_begin < k_end) {
        fetch(k_begin);
        stash(0);
    }
    __syncthreads();
    for (int k0 = k_begin; k0 < k_end; k0 += RB_K, b ^= 1) {
        const bool more = k0 + RB_K < k_end;
        if (more) fetch(k0 + RB_K);  // in flight during this chunk's math
        if (quantise) {
            // Q8_1 of this K chunk (one block) for the tile's tokens: warp w takes 8 tokens, one
            // warp reduction per token for the block maximum; the two IEEE divisions of the rule
            // (d = amax/127, then 1/d) run once for the 8 tokens side by side in lanes 0-7
            const int warp = tid >> 5, lane = tid & 31;
            constexpr int RPW = RB_M / 8;  // rows per warp
            float xv[RPW];
            unsigned amax_mine = 0;
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                xv[rr] = Xs[b][lane][warp * RPW + rr];
                const unsigned am = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(xv[rr])));
                if (lane == rr) amax_mine = am;
            }
            const float d = __fdiv_rn(__uint_as_float(amax_mine), 127.0f);
            const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
            if (lane < RPW && t0 + warp * RPW + lane < N)
                x_d[(size_t)(t0 + warp * RPW + lane) * (D / QK) + k0 / QK] = __half2float(__float2half_rn(d));
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                const int t = t0 + warp * RPW + rr;
                const float idr = __shfl_sync(0xffffffffu, id, rr);
                if (t < N) x_q[(size_t)t * D + k0 + lane] = (int8_t)(int)roundf(__fmul_rn(xv[rr], idr));
            }
        }
#pragma unroll 8
        for (int kk = 0; kk < RB_K; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&Xs[b][kk][ty * 4]);
            const float4 w = *reinterpret_cast<const float4 *>(&Ws[b][kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
        }
        if (more) stash(b ^ 1);  // the other buffer was last read two chunks ago
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= N) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < Eext) part[((size_t)split * N + t) * Eext + e] = acc[i][j];
        }
    }
}

// Small batches (N <= RS_MAX_N, decode): one CTA per expert row of routerW (row E: the
// shared gate), its 8 warps splitting K, every thread holding the partial dots of all N tokens;
// warp sums by a fixed butterfly, then the 8 warp sums in warp order, so the logits are
// deterministic and need no split-K partials.  The N hidden rows' Q8_1 blocks are spread over
// all warps of the grid.  Output: logits [N][Eext], read by softmax_topk_kernel as one split.
constexpr int RS_THREADS = 256;
constexpr int RS_MAX_N = 8;
__device__ __forceinline__ void router_small_body(const float *__restrict__ hidden, const float *__restrict__ routerW,
                                                  const float *__restrict__ shexp_gate, int N, int D, int E, int Eext,
                                                  float *__restrict__ logits, int8_t *__restrict__ x_q,
                                                  float *__restrict__ x_d) {
    __shared__ float red[RS_THREADS / 32][RS_MAX_N];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e = blockIdx.x;
    const float *w = e < E ? routerW + (size_t)e * D : shexp_gate;
    // launched early behind the previous layer's combine: the weight row first, hidden after the wait
    for (int c = 32 * tid; c < D; c += 32 * RS_THREADS) asm volatile("prefetch.global.L2 [%0];" ::"l"(w + c));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float acc[RS_MAX_N];
#pragma unroll
    for (int t = 0; t < RS_MAX_N; ++t) acc[t] = 0.0f;
#pragma unroll 2
    for (int c = 4 * tid; c < D; c += 4 * RS_THREADS) {
        const float4 wv = *reinterpret_cast<const float4 *>(w + c);
#pragma unroll
        for (int t = 0; t < RS_MAX_N; ++t)
            if (t < N) {
                const float4 xv = *reinterpret_cast<const float4 *>(hidden + (size_t)t * D + c);
                acc[t] = fmaf(xv.x, wv.x, acc[t]);
                acc[t] = fmaf(xv.y, wv.y, acc[t]);
                acc[t] = fmaf(xv.z, wv.z, acc[t]);
                acc[t] = fmaf(xv.w, wv.w, acc[t]);
            }
    }
#pragma unroll
    for (int t = 0; t < RS_MAX_N; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) red[warp][t] = v;
    }
    __syncthreads();
    if (tid < N) {
        float v = red[0][tid];
        for (int w2 = 1; w2 < RS_THREADS / 32; ++w2) v = __fadd_rn(v, red[w2][tid]);
        logits[(size_t)tid * Eext + e] = v;
    }
    // Q8_1 of the hidden rows: global warp g takes blocks g, g + (all warps), ...
    const int nblk = N * (D / QK);
    for (int b = blockIdx.x * (RS_THREADS / 32) + warp; b < nblk; b += gridDim.x * (RS_THREADS / 32)) {
        float d16f;
        const int q = q8_quantize_lane(hidden[(size_t)b * QK + lane], &d16f);
        x_q[(size_t)b * QK + lane] = (int8_t)q;
        if (lane == 0) x_d[b] = d16f;
    }
}

__global__ void __launch_bounds__(RS_THREADS)
router_small_kernel(const float *__restrict__ hidden, const float *__restrict__ routerW,
                    const float *__restrict__ shexp_gate, int N, int D, int E, int Eext, float *__restrict__ logits,
                    int8_t *__restrict__ x_q, float *__restrict__ x_d) {
    router_small_body(hidden, routerW, shexp_gate, N, D, E, Eext, logits, x_q, x_d);
}

// One warp per token: the split-K partials summed in split order (loads issued four at a time),
// then route_token.  EPL = experts per lane (power of two, EPL*32 >= E).
template <int EPL>
__device__ __forceinline__ void softmax_topk_token(const float *__restrict__ part, int nsplit, int N, int E, int Eext,
                                                   int top_k, int norm, int t, int lane, int32_t *__restrict__ topk_idx,
                                                   float *__restrict__ topk_w, float *__restrict__ shexp_scale,
                                                   float *__restrict__ logits_out) {
    const size_t stride = (size_t)N * Eext;
    auto logit = [&](int e) {
        const float *pp = part + (size_t)t * Eext + e;
        float v = __ldcg(pp);
        int s = 1;
        for (; s + 4 <= nsplit; s += 4) {
            const float a0 = __ldcg(pp + s * stride), a1 = __ldcg(pp + (s + 1) * stride),
                        a2 = __ldcg(pp + (s + 2) * stride), a3 = __ldcg(pp + (s + 3) * stride);
            v = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(v, a0), a1), a2), a3);
        }
        for (; s < nsplit; ++s) v = __fadd_rn(v, __ldcg(pp + s * stride));
        return v;
    };
    auto gate = [&]() {
        float g = __ldcg(part + (size_t)t * Eext + E);
        for (int s = 1; s < nsplit; ++s) g = __fadd_rn(g, __ldcg(part + ((size_t)s * N + t) * Eext + E));
        return g;
    };
    route_token<EPL>(logit, gate, E, top_k, norm, t, lane, topk_idx, topk_w, shexp_scale, logits_out);
}

// One warp per token.
template <int EPL>
__global__ void __launch_bounds__(256)
softmax_topk_kernel(const float *__restrict__ part, int nsplit, int N, int E, int Eext, int top_k,
                    int norm, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                    float *__restrict__ shexp_scale, float *__restrict__ logits_out) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= N) return;
    softmax_topk_token<EPL>(part, nsplit, N, E, Eext, top_k, norm, t, lane, topk_idx, topk_w, shexp_scale,
                            logits_out);
}

// Counting sort of a small batch's N*top_k (<= RS_THREADS) routing entries by expert, stable in
// t, into expStart/expTokI/expTokK -- the CSR the general bucketing kernel writes.  Whole CTA;
// idx was written by this CTA (visible after the caller's __syncthreads).  An index outside
// [0, E) raises MOE_DEV_BAD_ROUTING and leaves every segment empty.
__device__ __forceinline__ void bucket_small(const int32_t *idx, int N, int k, int E, int32_t *expStart,
                                             int32_t *expTokI, int32_t *expTokK, unsigned *status) {
    __shared__ int ids[RS_THREADS];
    __shared__ int st[MAX_E + 1];
    __shared__ int wsum[RS_THREADS / 32];
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = N * k;
    if (tid == 0) bad = 0;
    __syncthreads();
    if (tid < total) {
        const int e = idx[tid];
        ids[tid] = e;
        if (e < 0 || e >= E) bad = 1;
    }
    __syncthreads();
    if (bad) {
        for (int e = tid; e <= E; e += RS_THREADS) expStart[e] = 0;
        if (tid == 0) atomicOr(status, MOE_DEV_BAD_ROUTING);
        return;
    }
    // per-expert counts over a contiguous range of experts per thread, then a block scan
    const int per = (E + RS_THREADS - 1) / RS_THREADS;
    const int e0 = tid * per;
    int cnt[(MAX_E + RS_THREADS - 1) / RS_THREADS];
    int mine = 0;
#pragma unroll
    for (int i = 0; i < (MAX_E + RS_THREADS - 1) / RS_THREADS; ++i) {
        cnt[i] = 0;
        const int e = e0 + i;
        if (i < per && e < E)
            for (int j = 0; j < total; ++j) cnt[i] += ids[j] == e;
        mine += cnt[i];
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = incl - mine;
    for (int w = 0; w < warp; ++w) before += wsum[w];
#pragma unroll
    for (int i = 0; i < (MAX_E + RS_THREADS - 1) / RS_THREADS; ++i) {
        const int e = e0 + i;
        if (i < per && e < E) {
            st[e] = before;
            expStart[e] = before;
            before += cnt[i];
        }
    }
    if (tid == 0) expStart[E] = total;
    __syncthreads();
    // entry j = (t, s): its rank among the earlier entries of the same expert (earlier tokens:
    // a token picks an expert once)
    if (tid < total) {
        const int e = ids[tid];
        int rank = 0;
        for (int j = 0; j < tid; ++j) rank += ids[j] == e;
        const int pos = st[e] + rank;
        expTokI[pos] = tid / k;
        expTokK[pos] = tid % k;
    }
}

// The whole routing of a small batch in one launch: every CTA computes one expert row's logits
// (router_small_body); the last CTA to arrive (an arrival counter in the workspace, reset by that
// CTA) runs softmax + top-k for the N tokens (warp t: token t) and the bucketing.  No CTA waits
// for another.
template <int EPL>
__global__ void __launch_bounds__(RS_THREADS)
route_small_kernel(const float *__restrict__ hidden, const float *__restrict__ routerW,
                   const float *__restrict__ shexp_gate, int N, int D, int E, int Eext, int top_k, int norm,
                   float *__restrict__ logits, int8_t *__restrict__ x_q, float *__restrict__ x_d,
                   int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, float *__restrict__ shexp_scale,
                   int32_t *__restrict__ expStart, int32_t *__restrict__ expTokI, int32_t *__restrict__ expTokK,
                   unsigned *counter, unsigned *status) {
    __shared__ int is_last;
    router_small_body(hidden, routerW, shexp_gate, N, D, E, Eext, logits, x_q, x_d);
    __threadfence();  // this CTA's logits are visible before it is counted
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(counter, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (threadIdx.x == 0) *counter = 0;  // every CTA has arrived: ready for the next launch
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < N)
        softmax_topk_token<EPL>(logits, 1, N, E, Eext, top_k, norm, warp, lane, topk_idx, topk_w, shexp_scale,
                                nullptr);
    __syncthreads();
    bucket_small(topk_idx, N, top_k, E, expStart, expTokI, expTokK, status);
}

__global__ void quantize_q8_1_kernel(const float *__restrict__ x, int64_t nblk, int8_t *__restrict__ q,
                                     float *__restrict__ d) {
    const int lane = threadIdx.x & 31;
    int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= nblk) return;
    float d16f;
    int qi = q8_quantize_lane(x[b * QK + lane], &d16f);
    q[b * QK + lane] = (int8_t)qi;
    if (lane == 0) d[b] = d16f;
}

int launch_softmax(const float *part, int nsplit, int N, int E, int Eext, int top_k, int norm,
                   int32_t *idx, float *w, float *sh, float *logits_out, cudaStream_t s) {
    dim3 grid((N + 7) / 8), block(256);
    int epl = (E + 31) / 32;
    if (epl <= 1)
        softmax_topk_kernel<1><<<grid, block, 0, s>>>(part, nsplit, N, E, Eext, top_k, norm, idx, w, sh, logits_out);
    else if (epl <= 2)
        softmax_topk_kernel<2><<<grid, block, 0, s>>>(part, nsplit, N, E, Eext, top_k, norm, idx, w, sh, logits_out);
    else if (epl <= 4)
        softmax_topk_kernel<4><<<grid, block, 0, s>>>(part, nsplit, N, E, Eext, top_k, norm, idx, w, sh, logits_out);
    else if (epl <= 8)
        softmax_topk_kernel<8><<<grid, block, 0, s>>>(part, nsplit, N, E, Eext, top_k, norm, idx, w, sh, logits_out);
    else if (epl <= 16)
        softmax_topk_kernel<16><<<grid, block, 0, s>>>(part, nsplit, N, E, Eext, top_k, norm, idx, w, sh, logits_out);
    else
        softmax_topk_kernel<32><<<grid, block, 0, s>>>(part, nsplit, N, E, Eext, top_k, norm, idx, w, sh, logits_out);
    return launch_status();
}

}  // namespace

int router_nsplit(int N, int D, int E) {
    // about four 8-warp CTAs per SM; each split at least 128 deep, or one K chunk (32) when
    // the tiles are few (decode batches: one chunk per CTA, all of routerW read in one round).
    // The split sets the size of the workspace's partial-logit table, so a size query must run
    // with the same device current as the calls (without a device it assumes one SM).
    int tiles = ((N + RB_M - 1) / RB_M) * ((E + RB_N - 1) / RB_N);
    const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
    int want = (4 * sms + tiles - 1) / tiles;
    int depth = tiles <= 4 ? RB_K : 128;
    int maxs = D / depth > 0 ? D / depth : 1;
    int s = want < 1 ? 1 : (want > maxs ? maxs : want);
    while (s > 1 && (D / QK) % s != 0) --s;  // equal splits on block boundaries
    return s;
}

int router_split_used(int N, int D, int E) { return (N <= RS_MAX_N && D % 4 == 0) ? 1 : router_nsplit(N, D, E); }

int launch_router(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D,
                  int E, int top_k, int norm, int32_t *topk_idx, float *topk_w, float *shexp_scale,
                  int8_t *x_q, float *x_d, float *logits_out, float *part_logits, int nsplit,
                  cudaStream_t s, bool early, unsigned *status, int *tile_counts, bool *counted) {
    int Eext = E + (shexp_gate ? 1 : 0);
    if (counted) *counted = false;
    if (status != nullptr && router_tc_eligible(N, D, E, shexp_gate != nullptr, hidden, routerW, shexp_gate)) {
        const int rc = launch_router_tc(hidden, routerW, shexp_gate, N, D, E, top_k, norm, topk_idx, topk_w,
                                        shexp_scale, x_q, x_d, logits_out, status, s, early, tile_counts);
        if (rc == MOE_OK && counted) *counted = tile_counts != nullptr;
        if (rc != MOE_ERR_UNSUPPORTED_SHAPE) return rc;  // else: no room for the cluster, the SIMT router
    }
    if (N <= RS_MAX_N && D % 4 == 0) {
        int rc = MOE_OK;
        if (early)
            rc = launch_early(router_small_kernel, dim3(Eext), dim3(RS_THREADS), 0, s, hidden, routerW, shexp_gate, N, D,
                              E, Eext, part_logits, x_q, x_d);
        else {
            router_small_kernel<<<Eext, RS_THREADS, 0, s>>>(hidden, routerW, shexp_gate, N, D, E, Eext, part_logits,
                                                            x_q, x_d);
            rc = launch_status();
        }
        if (rc) return rc;
        return launch_softmax(part_logits, 1, N, E, Eext, top_k, norm, topk_idx, topk_w,
                              shexp_gate ? shexp_scale : nullptr, logits_out, s);
    }
    int ksplit = D / nsplit;
    dim3 grid((N + RB_M - 1) / RB_M, (Eext + RB_N - 1) / RB_N, nsplit);
    int rc = MOE_OK;
    if (early)
        rc = launch_early(router_logits_kernel, grid, dim3(R_THREADS), 0, s, hidden, routerW, shexp_gate, N, D, E, Eext,
                          ksplit, part_logits, x_q, x_d);
    else {
        router_logits_kernel<<<grid, R_THREADS, 0, s>>>(hidden, routerW, shexp_gate, N, D, E, Eext, ksplit,
                                                       part_logits, x_q, x_d);
        rc = launch_status();
    }
    if (rc) return rc;
    return launch_softmax(part_logits, nsplit, N, E, Eext, top_k, norm, topk_idx, topk_w,
                          shexp_gate ? shexp_scale : nullptr, logits_out, s);
}

int launch_route_small(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D, int E,
                       int top_k, int norm, int32_t *topk_idx, float *topk_w, float *shexp_scale, int8_t *x_q,
                       float *x_d, float *part_logits, int32_t *expStart, int32_t *expTokI, int32_t *expTokK,
                       unsigned *counter, unsigned *status, cudaStream_t s, bool early) {
    if (N > RS_MAX_N || N * top_k > RS_THREADS || D % 4 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int Eext = E + (shexp_gate ? 1 : 0);
    const int epl = (E + 31) / 32;
    float *sh = shexp_gate ? shexp_scale : nullptr;
    auto go = [&](auto kernel) {
        if (early)
            return launch_early(kernel, dim3(Eext), dim3(RS_THREADS), 0, s, hidden, routerW, shexp_gate, N, D, E, Eext,
                                top_k, norm, part_logits, x_q, x_d, topk_idx, topk_w, sh, expStart, expTokI, expTokK,
                                counter, status);
        kernel<<<Eext, RS_THREADS, 0, s>>>(hidden, routerW, shexp_gate, N, D, E, Eext, top_k, norm, part_logits, x_q,
                                           x_d, topk_idx, topk_w, sh, expStart, expTokI, expTokK, counter, status);
        return launch_status();
    };
    if (epl <= 1) return go(route_small_kernel<1>);
    if (epl <= 2) return go(route_small_kernel<2>);
    if (epl <= 4) return go(route_small_kernel<4>);
    if (epl <= 8) return go(route_small_kernel<8>);
    if (epl <= 16) return go(route_small_kernel<16>);
    return go(route_small_kernel<32>);
}

int launch_topk_from_logits(const float *logits, int N, int E, int top_k, int norm, int32_t *idx,
                            float *w, cudaStream_t s) {
    return launch_softmax(logits, 1, N, E, E, top_k, norm, idx, w, nullptr, nullptr, s);
}

int launch_quantize_q8_1(const float *x, int64_t nblk, int8_t *q, float *d, cudaStream_t s) {
    if (nblk <= 0) return MOE_OK;
    int64_t grid = (nblk + 7) / 8;
    quantize_q8_1_kernel<<<(unsigned)grid, 256, 0, s>>>(x, nblk, q, d);
    return launch_status();
}

}  // namespace moe
