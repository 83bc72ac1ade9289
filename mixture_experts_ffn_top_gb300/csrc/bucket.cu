// bucket.cu -- GPU-side expert bucketing into the expStart/expTokI/expTokK CSR
// ("Carnice prefill toward llama.cpp 676 t/s", #388, "Remaining levers" item 1:
// the bucketing that feeds the per-expert grouping must become GPU-side).
//
// One CTA, one launch: histogram, scan and a stable scatter.  The scatter
// works on chunks of 1024 tokens: a bitmap [E][32 words] marks which tokens
// of the chunk chose each expert; one warp per expert walks its 32 words in
// lane order with a popcount prefix, so entries come out ascending in t
// without sorting and without atomics on the output.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int B_THREADS = 1024;
constexpr int B_CHUNK = 1024;             // tokens per bitmap chunk
constexpr int B_WORDS = B_CHUNK / 32;     // bitmap words per expert

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__global__ void __launch_bounds__(B_THREADS)
bucket_kernel(const int32_t *__restrict__ idx, int N, int k, int E, int32_t *__restrict__ expStart,
              int32_t *__restrict__ expTokI, int32_t *__restrict__ expTokK, unsigned *status) {
    extern __shared__ unsigned sm[];
    unsigned *cnt = sm;                 // [E]  counts, then running fill offsets
    unsigned *wsum = sm + E;            // [32] warp totals for the scan
    unsigned *flag = wsum + 32;         // [1]  bad routing
    unsigned *bm = flag + 1;            // [E][B_WORDS]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = N * k;

    for (int e = tid; e < E; e += B_THREADS) cnt[e] = 0;
    if (tid == 0) *flag = 0;
    __syncthreads();
    // histogram + validation
    for (int i = tid; i < total; i += B_THREADS) {
        int e = idx[i];
        if ((unsigned)e >= (unsigned)E) {
            *flag = 1;
        } else {
            atomicAdd(&cnt[e], 1u);
            int t = i / k, s = i - t * k;
            for (int s2 = 0; s2 < s; ++s2)
                if (idx[t * k + s2] == e) *flag = 1;
        }
    }
    __syncthreads();
    if (*flag) {
        for (int e = tid; e <= E; e += B_THREADS) expStart[e] = 0;
        if (tid == 0) atomicOr(status, MOE_DEV_BAD_ROUTING);
        return;
    }
    // exclusive scan of cnt over E <= 1024 experts (one value per thread)
    int v = tid < E ? (int)cnt[tid] : 0;
    int inc = warp_incl_scan(v, lane);
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int wv = wsum[lane];
        int winc = warp_incl_scan(wv, lane);
        wsum[lane] = winc - wv;
    }
    __syncthreads();
    int excl = inc - v + (int)wsum[warp];
    __syncthreads();
    if (tid < E) {
        expStart[tid] = excl;
        cnt[tid] = excl;  // running fill offset
    }
    if (tid == 0) expStart[E] = total;
    __syncthreads();

    for (int t0 = 0; t0 < N; t0 += B_CHUNK) {
        const int nt = min(B_CHUNK, N - t0);
        for (int i = tid; i < E * B_WORDS; i += B_THREADS) bm[i] = 0;
        __syncthreads();
        for (int i = tid; i < nt * k; i += B_THREADS) {
            int tl = i / k;
            int e = idx[(size_t)t0 * k + i];
            atomicOr(&bm[e * B_WORDS + (tl >> 5)], 1u << (tl & 31));
        }
        __syncthreads();
        for (int e = warp; e < E; e += B_THREADS / 32) {
            unsigned word = bm[e * B_WORDS + lane];
            int c = __popc(word);
            int pre = warp_incl_scan(c, lane) - c;
            int tot = __shfl_sync(0xffffffffu, pre + c, 31);
            int pos = (int)cnt[e] + pre;
            while (word) {
                int b = __ffs(word) - 1;
                word &= word - 1;
                int t = t0 + lane * 32 + b;
                int slot = 0;
                for (int s = 0; s < k; ++s)
                    if (idx[(size_t)t * k + s] == e) slot = s;
                expTokI[pos] = t;
                expTokK[pos] = slot;
                ++pos;
            }
            __syncwarp();
            if (lane == 0) cnt[e] += tot;
            __syncwarp();
        }
        __syncthreads();
    }
}

}  // namespace

int launch_bucket(const int32_t *topk_idx, int N, int top_k, int E, int32_t *expStart,
                  int32_t *expTokI, int32_t *expTokK, unsigned *status, cudaStream_t s) {
    size_t smem = sizeof(unsigned) * ((size_t)E + 33 + (size_t)E * B_WORDS);
    static int configured = 0;
    if (int rc = ensure_dynamic_smem((const void *)bucket_kernel, smem, &configured)) return rc;
    bucket_kernel<<<1, B_THREADS, smem, s>>>(topk_idx, N, top_k, E, expStart, expTokI, expTokK, status);
    return launch_status();
}

}  // namespace moe
