// bucket.cu -- GPU-side expert bucketing into the expStart/expTokI/expTokK CSR
// ("Carnice prefill toward llama.cpp 676 t/s", #388, "Remaining levers" item 1:
// the bucketing that feeds the per-expert grouping must become GPU-side).
//
// One cooperative launch of G CTAs, each owning a contiguous range of tokens:
//   1. histogram: per range and expert, how many (token, slot) entries it holds;
//   2. grid barrier (bounded), then every CTA scans the G x E count table: segment
//      starts, and the base of its own entries inside each segment;
//   3. stable scatter of the range's entries, and (when asked) the tensor-core
//      path's plan: padded segments, tile list, row map.
// Within a range, token chunks are staged in shared memory (expert ids as int16).
// Per chunk a bitmap [E][chunk/32 words] marks which tokens chose each expert
// (built warp-synchronously, no atomics); counts are popcounts, and every entry
// finds its position as its base plus the popcount of the bits before it, so
// entries come out ascending in t without sorting.
#include "moe_internal.cuh"

#include <algorithm>

namespace moe {

namespace {

constexpr int B_THREADS = 1024;
constexpr int B_MIN_RANGE = 128;  // tokens per CTA at least
constexpr unsigned long long B_BARRIER_NS = 1000000000ull;  // 1 s: a healthy barrier takes microseconds
constexpr unsigned long long B_BARRIER_NS_MIN = 1000000ull;  // the shortest limit a caller may ask for (1 ms)

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid barrier for a cooperative launch: arrival counter plus a generation word (both in
// the workspace's status block, zero after moe_workspace_init and back to zero after every
// completed barrier).  The wait is bounded; on expiry the CTA raises MOE_DEV_TIMEOUT and
// reports failure (every CTA then returns without writing results).
__device__ bool grid_barrier(unsigned *count, unsigned *gen, unsigned nblocks, unsigned *status,
                             unsigned long long limit_ns) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok_s = 1;
        const unsigned g0 = *reinterpret_cast<volatile unsigned *>(gen);
        __threadfence();
        if (atomicAdd(count, 1u) == nblocks - 1) {
            *reinterpret_cast<volatile unsigned *>(count) = 0;
            __threadfence();
            atomicAdd(gen, 1u);
        } else {
            const unsigned long long t0 = gtimer();
            while (*reinterpret_cast<volatile unsigned *>(gen) == g0) {
                if (gtimer() - t0 > limit_ns) {
                    atomicOr(status, MOE_DEV_TIMEOUT);
                    ok_s = 0;
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    return ok_s != 0;
}

// Optional plan of the tensor path, derived from the CSR: padded segment starts
// (16-row aligned), token tiles of <= tile_n rows (routed experts first, then the
// shared expert's N rows) and, for every padded row, its source token, output row
// and CSR entry.
struct PlanOut {
    PlanHeader *hdr;
    int32_t *gstart;
    TileDesc *tiles;
    int4 *rowinfo;
    int with_shared, rows_max, tiles_max;
    int tile_n;  // token rows per tile
};

struct BucketArgs {
    const int32_t *idx;
    int N, k, E;
    int32_t *expStart, *expTokI, *expTokK;
    unsigned *status, *bar_count, *bar_gen;
    int *cnt_g;   // [G][E] per-range counts
    int *bad_g;   // [G] per-range "bad routing" flags
    int range;    // tokens per CTA (multiple of 32)
    int chunk;    // tokens staged at a time (256, 512 or 1024)
    unsigned long long barrier_ns;  // limit of the grid barrier's wait
    int extra_arrivals;  // failure-detection check: arrivals the barrier waits for beyond the grid (0 normally)
    int counts_ready;    // the count table (and zero bad flags) already written by the router launch, whose
                         // 128-token tiles are these ranges: no histogram pass, no grid barrier
};

__global__ void __launch_bounds__(B_THREADS, 1) bucket_kernel(const BucketArgs a, const PlanOut po) {
    extern __shared__ unsigned sm[];
    const int E = a.E, k = a.k, N = a.N;
    const int B_WORDS = a.chunk / 32;  // bitmap words per expert
    int *base = reinterpret_cast<int *>(sm);                   // [E] next entry of each expert (this range)
    int *st0 = base + E;                                       // [E+1] segment starts
    int *gst = st0 + (E + 1);                                  // [E+2] padded starts (plan)
    int *tst = gst + (E + 2);                                  // [E+2] tile starts (plan)
    unsigned *flag = reinterpret_cast<unsigned *>(tst + (E + 2));  // [1] bad routing in this range
    unsigned *bm = flag + 1;                                   // [E][B_WORDS] chunk bitmap
    unsigned *wpre = bm + E * B_WORDS;                         // [E][B_WORDS] popcount prefix of the words
    short *ids = reinterpret_cast<short *>(wpre + E * B_WORDS);  // [chunk][k] chunk expert ids
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, b = blockIdx.x;
    const int total = N * k;
    const int r0 = b * a.range, r1 = min(N, r0 + a.range);
    const int nchunks = r1 > r0 ? (r1 - r0 + a.chunk - 1) / a.chunk : 0;
    const bool plan = po.hdr != nullptr;

    for (int e = tid; e < E; e += B_THREADS) base[e] = 0;
    if (tid == 0) *flag = 0;
    // Stage a chunk's expert ids (int16: E <= 1024) and build its bitmap: warp w owns
    // word w of every expert (tokens 32w..32w+31), so for each slot the lanes that chose
    // the same expert pool their bits (__match_any_sync) and one of them writes the
    // word -- no atomics, no other warp touches it.  With validate, repeats and
    // out-of-range ids raise the flag.
    auto build = [&](int t0, bool validate) {
        const int nt = min(a.chunk, r1 - t0);
        const int32_t *src = a.idx + (size_t)t0 * k;
        for (int i = tid; i < nt * k; i += B_THREADS) ids[i] = (short)max(-1, min(src[i], 32767));
        for (int i = tid; i < E * B_WORDS; i += B_THREADS) bm[i] = 0;
        __syncthreads();
        const bool mine = tid < nt;
        for (int s = 0; s < k; ++s) {
            int e = mine ? ids[tid * k + s] : -1;
            if (mine && validate) {
                if (e < 0 || e >= E) *flag = 1;
                for (int s2 = 0; s2 < s; ++s2)
                    if (ids[tid * k + s2] == e) *flag = 1;
            }
            if (e < 0 || e >= E) e = -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && lane == __ffs(peers) - 1) bm[e * B_WORDS + warp] |= peers;
        }
        __syncthreads();
        // per expert: exclusive popcount prefix over its words (lane = word)
        for (int e = warp; e < E; e += B_THREADS / 32) {
            const int pc = lane < B_WORDS ? __popc(bm[e * B_WORDS + lane]) : 0;
            const int pre = warp_incl_scan(pc, lane) - pc;
            if (lane < B_WORDS) wpre[e * B_WORDS + lane] = pre;
        }
        __syncthreads();
    };
    auto chunk_count = [&](int e) {
        return (int)wpre[e * B_WORDS + B_WORDS - 1] + __popc(bm[e * B_WORDS + B_WORDS - 1]);
    };
    // 1. histogram of this range
    for (int c = 0; c < nchunks && !a.counts_ready; ++c) {
        build(r0 + c * a.chunk, true);
        for (int e = warp; e < E; e += B_THREADS / 32)
            if (lane == 0) base[e] += chunk_count(e);
        __syncthreads();
    }
    // 2. all ranges counted (a single range needs neither the count table nor the barrier)
    int bad = 0;
    if (a.counts_ready) {
        __syncthreads();
    } else if (G > 1) {
        for (int e = tid; e < E; e += B_THREADS) a.cnt_g[(size_t)b * E + e] = base[e];
        if (tid == 0) a.bad_g[b] = (int)*flag;
        if (!grid_barrier(a.bar_count, a.bar_gen, (unsigned)(G + a.extra_arrivals), a.status, a.barrier_ns)) return;
        for (int i = tid; i < G; i += B_THREADS) bad |= __ldcg(a.bad_g + i);
    } else {
        __syncthreads();
        bad = (int)*flag;
    }
    if (__syncthreads_or(bad)) {
        if (b == 0) {
            for (int e = tid; e <= E; e += B_THREADS) a.expStart[e] = 0;
            if (tid == 0) {
                atomicOr(a.status, MOE_DEV_BAD_ROUTING);
                if (plan) {
                    po.hdr->n_tiles = 0;
                    po.hdr->n_rows = 0;
                    po.hdr->shared_row0 = -1;
                    po.hdr->pad = 0;
                }
            }
        }
        return;
    }
    // per expert: total over all ranges and the entries of the ranges before this one;
    // then exclusive scans over experts (one per thread, E <= 1024): segment starts and,
    // for the plan, 16-row padded starts and tile_n-row tile starts
    {
        int c = 0, before = 0;
        if (tid < E) {
            if (G == 1 && !a.counts_ready) {
                c = base[tid];
            } else {
                // the column of expert tid, eight loads in flight at a time
                int j = 0;
                for (; j + 8 <= G; j += 8) {
                    int v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = __ldcg(a.cnt_g + (size_t)(j + u) * E + tid);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (j + u < b) before += v[u];
                        c += v[u];
                    }
                }
                for (; j < G; ++j) {
                    const int v = __ldcg(a.cnt_g + (size_t)j * E + tid);
                    if (j < b) before += v;
                    c += v;
                }
            }
        }
        __syncthreads();  // every count read before base[] is rewritten below
        const int pc = (c + SEG_ALIGN - 1) / SEG_ALIGN * SEG_ALIGN;
        const int tc = (c + po.tile_n - 1) / po.tile_n;
        const int i0 = warp_incl_scan(c, lane), i1 = warp_incl_scan(pc, lane), i2 = warp_incl_scan(tc, lane);
        __shared__ int wt[3][32];
        if (lane == 31) {
            wt[0][warp] = i0;
            wt[1][warp] = i1;
            wt[2][warp] = i2;
        }
        __syncthreads();
        if (warp < 3) {
            const int av = wt[warp][lane];
            const int ia = warp_incl_scan(av, lane);
            wt[warp][lane] = ia - av;
        }
        __syncthreads();
        if (tid < E) {
            const int s0 = i0 - c + wt[0][warp];
            st0[tid] = s0;
            if (b == 0) a.expStart[tid] = s0;
            base[tid] = s0 + before;  // this range's first entry of the segment
            gst[tid] = i1 - pc + wt[1][warp];
            tst[tid] = i2 - tc + wt[2][warp];
        }
        if (tid == E - 1) {
            st0[E] = i0 + wt[0][warp];
            if (b == 0) a.expStart[E] = total;
            const int g = i1 + wt[1][warp], t = i2 + wt[2][warp];
            gst[E] = g;
            tst[E] = t;
            const int ns = po.with_shared ? N : 0;
            gst[E + 1] = g + (ns + SEG_ALIGN - 1) / SEG_ALIGN * SEG_ALIGN;
            tst[E + 1] = t + (ns + po.tile_n - 1) / po.tile_n;
        }
        __syncthreads();
    }
    // 3. stable scatter: entry (t, s) of expert e goes to the range's base + (earlier words
    // of e in this chunk) + (earlier bits of its word) -- ascending in t
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = r0 + c * a.chunk;
        if (nchunks > 1 || a.counts_ready) build(t0, false);  // a single chunk stays in place from the count pass
        // one warp per expert; lane r writes the expert's r-th entry of the chunk, so the
        // CSR and row-map stores of a warp go to consecutive addresses
        for (int e = warp; e < E; e += B_THREADS / 32) {
            const unsigned *be = bm + e * B_WORDS;
            const unsigned *pe = wpre + e * B_WORDS;
            const int n = chunk_count(e);
            const int eb = base[e];
            for (int r = lane; r < n; r += 32) {
                int lo = 0, hi = B_WORDS;  // the word holding the r-th set bit: pe[w] <= r < pe[w+1]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if ((int)pe[mid] <= r) lo = mid;
                    else hi = mid;
                }
                const int bit = (int)__fns(be[lo], 0, r - (int)pe[lo] + 1);
                const int tl = lo * 32 + bit;
                const short *my = ids + tl * k;
                int slot = 0;
                for (int s = 0; s < k; ++s)
                    if (my[s] == e) slot = s;
                const int t = t0 + tl;
                const int pos = eb + r;
                if (pos >= total) continue;  // a count table that disagrees with the routing
                a.expTokI[pos] = t;
                a.expTokK[pos] = slot;
                if (plan) {
                    const int prow = gst[e] + (pos - st0[e]);
                    if (prow < po.rows_max) po.rowinfo[prow] = make_int4(t, t * k + slot, pos, 0);
                }
            }
        }
        __syncthreads();
        for (int e = warp; e < E; e += B_THREADS / 32)
            if (lane == 0) base[e] += chunk_count(e);
        __syncthreads();
    }
    if (!plan) return;
    // rest of the plan, spread over the CTAs: pad rows and tiles of the experts e = b (mod G)
    // (one warp each), the shared expert's rows of this token range and its tiles i = b
    // (mod G), the header
    if (b == 0)
        for (int e = tid; e <= E + 1; e += B_THREADS) po.gstart[e] = gst[e];
    for (int e = b + G * warp; e < E; e += G * (B_THREADS / 32)) {
        const int n = st0[e + 1] - st0[e];
        for (int r = gst[e] + n + lane; r < gst[e + 1] && r < po.rows_max; r += 32)
            po.rowinfo[r] = make_int4(-1, -1, -1, 0);
        for (int i = lane; i * po.tile_n < n; i += 32) {
            const int ti = tst[e] + i;
            if (ti >= po.tiles_max) break;
            TileDesc td;
            td.row0 = gst[e] + i * po.tile_n;
            td.nrows = min(po.tile_n, n - i * po.tile_n);
            td.expert = e;
            td.entry0 = st0[e] + i * po.tile_n;
            po.tiles[ti] = td;
        }
    }
    if (po.with_shared) {
        const int g = gst[E];
        const int rend = (b == G - 1) ? gst[E + 1] - g : r1;  // the last range also takes the pad rows
        for (int i = r0 + tid; i < rend; i += B_THREADS)
            if (g + i < po.rows_max) po.rowinfo[g + i] = i < N ? make_int4(i, i, -1, 0) : make_int4(-1, -1, -1, 0);
        for (int i = b + G * tid; i * po.tile_n < N; i += G * B_THREADS) {
            const int ti = tst[E] + i;
            if (ti >= po.tiles_max) continue;
            TileDesc td;
            td.row0 = g + i * po.tile_n;
            td.nrows = min(po.tile_n, N - i * po.tile_n);
            td.expert = E;
            td.entry0 = i * po.tile_n;
            po.tiles[ti] = td;
        }
    }
    if (b == 0 && tid == 0) {
        po.hdr->n_tiles = min(tst[E + 1], po.tiles_max);
        po.hdr->n_rows = min(gst[E + 1], po.rows_max);
        po.hdr->shared_row0 = po.with_shared ? gst[E] : -1;
        po.hdr->pad = tst[E];  // routed tiles
    }
}

}  // namespace

// Ranges: at least B_MIN_RANGE tokens per CTA, at most one CTA per SM, and a count table
// of at most BUCKET_TABLE_MAX ints.
int bucket_grid(int N, int E, int *range_out) {
    const int num_sms = std::max(1, device_sm_count());
    const int gmax = std::min(num_sms, std::max(1, BUCKET_TABLE_MAX / std::max(E, 1)));
    int range = std::max(B_MIN_RANGE, (N + gmax - 1) / gmax);
    range = (range + 31) / 32 * 32;
    if (range_out) *range_out = range;
    return std::max(1, (N + range - 1) / range);
}

size_t bucket_scratch_bytes(int N, int E) {
    const int G = bucket_grid(N, E, nullptr);
    return ((size_t)G * E + G) * sizeof(int);
}

int launch_bucket(const int32_t *topk_idx, int N, int top_k, int E, int32_t *expStart, int32_t *expTokI,
                  int32_t *expTokK, void *ws, cudaStream_t s, const WsLayout *L, bool with_shared, int tile_rows,
                  unsigned long long barrier_ns, int extra_arrivals, bool counts_ready) {
    if (tile_rows < SEG_ALIGN || tile_rows % SEG_ALIGN) return MOE_ERR_INVALID_ARG;
    if (barrier_ns == 0) barrier_ns = B_BARRIER_NS;
    if (barrier_ns < B_BARRIER_NS_MIN || extra_arrivals < 0) return MOE_ERR_INVALID_ARG;
    int range = 0;
    const int G = bucket_grid(N, E, &range);
    // the largest token chunk (<= the range) whose bitmaps and staged ids fit in shared memory
    auto smem_for = [&](int chunk) {
        const size_t ids_shorts = ((size_t)chunk * top_k + 1) & ~(size_t)1;
        return sizeof(unsigned) * ((size_t)E + (E + 1) + 2 * (E + 2) + 1 + 2 * (size_t)E * (chunk / 32)) +
               sizeof(short) * ids_shorts;
    };
    int chunk = 1024;
    while (chunk > 128 && (smem_for(chunk) > 200 * 1024 || chunk / 2 >= range)) chunk /= 2;
    const size_t smem = smem_for(chunk);
    static SmemOptIn configured;
    if (int rc = ensure_dynamic_smem((const void *)bucket_kernel, smem, &configured)) return rc;
    uint8_t *wb = static_cast<uint8_t *>(ws);
    BucketArgs a{};
    a.idx = topk_idx;
    a.N = N;
    a.k = top_k;
    a.E = E;
    a.expStart = expStart;
    a.expTokI = expTokI;
    a.expTokK = expTokK;
    a.status = reinterpret_cast<unsigned *>(wb);
    a.bar_count = reinterpret_cast<unsigned *>(wb + BUCKET_BARRIER_OFFSET);
    a.bar_gen = reinterpret_cast<unsigned *>(wb + BUCKET_BARRIER_OFFSET + 64);
    a.cnt_g = reinterpret_cast<int *>(wb + BUCKET_SCRATCH_OFFSET);
    a.bad_g = a.cnt_g + (size_t)G * E;
    a.range = range;
    a.chunk = chunk;
    a.barrier_ns = barrier_ns;
    a.extra_arrivals = extra_arrivals;
    a.counts_ready = counts_ready ? 1 : 0;
    if (extra_arrivals > 0 && (G == 1 || counts_ready)) return MOE_ERR_UNSUPPORTED_SHAPE;  // no grid barrier
    PlanOut po{};
    po.tile_n = tile_rows;
    if (L != nullptr) {
        po.hdr = ws_ptr<PlanHeader>(ws, L->plan);
        po.gstart = reinterpret_cast<int32_t *>(po.hdr + 1);
        po.tiles = ws_ptr<TileDesc>(ws, L->tiles);
        po.rowinfo = ws_ptr<int4>(ws, L->rowinfo);
        po.with_shared = with_shared ? 1 : 0;
        po.rows_max = L->rows_max;
        po.tiles_max = L->tiles_max;
    }
    if (G == 1 || counts_ready) {  // no grid barrier, so no cooperative launch either
        bucket_kernel<<<G, B_THREADS, smem, s>>>(a, po);
        return launch_status();
    }
    void *args[] = {(void *)&a, (void *)&po};
    return cuda_status(
        cudaLaunchCooperativeKernel((const void *)bucket_kernel, dim3(G), dim3(B_THREADS), args, smem, s));
}

}  // namespace moe
