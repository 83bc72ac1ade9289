// bucket.cu -- GPU-side expert bucketing into the expStart/expTokI/expTokK CSR
// ("Carnice prefill toward llama.cpp 676 t/s", #388, "Remaining levers" item 1:
// the bucketing that feeds the per-expert grouping must become GPU-side).
//
// One CTA, one launch: histogram, scan and a stable scatter.  Token chunks of
// 1024 are staged in shared memory (expert ids as int16).  Per chunk a bitmap
// [E][32 words] marks which tokens chose each expert (built warp-synchronously,
// no atomics); counts are popcounts, and every (token, slot) entry finds its
// position independently as the expert's base plus the popcount of the bits
// before it, so entries come out ascending in t without sorting.  When asked,
// the same CTA also writes the tensor-core path's plan (padded segments, tile
// list, row map), each row as its entry is placed.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int B_THREADS = 1024;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Optional plan of the tensor path, derived from the finished CSR in the same CTA:
// padded segment starts (16-row aligned), token tiles of <= TILE_N rows (routed
// experts first, then the shared expert's N rows) and, for every padded row, its
// source token, output row and CSR entry.
struct PlanOut {
    PlanHeader *hdr;
    int32_t *gstart;
    TileDesc *tiles;
    int4 *rowinfo;
    int with_shared, rows_max, tiles_max;
};

__global__ void __launch_bounds__(B_THREADS)
bucket_kernel(const int32_t *__restrict__ idx, int N, int k, int E, int32_t *__restrict__ expStart,
              int32_t *__restrict__ expTokI, int32_t *__restrict__ expTokK, unsigned *status, PlanOut po,
              int chunk) {
    extern __shared__ unsigned sm[];
    const int B_WORDS = chunk / 32;  // bitmap words per expert (chunk = 256, 512 or 1024 tokens)
    unsigned *cnt = sm;                                         // [E]  counts, then chunk base offsets
    int *st0 = reinterpret_cast<int *>(cnt + E);                // [E+1] segment starts
    int *gst = st0 + (E + 1);                                   // [E+2] padded starts (plan)
    int *tst = gst + (E + 2);                                   // [E+2] tile starts (plan)
    unsigned *flag = reinterpret_cast<unsigned *>(tst + (E + 2));  // [1] bad routing
    unsigned *bm = flag + 1;                                    // [E][B_WORDS] chunk bitmap
    unsigned *wpre = bm + E * B_WORDS;                          // [E][B_WORDS] popcount prefix of the words
    short *ids = reinterpret_cast<short *>(wpre + E * B_WORDS); // [B_CHUNK][k] chunk expert ids
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = N * k;
    const int nchunks = (N + chunk - 1) / chunk;
    const bool plan = po.hdr != nullptr;

    for (int e = tid; e < E; e += B_THREADS) cnt[e] = 0;
    if (tid == 0) *flag = 0;
    // Stage a chunk's expert ids (int16: E <= 1024) and build its bitmap: warp w owns
    // word w of every expert (tokens 32w..32w+31), so for each slot the lanes that chose
    // the same expert pool their bits (__match_any_sync) and one of them writes the
    // word -- no atomics, no other warp touches it.  With validate, repeats and
    // out-of-range ids raise the flag.
    auto build = [&](int t0, bool validate) {
        const int nt = min(chunk, N - t0);
        const int32_t *src = idx + (size_t)t0 * k;
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
    // counts: the popcount totals of each chunk
    for (int c = 0; c < nchunks; ++c) {
        build(c * chunk, true);
        for (int e = warp; e < E; e += B_THREADS / 32) {
            const int tot = (int)wpre[e * B_WORDS + B_WORDS - 1] + __popc(bm[e * B_WORDS + B_WORDS - 1]);
            if (lane == 0) cnt[e] += tot;
        }
        __syncthreads();
    }
    if (*flag) {
        for (int e = tid; e <= E; e += B_THREADS) expStart[e] = 0;
        if (tid == 0) {
            atomicOr(status, MOE_DEV_BAD_ROUTING);
            if (plan) {
                po.hdr->n_tiles = 0;
                po.hdr->n_rows = 0;
                po.hdr->shared_row0 = -1;
                po.hdr->pad = 0;
            }
        }
        return;
    }
    // exclusive scans (one expert per thread, E <= 1024): segment starts and, for the
    // plan, 16-row padded starts and TILE_N-row tile starts
    {
        const int c = tid < E ? (int)cnt[tid] : 0;
        const int pc = (c + SEG_ALIGN - 1) / SEG_ALIGN * SEG_ALIGN;
        const int tc = (c + TILE_N - 1) / TILE_N;
        const int i0 = warp_incl_scan(c, lane), i1 = warp_incl_scan(pc, lane), i2 = warp_incl_scan(tc, lane);
        __shared__ int wt[3][32];
        if (lane == 31) {
            wt[0][warp] = i0;
            wt[1][warp] = i1;
            wt[2][warp] = i2;
        }
        __syncthreads();
        if (warp < 3) {
            const int a = wt[warp][lane];
            const int ia = warp_incl_scan(a, lane);
            wt[warp][lane] = ia - a;
        }
        __syncthreads();
        if (tid < E) {
            const int s0 = i0 - c + wt[0][warp];
            st0[tid] = s0;
            expStart[tid] = s0;
            cnt[tid] = s0;  // base of the next chunk's entries
            gst[tid] = i1 - pc + wt[1][warp];
            tst[tid] = i2 - tc + wt[2][warp];
        }
        if (tid == E - 1) {
            st0[E] = i0 + wt[0][warp];
            expStart[E] = total;
            const int g = i1 + wt[1][warp], t = i2 + wt[2][warp];
            gst[E] = g;
            tst[E] = t;
            const int ns = po.with_shared ? N : 0;
            gst[E + 1] = g + (ns + SEG_ALIGN - 1) / SEG_ALIGN * SEG_ALIGN;
            tst[E + 1] = t + (ns + TILE_N - 1) / TILE_N;
        }
        __syncthreads();
    }
    // stable scatter: entry (t, s) of expert e goes to base + (earlier words of e in this
    // chunk) + (earlier bits of its word) -- ascending in t, computed for all entries at once
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * chunk;
        const int nt = min(chunk, N - t0);
        if (nchunks > 1) build(t0, false);  // a single chunk is still in place from the count pass
        (void)nt;
        // one warp per expert; lane r writes the expert's r-th entry of the chunk, so the
        // CSR and row-map stores of a warp go to consecutive addresses
        for (int e = warp; e < E; e += B_THREADS / 32) {
            const unsigned *be = bm + e * B_WORDS;
            const unsigned *pe = wpre + e * B_WORDS;
            const int n = (int)pe[B_WORDS - 1] + __popc(be[B_WORDS - 1]);
            const int base = (int)cnt[e];
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
                const int pos = base + r;
                expTokI[pos] = t;
                expTokK[pos] = slot;
                if (plan) {
                    const int prow = gst[e] + (pos - st0[e]);
                    if (prow < po.rows_max) po.rowinfo[prow] = make_int4(t, t * k + slot, pos, 0);
                }
            }
        }
        __syncthreads();
        for (int e = warp; e < E; e += B_THREADS / 32) {
            const int tot = (int)wpre[e * B_WORDS + B_WORDS - 1] + __popc(bm[e * B_WORDS + B_WORDS - 1]);
            if (lane == 0) cnt[e] += tot;
        }
        __syncthreads();
    }
    if (!plan) return;
    // rest of the plan: pad rows, the shared expert's rows, the tile list, the header
    for (int e = tid; e <= E + 1; e += B_THREADS) po.gstart[e] = gst[e];
    for (int e = tid; e < E; e += B_THREADS) {
        const int n = st0[e + 1] - st0[e];
        for (int r = gst[e] + n; r < gst[e + 1] && r < po.rows_max; ++r) po.rowinfo[r] = make_int4(-1, -1, -1, 0);
        for (int i = 0; i * TILE_N < n; ++i) {
            const int ti = tst[e] + i;
            if (ti >= po.tiles_max) break;
            TileDesc td;
            td.row0 = gst[e] + i * TILE_N;
            td.nrows = min(TILE_N, n - i * TILE_N);
            td.expert = e;
            td.entry0 = st0[e] + i * TILE_N;
            po.tiles[ti] = td;
        }
    }
    if (po.with_shared) {
        const int g = gst[E];
        for (int i = tid; i < gst[E + 1] - g; i += B_THREADS)
            if (g + i < po.rows_max) po.rowinfo[g + i] = i < N ? make_int4(i, i, -1, 0) : make_int4(-1, -1, -1, 0);
        for (int i = tid; i * TILE_N < N; i += B_THREADS) {
            const int ti = tst[E] + i;
            if (ti >= po.tiles_max) continue;
            TileDesc td;
            td.row0 = g + i * TILE_N;
            td.nrows = min(TILE_N, N - i * TILE_N);
            td.expert = E;
            td.entry0 = i * TILE_N;
            po.tiles[ti] = td;
        }
    }
    if (tid == 0) {
        po.hdr->n_tiles = min(tst[E + 1], po.tiles_max);
        po.hdr->n_rows = min(gst[E + 1], po.rows_max);
        po.hdr->shared_row0 = po.with_shared ? gst[E] : -1;
        po.hdr->pad = tst[E];  // routed tiles
    }
}

}  // namespace

int launch_bucket(const int32_t *topk_idx, int N, int top_k, int E, int32_t *expStart,
                  int32_t *expTokI, int32_t *expTokK, unsigned *status, cudaStream_t s, void *plan_ws,
                  const WsLayout *L, bool with_shared) {
    // the largest token chunk whose bitmaps and staged ids fit in shared memory
    auto smem_for = [&](int chunk) {
        const size_t ids_shorts = ((size_t)chunk * top_k + 1) & ~(size_t)1;
        return sizeof(unsigned) * ((size_t)E + (E + 1) + 2 * (E + 2) + 1 + 2 * (size_t)E * (chunk / 32)) +
               sizeof(short) * ids_shorts;
    };
    int chunk = 1024;
    while (chunk > 256 && smem_for(chunk) > 200 * 1024) chunk /= 2;
    const size_t smem = smem_for(chunk);
    static int configured = 0;
    if (int rc = ensure_dynamic_smem((const void *)bucket_kernel, smem, &configured)) return rc;
    PlanOut po{};
    if (plan_ws != nullptr && L != nullptr) {
        po.hdr = ws_ptr<PlanHeader>(plan_ws, L->plan);
        po.gstart = reinterpret_cast<int32_t *>(po.hdr + 1);
        po.tiles = ws_ptr<TileDesc>(plan_ws, L->tiles);
        po.rowinfo = ws_ptr<int4>(plan_ws, L->rowinfo);
        po.with_shared = with_shared ? 1 : 0;
        po.rows_max = L->rows_max;
        po.tiles_max = L->tiles_max;
    }
    bucket_kernel<<<1, B_THREADS, smem, s>>>(topk_idx, N, top_k, E, expStart, expTokI, expTokK, status, po, chunk);
    return launch_status();
}

}  // namespace moe
