// expert_matvec.cu -- fused gather-matvec expert FFN on int8 dp4a
// ("full-offload MoE decode ~3.4x behind llama.cpp", #408, lever 1: one
// mul_mat_id-style launch that gathers the selected experts' rows instead of
// per-expert launches; lever 2: Q8_1 activations with int8 dp4a dots).
//
// Weight-stationary: a work item is 32 rows of one expert's matrix, streamed
// once per chunk of up to TMAX tokens of the expert's CSR segment (TMAX from
// the batch: 1, 2, 4 or 8), so for decode batches (a few tokens per expert)
// every touched weight byte is read once.  The chunk's arithmetic is
// specialised on its token count, so a one-token segment costs one token's
// work.  The grid is persistent (the GPU's resident CTAs) over the items of
// the experts that received tokens, listed by every CTA from expStart, so an
// untouched expert costs no CTA.
// Each warp takes its rows R at a time (R = 4 for chunks of at most 2 tokens,
// else 2: gate and up of one or two features, or two or four output
// columns); lane l owns the 32-wide blocks l, l + 32, ... of those rows and
// loads all of them (2 x 16 contiguous bytes per block and row) before any
// arithmetic, so their bytes are in flight together.  Per block the lane
// forms the exact int32 dot isum_b (8 dp4a) with each staged token and
// accumulates (d_w * d_x) * isum_b; the lanes' sums are reduced at the end.
// Q4_K weights (repacked to quants 0..15 with per-block scale d*sc and min
// dmin*m) add the min term: the lane also sums the activation codes (dp4a
// with ones) and accumulates -(m_w * d_x) * xsum_b.
//
// gate/up kernel: rows = features f (gate and up), output h = SiLU(g) * u,
//   requantised to Q8_1 per 32 features inside the CTA (the CTA owns exactly
//   one 32-feature block per item).
// down kernel: rows = output columns c, output partial rows (scattered to
//   t*top_k + slot) or, for the shared expert, s_t * y to shared_out[t].
#include "moe_internal.cuh"

#include <algorithm>

namespace moe {

namespace {

constexpr int MV_T = 8;         // tokens per chunk at most
constexpr int MV_WARPS = 8;     // 256 threads
constexpr int MV_ROWS_PER_WARP = 4;

__device__ __forceinline__ int dp4a32(const int4 (&w)[2], int4 x0, int4 x1) {
    int s = 0;
    s = __dp4a(w[0].x, x0.x, s);
    s = __dp4a(w[0].y, x0.y, s);
    s = __dp4a(w[0].z, x0.z, s);
    s = __dp4a(w[0].w, x0.w, s);
    s = __dp4a(w[1].x, x1.x, s);
    s = __dp4a(w[1].y, x1.y, s);
    s = __dp4a(w[1].z, x1.z, s);
    s = __dp4a(w[1].w, x1.w, s);
    return s;
}
// sum of the 32 int8 codes of an activation block
__device__ __forceinline__ int codesum32(int4 x0, int4 x1) {
    const int4 ones[2] = {make_int4(0x01010101, 0x01010101, 0x01010101, 0x01010101),
                          make_int4(0x01010101, 0x01010101, 0x01010101, 0x01010101)};
    return dp4a32(ones, x0, x1);
}

// Segment of expert e: [s0, s1) in CSR entries; shared expert: all N tokens.
struct Seg {
    int s0, s1;
    bool ok;
};
__device__ __forceinline__ Seg segment_of(bool is_shared, int e, const int32_t *expStart, int N, int top_k) {
    Seg g;
    if (is_shared) {
        g.s0 = 0;
        g.s1 = N;
        g.ok = true;
        return g;
    }
    g.s0 = expStart[e];
    g.s1 = expStart[e + 1];
    g.ok = (g.s0 >= 0 && g.s1 >= g.s0 && g.s1 <= N * top_k);
    return g;
}

// Asks L2 for [p, p + bytes) (16-byte aligned, a multiple of 16 bytes) in pieces of at most
// 32 KB; a hint with no completion to wait for.
__device__ __forceinline__ void l2_prefetch(const void *p, size_t bytes) {
    const char *c = static_cast<const char *>(p);
    for (size_t off = 0; off < bytes; off += 32768) {
        const unsigned n = (unsigned)min((size_t)32768, bytes - off);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + off), "r"(n) : "memory");
    }
}

// List of the experts with a non-empty segment (the shared expert: {0}) in act[], count in
// *n_act; a malformed CSR raises MOE_DEV_BAD_CSR and its expert counts as empty.  Whole CTA.
__device__ __forceinline__ void active_experts(bool is_shared, int nexp, const int32_t *__restrict__ expStart, int N,
                                               int top_k, int *act, int *n_act, unsigned *status) {
    __shared__ int warp_cnt[MV_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (is_shared) {
        if (threadIdx.x == 0) {
            act[0] = 0;
            *n_act = 1;
        }
        __syncthreads();
        return;
    }
    int base = 0;
    for (int e0 = 0; e0 < nexp; e0 += MV_WARPS * 32) {
        const int e = e0 + threadIdx.x;
        bool nonempty = false;
        if (e < nexp) {
            const int s0 = expStart[e], s1 = expStart[e + 1];
            const bool ok = s0 >= 0 && s1 >= s0 && s1 <= N * top_k;
            if (!ok) atomicOr(status, MOE_DEV_BAD_CSR);
            nonempty = ok && s1 > s0;
        }
        const unsigned m = __ballot_sync(0xffffffffu, nonempty);
        if (lane == 0) warp_cnt[warp] = __popc(m);
        __syncthreads();
        int before = base;
        for (int w = 0; w < warp; ++w) before += warp_cnt[w];
        if (nonempty) act[before + __popc(m & ((1u << lane) - 1))] = e;
        for (int w = 0; w < MV_WARPS; ++w) base += warp_cnt[w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *n_act = base;
    __syncthreads();
}

// Dots of R weight rows (int8 [K], fp32 scales [K/32], fp32 mins or NULL for every row) with T
// staged activation rows (xs [T][K] int8, xds [T][K/32] fp32).  Lane l owns the 32-wide blocks
// l, l + 32, ... and loads them for all R rows before any arithmetic.  Returns per-row, per-token
// fp32 sums reduced across the warp (valid in every lane); the lane owning block dbg_block
// stores its isums.
template <int T, int R>
__device__ __forceinline__ void rows_dot(const int8_t *const (&w)[R], const float *const (&d)[R],
                                         const float *const (&m)[R], bool mins, int K, const int8_t *xs,
                                         const float *xds, int lane, float (&acc)[R][T], int dbg_block,
                                         int (&dbg)[R][T]) {
    const int nblk = K / QK;
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int tt = 0; tt < T; ++tt) acc[i][tt] = 0.0f;
    for (int b0 = 0; b0 < nblk; b0 += 64) {
        int4 q[2][R][2];
        float sc[2][R], mn[2][R];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = b0 + 32 * u + lane;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                q[u][i][0] = q[u][i][1] = make_int4(0, 0, 0, 0);
                sc[u][i] = mn[u][i] = 0.0f;
                if (b < nblk) {
                    const int4 *p = reinterpret_cast<const int4 *>(w[i] + (size_t)b * QK);
                    q[u][i][0] = __ldcs(p);
                    q[u][i][1] = __ldcs(p + 1);
                    sc[u][i] = __ldcs(d[i] + b);
                    if (mins) mn[u][i] = __ldcs(m[i] + b);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = b0 + 32 * u + lane;
            if (b >= nblk) continue;
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
                const int4 *px = reinterpret_cast<const int4 *>(xs + (size_t)tt * K + (size_t)b * QK);
                const int4 x0 = px[0], x1 = px[1];
                const float dx = xds[tt * nblk + b];
                const float xsum = mins ? (float)codesum32(x0, x1) : 0.0f;
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const int is = dp4a32(q[u][i], x0, x1);
                    acc[i][tt] = fmaf(sc[u][i] * dx, (float)is, acc[i][tt]);
                    if (mins) acc[i][tt] = fmaf(-(mn[u][i] * dx), xsum, acc[i][tt]);
                    if (b == dbg_block) dbg[i][tt] = is;
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int tt = 0; tt < T; ++tt) acc[i][tt] = warp_sum(acc[i][tt]);
}

// Rows per rows_dot call for a kernel whose chunks have at most TMAX token slots: four when the
// chunks are narrow (decode batches), two otherwise (register budget).
template <int TMAX>
struct RowsPerCall {
    static constexpr int value = TMAX <= 2 ? 4 : 2;
};

// Stage T activation rows (int8 [K] + fp32 scales [K/32]) into shared memory; rows[tt] < 0
// (no row) stages zeros.
__device__ __forceinline__ void stage_rows(const int8_t *__restrict__ q, const float *__restrict__ d, int K,
                                           const int *rows, int T, int8_t *xs, float *xds) {
    const int per_row16 = K / 16;
    for (int i = threadIdx.x; i < T * per_row16; i += blockDim.x) {
        int tt = i / per_row16, c = i - tt * per_row16;
        int4 v = make_int4(0, 0, 0, 0);
        if (rows[tt] >= 0) v = *reinterpret_cast<const int4 *>(q + (size_t)rows[tt] * K + c * 16);
        *reinterpret_cast<int4 *>(xs + (size_t)tt * K + c * 16) = v;
    }
    const int nb = K / QK;
    for (int i = threadIdx.x; i < T * nb; i += blockDim.x) {
        int tt = i / nb, b = i - tt * nb;
        xds[i] = rows[tt] >= 0 ? d[(size_t)rows[tt] * nb + b] : 0.0f;
    }
}

// Slots of a chunk of cnt tokens, rounded up to the specialisations 1, 2, 4, 8.
__device__ __forceinline__ int chunk_slots(int cnt) { return cnt <= 1 ? 1 : cnt <= 2 ? 2 : cnt <= 4 ? 4 : 8; }

struct GateUpArgs {
    const int8_t *gq, *uq;
    const float *gd, *gm, *ud, *um;
    int D, F;
    size_t mat_off;
    int8_t *h_q;
    float *h_d;
    int32_t *dbg_dots;
    int dbg_block;
};

// One chunk of T token slots of the gate/up kernel: every warp's 4 features (R/2 per rows_dot
// call: gate and up rows of each), then the Q8_1 requantisation of the 32-feature block per token.
template <int T, int R>
__device__ __forceinline__ void gate_up_chunk(const GateUpArgs &a, int fb, const int *rows, const int *entries,
                                              const int8_t *xs, const float *xds, float *hs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D;
    constexpr int NF = R / 2;  // features per call
    for (int r = 0; r < MV_ROWS_PER_WARP; r += NF) {
        const int fl0 = warp * MV_ROWS_PER_WARP + r;  // first feature within the 32-block
        const int8_t *wr[R];
        const float *dr[R], *mr[R];
#pragma unroll
        for (int i = 0; i < NF; ++i) {
            const size_t f = a.mat_off + fb * QK + fl0 + i;
            wr[2 * i] = a.gq + f * D;
            wr[2 * i + 1] = a.uq + f * D;
            dr[2 * i] = a.gd + f * (D / QK);
            dr[2 * i + 1] = a.ud + f * (D / QK);
            mr[2 * i] = a.gm ? a.gm + f * (D / QK) : nullptr;
            mr[2 * i + 1] = a.um ? a.um + f * (D / QK) : nullptr;
        }
        float acc[R][T];
        int dbg[R][T];
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int tt = 0; tt < T; ++tt) dbg[i][tt] = 0;
        rows_dot<T, R>(wr, dr, mr, a.gm != nullptr, D, xs, xds, lane, acc, a.dbg_block, dbg);
#pragma unroll
        for (int i = 0; i < NF; ++i) {
            const int fl = fl0 + i;
            const int f = fb * QK + fl;
            if (a.dbg_dots != nullptr && a.dbg_block >= 0 && lane == (a.dbg_block & 31)) {
#pragma unroll
                for (int tt = 0; tt < T; ++tt) {
                    const int j = entries[tt];
                    if (j < 0 || rows[tt] < 0) continue;
                    a.dbg_dots[((size_t)j * 2 + 0) * a.F + f] = dbg[2 * i][tt];
                    a.dbg_dots[((size_t)j * 2 + 1) * a.F + f] = dbg[2 * i + 1][tt];
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int tt = 0; tt < T; ++tt) {
                    const float gv = acc[2 * i][tt];
                    const float silu = gv / (1.0f + expf(-gv));
                    hs[tt * QK + fl] = silu * acc[2 * i + 1][tt];
                }
            }
        }
    }
    __syncthreads();
    // requantise: warp tt takes token tt, lane = feature of the 32-block
    if (warp < T) {
        const int tt = warp;
        float d16f;
        const int q = q8_quantize_lane(hs[tt * QK + lane], &d16f);
        const int j = entries[tt];
        if (j >= 0 && rows[tt] >= 0) {
            a.h_q[(size_t)j * a.F + fb * QK + lane] = (int8_t)q;
            if (lane == 0) a.h_d[(size_t)j * (a.F / QK) + fb] = d16f;
        }
    }
}

// Persistent grid over the work items (active expert, 32-feature block), expert-major;
// h_q/h_d rows: routed -> CSR entry j, shared -> token t.  TMAX: the most token slots a chunk
// can need (the launch's batch bounds every segment).
template <int TMAX>
__global__ void __launch_bounds__(MV_WARPS * 32)
matvec_gate_up_kernel(const int8_t *__restrict__ gq, const float *__restrict__ gd, const float *__restrict__ gm,
                      const int8_t *__restrict__ uq, const float *__restrict__ ud, const float *__restrict__ um,
                      int D, int F, int nexp,
                      bool is_shared, const int8_t *__restrict__ x_q, const float *__restrict__ x_d,
                      const int32_t *__restrict__ expStart, const int32_t *__restrict__ expTokI, int N,
                      int top_k, int8_t *__restrict__ h_q, float *__restrict__ h_d,
                      int32_t *__restrict__ dbg_dots, int dbg_block, unsigned *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    int8_t *xs = reinterpret_cast<int8_t *>(smem);                       // [MV_T][D]
    float *xds = reinterpret_cast<float *>(smem + (size_t)MV_T * D);    // [MV_T][D/32]
    float *hs = xds + MV_T * (D / QK);                                   // [MV_T][32]
    __shared__ int rows[MV_T];
    __shared__ int entries[MV_T];
    __shared__ int act[MAX_E];
    __shared__ int n_act;
    // the down launch that follows may start now (it waits for this kernel's h_q itself)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    active_experts(is_shared, nexp, expStart, N, top_k, act, &n_act, status);
    const int nfb = F / QK;
    for (int item = blockIdx.x; item < n_act * nfb; item += gridDim.x) {
    const int e = act[item / nfb], fb = item % nfb;
    const Seg sg = segment_of(is_shared, e, expStart, N, top_k);
    GateUpArgs a{gq, uq, gd, gm, ud, um, D, F, (size_t)(is_shared ? 0 : e) * F, h_q, h_d, dbg_dots, dbg_block};
    for (int j0 = sg.s0; j0 < sg.s1; j0 += TMAX) {
        __syncthreads();  // previous chunk fully consumed
        const int T = chunk_slots(min(TMAX, sg.s1 - j0));
        if (threadIdx.x < MV_T) {
            int j = j0 + threadIdx.x;
            int t = -1;
            if (threadIdx.x < TMAX && j < sg.s1) {
                t = is_shared ? j : expTokI[j];
                if ((unsigned)t >= (unsigned)N) {
                    atomicOr(status, MOE_DEV_BAD_CSR);
                    t = -1;
                }
            }
            rows[threadIdx.x] = t;
            entries[threadIdx.x] = (threadIdx.x < TMAX && j < sg.s1) ? j : -1;
        }
        __syncthreads();
        stage_rows(x_q, x_d, D, rows, T, xs, xds);
        __syncthreads();
        constexpr int R = RowsPerCall<TMAX>::value;
        if (T == 1) gate_up_chunk<1, R>(a, fb, rows, entries, xs, xds, hs);
        else if (TMAX >= 2 && T == 2) gate_up_chunk<(TMAX >= 2 ? 2 : 1), R>(a, fb, rows, entries, xs, xds, hs);
        else if (TMAX >= 4 && T == 4) gate_up_chunk<(TMAX >= 4 ? 4 : 1), R>(a, fb, rows, entries, xs, xds, hs);
        else if (TMAX >= 8) gate_up_chunk<(TMAX >= 8 ? 8 : 1), R>(a, fb, rows, entries, xs, xds, hs);
    }
    __syncthreads();  // the item's last chunk fully consumed before the next item stages
    }
}

struct DownArgs {
    const int8_t *dq;
    const float *dd, *dm;
    int D, F;
    size_t mat_off;
    bool is_shared;
    float *out;
    int32_t *dbg_dots;  // [entries][D] int32 dots of block dbg_block (the debug entry point), or NULL
    int dbg_block;
};

// One chunk of T token slots of the down kernel: every warp's 4 output columns (R per rows_dot
// call), then the stores of the 32-column block per token.
template <int T, int R>
__device__ __forceinline__ void down_chunk(const DownArgs &a, int cb, const int *hrows, const int *orows,
                                           const float *oscale, const int8_t *hs, const float *hds, float *ys) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int F = a.F;
    for (int r = 0; r < MV_ROWS_PER_WARP; r += R) {
        const int cl0 = warp * MV_ROWS_PER_WARP + r;
        const int8_t *wr[R];
        const float *dr[R], *mr[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const size_t c = a.mat_off + cb * QK + cl0 + i;
            wr[i] = a.dq + c * F;
            dr[i] = a.dd + c * (F / QK);
            mr[i] = a.dm ? a.dm + c * (F / QK) : nullptr;
        }
        float y[R][T];
        int dbg[R][T];
        rows_dot<T, R>(wr, dr, mr, a.dm != nullptr, F, hs, hds, lane, y, a.dbg_dots ? a.dbg_block : -1, dbg);
        if (a.dbg_dots != nullptr && !a.is_shared && lane == (a.dbg_block & 31)) {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int tt = 0; tt < T; ++tt)
                    if (hrows[tt] >= 0) a.dbg_dots[(size_t)hrows[tt] * a.D + cb * QK + cl0 + i] = dbg[i][tt];
        }
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int tt = 0; tt < T; ++tt) ys[tt * QK + cl0 + i] = y[i][tt];
        }
    }
    __syncthreads();
    if (warp < T) {
        const int tt = warp;
        if (orows[tt] >= 0) {
            float v = ys[tt * QK + lane];
            if (a.is_shared) v = oscale[tt] * v;
            a.out[(size_t)orows[tt] * a.D + cb * QK + lane] = v;
        }
    }
}

// Persistent grid over the work items (active expert, 32-column block), expert-major.
template <int TMAX>
__global__ void __launch_bounds__(MV_WARPS * 32)
matvec_down_kernel(const int8_t *__restrict__ dq, const float *__restrict__ dd, const float *__restrict__ dm,
                   int D, int F, int nexp,
                   bool is_shared, const int8_t *__restrict__ h_q, const float *__restrict__ h_d,
                   const int32_t *__restrict__ expStart, const int32_t *__restrict__ expTokI,
                   const int32_t *__restrict__ expTokK, int N, int top_k,
                   const float *__restrict__ shexp_scale, float *__restrict__ out, unsigned *status,
                   int32_t *__restrict__ dbg_dots, int dbg_block) {
    extern __shared__ __align__(16) unsigned char smem[];
    int8_t *hs = reinterpret_cast<int8_t *>(smem);                      // [MV_T][F]
    float *hds = reinterpret_cast<float *>(smem + (size_t)MV_T * F);   // [MV_T][F/32]
    float *ys = hds + MV_T * (F / QK);                                  // [MV_T][32]
    __shared__ int hrows[MV_T];
    __shared__ int orows[MV_T];
    __shared__ float oscale[MV_T];
    __shared__ int act[MAX_E];
    __shared__ int n_act;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the CSR comes from a kernel before the gate/up launch; only h_q/h_d are that launch's output
    active_experts(is_shared, nexp, expStart, N, top_k, act, &n_act, status);
    const int ncb = D / QK;
    if (threadIdx.x == 0 && (int)blockIdx.x < n_act * ncb) {
        // launched early: start this CTA's first item's rows towards L2 while gate/up finishes
        const int e = act[blockIdx.x / ncb], cb = blockIdx.x % ncb;
        const size_t r0 = (size_t)(is_shared ? 0 : e) * D + (size_t)cb * QK, sbytes = (size_t)QK * (F / QK) * 4;
        l2_prefetch(dq + r0 * F, (size_t)QK * F);
        l2_prefetch(dd + r0 * (F / QK), sbytes);
        if (dm != nullptr) l2_prefetch(dm + r0 * (F / QK), sbytes);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int item = blockIdx.x; item < n_act * ncb; item += gridDim.x) {
    const int e = act[item / ncb], cb = item % ncb;
    const Seg sg = segment_of(is_shared, e, expStart, N, top_k);
    DownArgs a{dq, dd, dm, D, F, (size_t)(is_shared ? 0 : e) * D, is_shared, out, dbg_dots, dbg_block};
    if (threadIdx.x == 0) {
        const size_t r0 = a.mat_off + (size_t)cb * QK, sbytes = (size_t)QK * (F / QK) * 4;
        l2_prefetch(dq + r0 * F, (size_t)QK * F);
        l2_prefetch(dd + r0 * (F / QK), sbytes);
        if (dm != nullptr) l2_prefetch(dm + r0 * (F / QK), sbytes);
    }
    for (int j0 = sg.s0; j0 < sg.s1; j0 += TMAX) {
        __syncthreads();
        const int T = chunk_slots(min(TMAX, sg.s1 - j0));
        if (threadIdx.x < MV_T) {
            int j = j0 + threadIdx.x;
            int hr = -1, orow = -1;
            float sc = 1.0f;
            if (threadIdx.x < TMAX && j < sg.s1) {
                if (is_shared) {
                    hr = j;
                    orow = j;
                    sc = shexp_scale[j];
                } else {
                    int t = expTokI[j], s = expTokK[j];
                    if ((unsigned)t < (unsigned)N && (unsigned)s < (unsigned)top_k) {
                        hr = j;
                        orow = t * top_k + s;
                    } else {
                        atomicOr(status, MOE_DEV_BAD_CSR);
                    }
                }
            }
            hrows[threadIdx.x] = hr;
            orows[threadIdx.x] = orow;
            oscale[threadIdx.x] = sc;
        }
        __syncthreads();
        stage_rows(h_q, h_d, F, hrows, T, hs, hds);
        __syncthreads();
        constexpr int R = RowsPerCall<TMAX>::value;
        if (T == 1) down_chunk<1, R>(a, cb, hrows, orows, oscale, hs, hds, ys);
        else if (TMAX >= 2 && T == 2) down_chunk<(TMAX >= 2 ? 2 : 1), R>(a, cb, hrows, orows, oscale, hs, hds, ys);
        else if (TMAX >= 4 && T == 4) down_chunk<(TMAX >= 4 ? 4 : 1), R>(a, cb, hrows, orows, oscale, hs, hds, ys);
        else if (TMAX >= 8) down_chunk<(TMAX >= 8 ? 8 : 1), R>(a, cb, hrows, orows, oscale, hs, hds, ys);
    }
    __syncthreads();  // the item's last chunk fully consumed before the next item stages
    }
}

// Persistent grid: the resident CTAs of the whole GPU, at most one per work item.  The
// occupancy query is remembered for the last dynamic shared-memory size seen (per kernel).
struct GridCache {
    size_t smem[MAX_DEVICES];
    int resident[MAX_DEVICES] = {};
    GridCache() {
        for (auto &v : smem) v = ~(size_t)0;
    }
};
int persistent_grid(const void *kernel, size_t smem, int max_items, GridCache *cache) {
    const int dev = current_device();
    if (dev < 0) return -1;
    if (cache->smem[dev] != smem) {
        const int n = device_sm_count();
        int per_sm = 0;
        if (n <= 0 || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, MV_WARPS * 32, smem) != cudaSuccess ||
            per_sm <= 0)
            return -1;
        cache->resident[dev] = n * per_sm;
        cache->smem[dev] = smem;
    }
    return std::max(1, std::min(cache->resident[dev], max_items));
}

}  // namespace

namespace {

// Chunk width bound of a launch: no segment is longer than the batch (a token picks an expert
// at most once; the shared expert's segment is the batch itself).
int tmax_for(int N) { return N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : MV_T; }

template <int TMAX>
int gate_up_launch(const WeightSet &set, int D, int F, int nexp, bool is_shared, const int8_t *x_q, const float *x_d,
                   const int32_t *expStart, const int32_t *expTokI, int N, int top_k, int8_t *h_q, float *h_d,
                   int32_t *dbg_dots, int dbg_block, unsigned *status, cudaStream_t s) {
    const size_t smem = (size_t)MV_T * D + sizeof(float) * ((size_t)MV_T * (D / QK) + MV_T * QK);
    static SmemOptIn configured;
    if (int rc = ensure_dynamic_smem((const void *)matvec_gate_up_kernel<TMAX>, smem, &configured)) return rc;
    static GridCache gc;
    const int grid = persistent_grid((const void *)matvec_gate_up_kernel<TMAX>, smem, nexp * (F / QK), &gc);
    if (grid < 0) return MOE_ERR_CUDA;
    matvec_gate_up_kernel<TMAX><<<grid, MV_WARPS * 32, smem, s>>>(set.gate_q, set.gate_d, set.gate_m, set.up_q,
                                                                 set.up_d, set.up_m, D, F, nexp, is_shared, x_q, x_d,
                                                                 expStart, expTokI, N, top_k, h_q, h_d, dbg_dots,
                                                                 dbg_block, status);
    return launch_status();
}

template <int TMAX>
int down_launch(const WeightSet &set, int D, int F, int nexp, bool is_shared, const int8_t *h_q, const float *h_d,
                const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK, int N, int top_k,
                const float *shexp_scale, float *out, unsigned *status, cudaStream_t s, bool early,
                int32_t *dbg_dots, int dbg_block) {
    const size_t smem = (size_t)MV_T * F + sizeof(float) * ((size_t)MV_T * (F / QK) + MV_T * QK);
    static SmemOptIn configured;
    if (int rc = ensure_dynamic_smem((const void *)matvec_down_kernel<TMAX>, smem, &configured)) return rc;
    static GridCache gc;
    const int grid = persistent_grid((const void *)matvec_down_kernel<TMAX>, smem, nexp * (D / QK), &gc);
    if (grid < 0) return MOE_ERR_CUDA;
    if (early)
        return launch_early(matvec_down_kernel<TMAX>, dim3(grid), dim3(MV_WARPS * 32), smem, s, set.down_q, set.down_d,
                            set.down_m, D, F, nexp, is_shared, h_q, h_d, expStart, expTokI, expTokK, N, top_k,
                            shexp_scale, out, status, dbg_dots, dbg_block);
    matvec_down_kernel<TMAX><<<grid, MV_WARPS * 32, smem, s>>>(set.down_q, set.down_d, set.down_m, D, F, nexp,
                                                              is_shared, h_q, h_d, expStart, expTokI, expTokK, N,
                                                              top_k, shexp_scale, out, status, dbg_dots, dbg_block);
    return launch_status();
}

}  // namespace

int launch_matvec_gate_up(const moe_weights_s *w, const WeightSet &set, bool is_shared,
                          const int8_t *x_q, const float *x_d, const int32_t *expStart,
                          const int32_t *expTokI, int N, int top_k, int8_t *h_q, float *h_d,
                          int32_t *dbg_dots, int dbg_block, unsigned *status, cudaStream_t s) {
    const int D = w->D, F = set.F;
    const int nexp = is_shared ? 1 : w->E;
    if (matvec_ring_eligible(N, D, F, N, nexp, is_shared ? N : N * top_k, set.gate_m != nullptr, x_q, x_d, set))
        return launch_matvec_ring_gate_up(set, D, F, nexp, is_shared, x_q, x_d, expStart, expTokI, N, top_k, h_q, h_d,
                                          dbg_dots, dbg_block, status, s);
    switch (tmax_for(N)) {
    case 1:
        return gate_up_launch<1>(set, D, F, nexp, is_shared, x_q, x_d, expStart, expTokI, N, top_k, h_q, h_d,
                                 dbg_dots, dbg_block, status, s);
    case 2:
        return gate_up_launch<2>(set, D, F, nexp, is_shared, x_q, x_d, expStart, expTokI, N, top_k, h_q, h_d,
                                 dbg_dots, dbg_block, status, s);
    case 4:
        return gate_up_launch<4>(set, D, F, nexp, is_shared, x_q, x_d, expStart, expTokI, N, top_k, h_q, h_d,
                                 dbg_dots, dbg_block, status, s);
    default:
        return gate_up_launch<MV_T>(set, D, F, nexp, is_shared, x_q, x_d, expStart, expTokI, N, top_k, h_q, h_d,
                                    dbg_dots, dbg_block, status, s);
    }
}

int launch_matvec_down(const moe_weights_s *w, const WeightSet &set, bool is_shared, const int8_t *h_q,
                       const float *h_d, const int32_t *expStart, const int32_t *expTokI,
                       const int32_t *expTokK, int N, int top_k, const float *shexp_scale, float *out,
                       unsigned *status, cudaStream_t s, bool early, int32_t *dbg_dots, int dbg_block) {
    const int D = w->D, F = set.F;
    const int nexp = is_shared ? 1 : w->E;
    const int rows = is_shared ? N : N * top_k;
    if (matvec_ring_eligible(N, F, D, rows, nexp, rows, set.down_m != nullptr, h_q, h_d, set))
        return launch_matvec_ring_down(set, D, F, nexp, is_shared, h_q, h_d, expStart, expTokI, expTokK, N, top_k,
                                       shexp_scale, out, status, s, early, dbg_dots, dbg_block);
    switch (tmax_for(N)) {
    case 1:
        return down_launch<1>(set, D, F, nexp, is_shared, h_q, h_d, expStart, expTokI, expTokK, N, top_k,
                              shexp_scale, out, status, s, early, dbg_dots, dbg_block);
    case 2:
        return down_launch<2>(set, D, F, nexp, is_shared, h_q, h_d, expStart, expTokI, expTokK, N, top_k,
                              shexp_scale, out, status, s, early, dbg_dots, dbg_block);
    case 4:
        return down_launch<4>(set, D, F, nexp, is_shared, h_q, h_d, expStart, expTokI, expTokK, N, top_k,
                              shexp_scale, out, status, s, early, dbg_dots, dbg_block);
    default:
        return down_launch<MV_T>(set, D, F, nexp, is_shared, h_q, h_d, expStart, expTokI, expTokK, N, top_k,
                                 shexp_scale, out, status, s, early, dbg_dots, dbg_block);
    }
}

}  // namespace moe
