// expert_matvec.cu -- fused gather-matvec expert FFN on int8 dp4a
// ("full-offload MoE decode ~3.4x behind llama.cpp", #408, lever 1: one
// mul_mat_id-style launch that gathers the selected experts' rows instead of
// per-expert launches; lever 2: Q8_1 activations with int8 dp4a dots).
//
// Weight-stationary: a work item is 32 rows of one expert's matrix, whose
// rows are streamed once per chunk of up to 8 tokens of the expert's CSR
// segment, so
// for decode batches (a few tokens per expert) every touched weight byte is
// read once.  The chunk's arithmetic is specialised on its token count
// (1, 2, 4 or 8 slots), so a one-token segment costs one token's work.  The
// grid is persistent (the GPU's resident CTAs) over the items of the experts
// that received tokens, listed by every CTA from expStart, so an untouched
// expert costs no CTA.
// Each warp takes its rows two at a time (gate and up of one feature, or two
// output columns); lane l owns the 32-wide blocks l, l + 32, ... of both rows
// and loads all of them (2 x 16 contiguous bytes per block and row) before
// any arithmetic, so the row pair's bytes are in flight together.  Per block
// the lane forms the exact int32 dot isum_b (8 dp4a) with each staged token
// and accumulates (d_w * d_x) * isum_b; the lanes' sums are reduced at the
// end.  Q4_K weights (repacked to quants 0..15 with per-block scale d*sc and
// min dmin*m) add the min term: the lane also sums the activation codes
// (dp4a with ones) and accumulates -(m_w * d_x) * xsum_b.
//
// gate/up kernel: rows = features f (gate and up), output h = SiLU(g) * u,
//   requantised to Q8_1 per 32 features inside the CTA (the CTA owns exactly
//   one 32-feature block).
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

// Dots of two weight rows a, b (int8 [K], fp32 scales [K/32], fp32 mins or NULL) with T staged
// activation rows (xs [T][K] int8, xds [T][K/32] fp32).  Returns per-token fp32 sums, reduced
// across the warp (valid in every lane).  The lane owning block dbg_block stores its isums.
template <int T>
__device__ __forceinline__ void two_rows_dot(const int8_t *__restrict__ wa, const float *__restrict__ da,
                                             const float *__restrict__ ma, const int8_t *__restrict__ wb,
                                             const float *__restrict__ db, const float *__restrict__ mb, int K,
                                             const int8_t *xs, const float *xds, int lane, float (&acc_a)[T],
                                             float (&acc_b)[T], int dbg_block, int (&dbg_a)[T], int (&dbg_b)[T]) {
    const int nblk = K / QK;
#pragma unroll
    for (int tt = 0; tt < T; ++tt) acc_a[tt] = acc_b[tt] = 0.0f;
    for (int b0 = 0; b0 < nblk; b0 += 64) {
        int4 qa[2][2], qb[2][2];
        float sa[2], sb[2], na[2], nb[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = b0 + 32 * u + lane;
            qa[u][0] = qa[u][1] = qb[u][0] = qb[u][1] = make_int4(0, 0, 0, 0);
            sa[u] = sb[u] = na[u] = nb[u] = 0.0f;
            if (b < nblk) {
                const int4 *pa = reinterpret_cast<const int4 *>(wa + (size_t)b * QK);
                const int4 *pb = reinterpret_cast<const int4 *>(wb + (size_t)b * QK);
                qa[u][0] = __ldcs(pa);
                qa[u][1] = __ldcs(pa + 1);
                qb[u][0] = __ldcs(pb);
                qb[u][1] = __ldcs(pb + 1);
                sa[u] = __ldcs(da + b);
                sb[u] = __ldcs(db + b);
                if (ma != nullptr) {
                    na[u] = __ldcs(ma + b);
                    nb[u] = __ldcs(mb + b);
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
                const int ia = dp4a32(qa[u], x0, x1), ib = dp4a32(qb[u], x0, x1);
                acc_a[tt] = fmaf(sa[u] * dx, (float)ia, acc_a[tt]);
                acc_b[tt] = fmaf(sb[u] * dx, (float)ib, acc_b[tt]);
                if (ma != nullptr) {
                    const float xsum = (float)codesum32(x0, x1);
                    acc_a[tt] = fmaf(-(na[u] * dx), xsum, acc_a[tt]);
                    acc_b[tt] = fmaf(-(nb[u] * dx), xsum, acc_b[tt]);
                }
                if (b == dbg_block) {
                    dbg_a[tt] = ia;
                    dbg_b[tt] = ib;
                }
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
        acc_a[tt] = warp_sum(acc_a[tt]);
        acc_b[tt] = warp_sum(acc_b[tt]);
    }
}

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

// One chunk of T token slots of the gate/up kernel: every warp's 4 features, then the Q8_1
// requantisation of the 32-feature block per token.
template <int T>
__device__ __forceinline__ void gate_up_chunk(const GateUpArgs &a, int fb, const int *rows, const int *entries,
                                              const int8_t *xs, const float *xds, float *hs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D;
    for (int r = 0; r < MV_ROWS_PER_WARP; ++r) {
        const int fl = warp * MV_ROWS_PER_WARP + r;  // feature within the 32-block
        const int f = fb * QK + fl;
        float g[T], u[T];
        int dg[T], du[T];
#pragma unroll
        for (int tt = 0; tt < T; ++tt) dg[tt] = du[tt] = 0;
        const size_t so = (a.mat_off + f) * (D / QK);
        two_rows_dot<T>(a.gq + (a.mat_off + f) * D, a.gd + so, a.gm ? a.gm + so : nullptr, a.uq + (a.mat_off + f) * D,
                        a.ud + so, a.um ? a.um + so : nullptr, D, xs, xds, lane, g, u, a.dbg_block, dg, du);
        if (a.dbg_dots != nullptr && a.dbg_block >= 0 && lane == (a.dbg_block & 31)) {
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
                const int j = entries[tt];
                if (j < 0 || rows[tt] < 0) continue;
                a.dbg_dots[((size_t)j * 2 + 0) * a.F + f] = dg[tt];
                a.dbg_dots[((size_t)j * 2 + 1) * a.F + f] = du[tt];
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
                const float gv = g[tt];
                const float silu = gv / (1.0f + expf(-gv));
                hs[tt * QK + fl] = silu * u[tt];
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
// h_q/h_d rows: routed -> CSR entry j, shared -> token t.
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
    active_experts(is_shared, nexp, expStart, N, top_k, act, &n_act, status);
    const int nfb = F / QK;
    for (int item = blockIdx.x; item < n_act * nfb; item += gridDim.x) {
    const int e = act[item / nfb], fb = item % nfb;
    const Seg sg = segment_of(is_shared, e, expStart, N, top_k);
    GateUpArgs a{gq, uq, gd, gm, ud, um, D, F, (size_t)(is_shared ? 0 : e) * F, h_q, h_d, dbg_dots, dbg_block};
    for (int j0 = sg.s0; j0 < sg.s1; j0 += MV_T) {
        __syncthreads();  // previous chunk fully consumed
        const int T = chunk_slots(min(MV_T, sg.s1 - j0));
        if (threadIdx.x < MV_T) {
            int j = j0 + threadIdx.x;
            int t = -1;
            if (j < sg.s1) {
                t = is_shared ? j : expTokI[j];
                if ((unsigned)t >= (unsigned)N) {
                    atomicOr(status, MOE_DEV_BAD_CSR);
                    t = -1;
                }
            }
            rows[threadIdx.x] = t;
            entries[threadIdx.x] = (j < sg.s1) ? j : -1;
        }
        __syncthreads();
        stage_rows(x_q, x_d, D, rows, T, xs, xds);
        __syncthreads();
        switch (T) {
        case 1: gate_up_chunk<1>(a, fb, rows, entries, xs, xds, hs); break;
        case 2: gate_up_chunk<2>(a, fb, rows, entries, xs, xds, hs); break;
        case 4: gate_up_chunk<4>(a, fb, rows, entries, xs, xds, hs); break;
        default: gate_up_chunk<8>(a, fb, rows, entries, xs, xds, hs); break;
        }
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
};

// One chunk of T token slots of the down kernel: every warp's 4 output columns (two pairs),
// then the stores of the 32-column block per token.
template <int T>
__device__ __forceinline__ void down_chunk(const DownArgs &a, int cb, const int *orows, const float *oscale,
                                           const int8_t *hs, const float *hds, float *ys) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int F = a.F;
    for (int r = 0; r < MV_ROWS_PER_WARP; r += 2) {
        const int cl = warp * MV_ROWS_PER_WARP + r;
        const int c = cb * QK + cl;
        float ya[T], yb[T];
        int unused_a[T], unused_b[T];
        const size_t so = (a.mat_off + c) * (F / QK), so1 = so + F / QK;
        two_rows_dot<T>(a.dq + (a.mat_off + c) * F, a.dd + so, a.dm ? a.dm + so : nullptr,
                        a.dq + (a.mat_off + c + 1) * F, a.dd + so1, a.dm ? a.dm + so1 : nullptr, F, hs, hds, lane,
                        ya, yb, -1, unused_a, unused_b);
        if (lane == 0) {
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
                ys[tt * QK + cl] = ya[tt];
                ys[tt * QK + cl + 1] = yb[tt];
            }
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
__global__ void __launch_bounds__(MV_WARPS * 32)
matvec_down_kernel(const int8_t *__restrict__ dq, const float *__restrict__ dd, const float *__restrict__ dm,
                   int D, int F, int nexp,
                   bool is_shared, const int8_t *__restrict__ h_q, const float *__restrict__ h_d,
                   const int32_t *__restrict__ expStart, const int32_t *__restrict__ expTokI,
                   const int32_t *__restrict__ expTokK, int N, int top_k,
                   const float *__restrict__ shexp_scale, float *__restrict__ out, unsigned *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    int8_t *hs = reinterpret_cast<int8_t *>(smem);                      // [MV_T][F]
    float *hds = reinterpret_cast<float *>(smem + (size_t)MV_T * F);   // [MV_T][F/32]
    float *ys = hds + MV_T * (F / QK);                                  // [MV_T][32]
    __shared__ int hrows[MV_T];
    __shared__ int orows[MV_T];
    __shared__ float oscale[MV_T];
    __shared__ int act[MAX_E];
    __shared__ int n_act;
    active_experts(is_shared, nexp, expStart, N, top_k, act, &n_act, status);
    const int ncb = D / QK;
    for (int item = blockIdx.x; item < n_act * ncb; item += gridDim.x) {
    const int e = act[item / ncb], cb = item % ncb;
    const Seg sg = segment_of(is_shared, e, expStart, N, top_k);
    DownArgs a{dq, dd, dm, D, F, (size_t)(is_shared ? 0 : e) * D, is_shared, out};
    for (int j0 = sg.s0; j0 < sg.s1; j0 += MV_T) {
        __syncthreads();
        const int T = chunk_slots(min(MV_T, sg.s1 - j0));
        if (threadIdx.x < MV_T) {
            int j = j0 + threadIdx.x;
            int hr = -1, orow = -1;
            float sc = 1.0f;
            if (j < sg.s1) {
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
        switch (T) {
        case 1: down_chunk<1>(a, cb, orows, oscale, hs, hds, ys); break;
        case 2: down_chunk<2>(a, cb, orows, oscale, hs, hds, ys); break;
        case 4: down_chunk<4>(a, cb, orows, oscale, hs, hds, ys); break;
        default: down_chunk<8>(a, cb, orows, oscale, hs, hds, ys); break;
        }
    }
    __syncthreads();  // the item's last chunk fully consumed before the next item stages
    }
}

// Persistent grid: the resident CTAs of the whole GPU, at most one per work item.  The
// occupancy query is remembered for the last dynamic shared-memory size seen (per kernel).
struct GridCache {
    size_t smem = ~(size_t)0;
    int resident = 0;
};
int persistent_grid(const void *kernel, size_t smem, int max_items, GridCache *cache) {
    if (cache->smem != smem) {
        int dev = 0, n = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0 ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, MV_WARPS * 32, smem) != cudaSuccess ||
            per_sm <= 0)
            return -1;
        cache->resident = n * per_sm;
        cache->smem = smem;
    }
    return std::max(1, std::min(cache->resident, max_items));
}

}  // namespace

int launch_matvec_gate_up(const moe_weights_s *w, const WeightSet &set, bool is_shared,
                          const int8_t *x_q, const float *x_d, const int32_t *expStart,
                          const int32_t *expTokI, int N, int top_k, int8_t *h_q, float *h_d,
                          int32_t *dbg_dots, int dbg_block, unsigned *status, cudaStream_t s) {
    const int D = w->D, F = set.F;
    const int nexp = is_shared ? 1 : w->E;
    size_t smem = (size_t)MV_T * D + sizeof(float) * ((size_t)MV_T * (D / QK) + MV_T * QK);
    static int configured = 0;
    if (int rc = ensure_dynamic_smem((const void *)matvec_gate_up_kernel, smem, &configured)) return rc;
    static GridCache gc;
    const int grid = persistent_grid((const void *)matvec_gate_up_kernel, smem, nexp * (F / QK), &gc);
    if (grid < 0) return MOE_ERR_CUDA;
    matvec_gate_up_kernel<<<grid, MV_WARPS * 32, smem, s>>>(set.gate_q, set.gate_d, set.gate_m, set.up_q, set.up_d,
                                                           set.up_m, D, F, nexp,
                                                           is_shared, x_q, x_d, expStart, expTokI, N, top_k,
                                                           h_q, h_d, dbg_dots, dbg_block, status);
    return launch_status();
}

int launch_matvec_down(const moe_weights_s *w, const WeightSet &set, bool is_shared, const int8_t *h_q,
                       const float *h_d, const int32_t *expStart, const int32_t *expTokI,
                       const int32_t *expTokK, int N, int top_k, const float *shexp_scale, float *out,
                       unsigned *status, cudaStream_t s) {
    const int D = w->D, F = set.F;
    const int nexp = is_shared ? 1 : w->E;
    size_t smem = (size_t)MV_T * F + sizeof(float) * ((size_t)MV_T * (F / QK) + MV_T * QK);
    static int configured = 0;
    if (int rc = ensure_dynamic_smem((const void *)matvec_down_kernel, smem, &configured)) return rc;
    static GridCache gc;
    const int grid = persistent_grid((const void *)matvec_down_kernel, smem, nexp * (D / QK), &gc);
    if (grid < 0) return MOE_ERR_CUDA;
    matvec_down_kernel<<<grid, MV_WARPS * 32, smem, s>>>(set.down_q, set.down_d, set.down_m, D, F, nexp, is_shared,
                                                        h_q, h_d,
                                                        expStart, expTokI, expTokK, N, top_k, shexp_scale,
                                                        out, status);
    return launch_status();
}

}  // namespace moe
