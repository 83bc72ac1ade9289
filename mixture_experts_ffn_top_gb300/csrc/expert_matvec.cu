// expert_matvec.cu -- fused gather-matvec expert FFN on int8 dp4a
// ("full-offload MoE decode ~3.4x behind llama.cpp", #408, lever 1: one
// mul_mat_id-style launch that gathers the selected experts' rows instead of
// per-expert launches; lever 2: Q8_1 activations with int8 dp4a dots).
//
// Weight-stationary: a CTA owns 32 rows of one expert's matrix and streams
// each row once per chunk of 8 tokens of the expert's CSR segment, so for
// decode batches (a few tokens per expert) every touched weight byte is read
// once.  Each warp owns 4 rows; lane l reads 16-byte pieces l, l+32, ... of a
// row (coalesced 512 B per warp step).  Two neighbouring lanes hold the two
// halves of a 32-block; their dp4a sums are exchanged with one shuffle, which
// gives the exact int32 block dot isum_b, then acc += (d_w * d_x) * isum_b.  Q4_K
// weights (repacked to quants 0..15 with per-block scale d*sc and min dmin*m)
// add the min term: the same lanes also sum the activation codes (dp4a with
// ones), and acc -= (m_w * d_x) * xsum_b.
//
// gate/up kernel: rows = features f (gate and up), output h = SiLU(g) * u,
//   requantised to Q8_1 per 32 features inside the CTA (the CTA owns exactly
//   one 32-feature block).
// down kernel: rows = output columns c, output partial rows (scattered to
//   t*top_k + slot) or, for the shared expert, s_t * y to shared_out[t].
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int MV_T = 8;         // tokens per chunk
constexpr int MV_WARPS = 8;     // 256 threads
constexpr int MV_ROWS_PER_WARP = 4;

__device__ __forceinline__ int dp4a16(int4 w, int4 x) {
    int s = 0;
    s = __dp4a(w.x, x.x, s);
    s = __dp4a(w.y, x.y, s);
    s = __dp4a(w.z, x.z, s);
    s = __dp4a(w.w, x.w, s);
    return s;
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

// Dot of one weight row (int8 [K], scales [K/32]) against MV_T staged activation rows.
// Returns per-token fp32 sums, reduced across the warp (valid in every lane).
// If dbg != nullptr, the even lane owning block dbg_block stores its isum per token.
__device__ __forceinline__ void row_dot(const int8_t *__restrict__ wq, const float *__restrict__ wd,
                                        const float *__restrict__ wm, int K, const int8_t *xs, const float *xds,
                                        int lane, float acc[MV_T], int dbg_block, int dbg_isum[MV_T]) {
#pragma unroll
    for (int tt = 0; tt < MV_T; ++tt) acc[tt] = 0.0f;
    const int nchunks = K / 16;  // even: K is a multiple of 32
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
        // every lane runs every step (the shuffle below needs the whole warp)
        const int c = c0 + lane;
        const bool active = c < nchunks;  // lanes l and l^1 are active together
        const int b = c >> 1;
        int4 w = make_int4(0, 0, 0, 0);
        float dw = 0.0f, mw = 0.0f;
        if (active) {
            w = *reinterpret_cast<const int4 *>(wq + (size_t)c * 16);
            dw = wd[b];
            if (wm != nullptr) mw = wm[b];
        }
        const int4 ones = make_int4(0x01010101, 0x01010101, 0x01010101, 0x01010101);
        int part[MV_T], xpart[MV_T];
#pragma unroll
        for (int tt = 0; tt < MV_T; ++tt) {
            part[tt] = 0;
            xpart[tt] = 0;
            if (active) {
                int4 x = *reinterpret_cast<const int4 *>(xs + (size_t)tt * K + c * 16);
                part[tt] = dp4a16(w, x);
                if (wm != nullptr) xpart[tt] = dp4a16(ones, x);
            }
        }
#pragma unroll
        for (int tt = 0; tt < MV_T; ++tt) {
            int isum = part[tt] + __shfl_xor_sync(0xffffffffu, part[tt], 1);
            int xsum = 0;
            if (wm != nullptr) xsum = xpart[tt] + __shfl_xor_sync(0xffffffffu, xpart[tt], 1);
            if (active && (c & 1) == 0) {
                const float dx = xds[tt * (K / QK) + b];
                acc[tt] = fmaf(dw * dx, (float)isum, acc[tt]);
                if (wm != nullptr) acc[tt] = fmaf(-(mw * dx), (float)xsum, acc[tt]);
                if (b == dbg_block) dbg_isum[tt] = isum;
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < MV_T; ++tt) acc[tt] = warp_sum(acc[tt]);
}

// Stage up to MV_T activation rows (int8 [K] + fp32 scales [K/32]) into shared memory;
// missing rows are zero.  rows[tt] < 0 means "no row".
__device__ __forceinline__ void stage_rows(const int8_t *__restrict__ q, const float *__restrict__ d, int K,
                                           const int *rows, int8_t *xs, float *xds) {
    const int per_row16 = K / 16;
    for (int i = threadIdx.x; i < MV_T * per_row16; i += blockDim.x) {
        int tt = i / per_row16, c = i - tt * per_row16;
        int4 v = make_int4(0, 0, 0, 0);
        if (rows[tt] >= 0) v = *reinterpret_cast<const int4 *>(q + (size_t)rows[tt] * K + c * 16);
        *reinterpret_cast<int4 *>(xs + (size_t)tt * K + c * 16) = v;
    }
    const int nb = K / QK;
    for (int i = threadIdx.x; i < MV_T * nb; i += blockDim.x) {
        int tt = i / nb, b = i - tt * nb;
        xds[i] = rows[tt] >= 0 ? d[(size_t)rows[tt] * nb + b] : 0.0f;
    }
}

// grid (F/32, nexp); h_q/h_d rows: routed -> CSR entry j, shared -> token t.
__global__ void __launch_bounds__(MV_WARPS * 32)
matvec_gate_up_kernel(const int8_t *__restrict__ gq, const float *__restrict__ gd, const float *__restrict__ gm,
                      const int8_t *__restrict__ uq, const float *__restrict__ ud, const float *__restrict__ um,
                      int D, int F,
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
    const int fb = blockIdx.x, e = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Seg sg = segment_of(is_shared, e, expStart, N, top_k);
    if (!sg.ok) {
        if (threadIdx.x == 0) atomicOr(status, MOE_DEV_BAD_CSR);
        return;
    }
    const size_t mat_off = (size_t)(is_shared ? 0 : e) * F;
    for (int j0 = sg.s0; j0 < sg.s1; j0 += MV_T) {
        __syncthreads();  // previous chunk fully consumed
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
        stage_rows(x_q, x_d, D, rows, xs, xds);
        __syncthreads();
        for (int r = 0; r < MV_ROWS_PER_WARP; ++r) {
            const int fl = warp * MV_ROWS_PER_WARP + r;  // feature within the 32-block
            const int f = fb * QK + fl;
            float g[MV_T], u[MV_T];
            int dg[MV_T], du[MV_T];
            const size_t so = (mat_off + f) * (D / QK);
            row_dot(gq + (mat_off + f) * D, gd + so, gm ? gm + so : nullptr, D, xs, xds, lane, g, dbg_block, dg);
            row_dot(uq + (mat_off + f) * D, ud + so, um ? um + so : nullptr, D, xs, xds, lane, u, dbg_block, du);
            if (dbg_dots != nullptr && dbg_block >= 0) {
                // the even lane that owns block dbg_block (16-byte piece 2*dbg_block) holds the isums
                if (lane == ((2 * dbg_block) & 31)) {
#pragma unroll
                    for (int tt = 0; tt < MV_T; ++tt) {
                        int j = entries[tt];
                        if (j < 0 || rows[tt] < 0) continue;
                        dbg_dots[((size_t)j * 2 + 0) * F + f] = dg[tt];
                        dbg_dots[((size_t)j * 2 + 1) * F + f] = du[tt];
                    }
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int tt = 0; tt < MV_T; ++tt) {
                    float gv = g[tt];
                    float silu = gv / (1.0f + expf(-gv));
                    hs[tt * QK + fl] = silu * u[tt];
                }
            }
        }
        __syncthreads();
        // requantise: warp tt takes token tt, lane = feature of the 32-block
        if (warp < MV_T) {
            const int tt = warp;
            float d16f;
            int q = q8_quantize_lane(hs[tt * QK + lane], &d16f);
            int j = entries[tt];
            if (j >= 0 && rows[tt] >= 0) {
                h_q[(size_t)j * F + fb * QK + lane] = (int8_t)q;
                if (lane == 0) h_d[(size_t)j * (F / QK) + fb] = d16f;
            }
        }
    }
}

// grid (D/32, nexp)
__global__ void __launch_bounds__(MV_WARPS * 32)
matvec_down_kernel(const int8_t *__restrict__ dq, const float *__restrict__ dd, const float *__restrict__ dm,
                   int D, int F,
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
    const int cb = blockIdx.x, e = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Seg sg = segment_of(is_shared, e, expStart, N, top_k);
    if (!sg.ok) {
        if (threadIdx.x == 0) atomicOr(status, MOE_DEV_BAD_CSR);
        return;
    }
    const size_t mat_off = (size_t)(is_shared ? 0 : e) * D;
    for (int j0 = sg.s0; j0 < sg.s1; j0 += MV_T) {
        __syncthreads();
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
        stage_rows(h_q, h_d, F, hrows, hs, hds);
        __syncthreads();
        for (int r = 0; r < MV_ROWS_PER_WARP; ++r) {
            const int cl = warp * MV_ROWS_PER_WARP + r;
            const int c = cb * QK + cl;
            float y[MV_T];
            int unused[MV_T];
            const size_t so = (mat_off + c) * (F / QK);
            row_dot(dq + (mat_off + c) * F, dd + so, dm ? dm + so : nullptr, F, hs, hds, lane, y, -1, unused);
            if (lane == 0) {
#pragma unroll
                for (int tt = 0; tt < MV_T; ++tt) ys[tt * QK + cl] = y[tt];
            }
        }
        __syncthreads();
        if (warp < MV_T) {
            const int tt = warp;
            if (orows[tt] >= 0) {
                float v = ys[tt * QK + lane];
                if (is_shared) v = oscale[tt] * v;
                out[(size_t)orows[tt] * D + cb * QK + lane] = v;
            }
        }
    }
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
    dim3 grid(F / QK, nexp);
    matvec_gate_up_kernel<<<grid, MV_WARPS * 32, smem, s>>>(set.gate_q, set.gate_d, set.gate_m, set.up_q, set.up_d,
                                                           set.up_m, D, F,
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
    dim3 grid(D / QK, nexp);
    matvec_down_kernel<<<grid, MV_WARPS * 32, smem, s>>>(set.down_q, set.down_d, set.down_m, D, F, is_shared, h_q, h_d,
                                                        expStart, expTokI, expTokK, N, top_k, shexp_scale,
                                                        out, status);
    return launch_status();
}

}  // namespace moe
