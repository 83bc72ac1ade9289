// matvec_ring.cu -- the expert matvecs of decode batches (at most 8 tokens) with the weight rows
// streamed through a shared-memory ring ("full-offload MoE decode ~3.4x behind llama.cpp", #408,
// lever 1: one mul_mat_id-style launch over the selected experts' rows; lever 2: Q8_1
// activations with int8 dp4a dots).
//
// A decode batch reads every touched weight byte once, so the launch is bound by how many bytes
// each SM keeps in flight.  Here one thread per CTA (the producer) issues bulk copies of whole
// weight-row spans (contiguous in the repacked layout) into a ring of stages, each completing on
// its own mbarrier, and runs ahead of the arithmetic by the ring's depth; eight consumer warps
// take the stages in order and hand each one back with one arrival per warp.  The activation
// rows of the whole batch (x for gate/up, every CSR entry's h for down) are staged once per CTA.
//
// Work item: 32 output rows of one expert (gate/up: a 32-feature block, both matrices; down: a
// 32-column block) for one chunk of at most 8 of the expert's CSR entries; stage: 8 features
// (8 gate + 8 up rows) or 16 down rows, with their block scales (and Q4_K mins).  Consumer warp w
// takes rows w and w + 8 of each stage; lane l the 32-wide blocks l, l + 32, ...  Per block the
// exact int32 dot isum_b (8 dp4a) and acc = fma(d_w * d_x, isum_b, acc) (Q4_K: then
// acc = fma(-(m_w * d_x), xsum_b, acc)), the lanes' sums reduced by warp_sum: the same
// operations in the same order as the register-loading matvec kernels, so both give identical
// bits.  gate/up: SiLU(g) * u per feature into a shared block buffer; the warp that finishes an
// item last requantises its 32 features per token (Q8_1).  down: unweighted partial rows to
// t * top_k + slot, or s_t * y for the shared expert.
//
// Q4_K weights stream in their nibble-packed copy (16 bytes per 32-block, byte j = q[j] | q[j+16] << 4):
// half the quant bytes; each lane unpacks its block into the same two 16-code halves, so the int32
// dots, and with them the results, are the same bits.
//
// Every wait is bounded (MOE_DEV_TIMEOUT, then every role drains out; the producer waits, bounded,
// for its copies in flight before the CTA exits).
#include "moe_internal.cuh"
#include "tc_glue.cuh"

#include <algorithm>

namespace moe {

namespace {

using namespace tc;

constexpr int RG_CW = 8;                      // consumer warps
constexpr int RG_THREADS = 32 * (RG_CW + 1);  // + the producer warp (warp 0)
constexpr int RG_CHUNK = 8;                   // CSR entries per work item at most
constexpr int RG_MAX_STAGES = 8;
constexpr int RG_HBUF = 3;                    // gate/up block buffers (see the consumer loop)
constexpr unsigned long long RG_WAIT_NS = 2000000000ull;
constexpr int RG_PAIR_SHIFT = 11;             // act entry: expert | chunk << 11 (experts < 2048)

struct RingArgs {
    // weights of the launch's matrices: gate/up q0/d0/m0 = gate, q1/d1/m1 = up ([nexp*F][D]);
    // down q0/d0/m0 ([nexp*D][F]); m* NULL without mins
    const int8_t *q0, *q1;
    const float *d0, *d1, *m0, *m1;
    int K;            // reduction length: D (gate/up) or F (down)
    int rows_e;       // rows per expert: F (gate/up) or D (down)
    int nexp;
    int is_shared;
    const int8_t *xq;  // activation codes: x_q [N][D] (gate/up) or h_q [entries][F] (down)
    const float *xd;
    int n_xrows;       // rows staged: N (gate/up, shared down) or N*top_k (routed down)
    const int32_t *expStart, *expTokI, *expTokK;
    int N, top_k;
    int8_t *h_q;       // gate/up outputs, rows by CSR entry (shared: by token)
    float *h_d;
    const float *shexp_scale;  // down: shared-expert scale per token
    float *out;                // down: partials [N*top_k][D] or shared rows [N][D]
    int D;
    int32_t *dbg_dots;
    int dbg_block;
    unsigned *status;
    int stages, stage_bytes, pairs_max;
};

__device__ __forceinline__ int dp4a4(int4 a, int4 b) {
    int s = __dp4a(a.x, b.x, 0);
    s = __dp4a(a.y, b.y, s);
    s = __dp4a(a.z, b.z, s);
    return __dp4a(a.w, b.w, s);
}

// Per-lane dots of two weight rows (quants w0/w1 [K], or [K/2] nibble-packed with PK; scales s0/s1
// [K/32], mins n0/n1 or NULL) with T staged activation rows tok[0..T-1] (xs [rows][K], xds
// [rows][K/32]); returns each lane's partial sums over its blocks (reduce_lanes adds them across
// the warp).  DBG: the lane owning block dbg_block keeps its isums in dbg.
template <int T, bool DBG, bool PK>
__device__ __forceinline__ void ring_dot(const int8_t *w0, const int8_t *w1, const float *s0, const float *s1,
                                         const float *n0, const float *n1, int K, const int8_t *xs, const float *xds,
                                         const int (&tok)[T], int lane, float (&acc)[2][T], int dbg_block,
                                         int (&dbg)[2][T]) {
    const int nblk = K / QK;
    const bool mins = n0 != nullptr;
#pragma unroll
    for (int tt = 0; tt < T; ++tt) acc[0][tt] = acc[1][tt] = 0.0f;
    constexpr int UNR = T <= 2 ? 2 : 1;  // register budget: two CTAs of 288 threads per SM
    // lane l reads the half (l >> 2) & 1 of its 32-byte block first: a quarter warp's 16-byte loads
    // then fall on eight different bank groups (the integer sums do not depend on the order)
    const int h = (lane >> 2) & 1;
#pragma unroll UNR
    for (int b = lane; b < nblk; b += 32) {
        int4 q0a, q0b, q1a, q1b;  // codes of the halves h and h ^ 1 of the block
        if (PK) {
            // one 16-byte load per row: low nibbles are codes 0-15, high nibbles codes 16-31
            const int4 v0 = reinterpret_cast<const int4 *>(w0)[b], v1 = reinterpret_cast<const int4 *>(w1)[b];
            const int4 l0 = make_int4(v0.x & 0x0F0F0F0F, v0.y & 0x0F0F0F0F, v0.z & 0x0F0F0F0F, v0.w & 0x0F0F0F0F);
            const int4 u0 = make_int4((v0.x >> 4) & 0x0F0F0F0F, (v0.y >> 4) & 0x0F0F0F0F, (v0.z >> 4) & 0x0F0F0F0F,
                                      (v0.w >> 4) & 0x0F0F0F0F);
            const int4 l1 = make_int4(v1.x & 0x0F0F0F0F, v1.y & 0x0F0F0F0F, v1.z & 0x0F0F0F0F, v1.w & 0x0F0F0F0F);
            const int4 u1 = make_int4((v1.x >> 4) & 0x0F0F0F0F, (v1.y >> 4) & 0x0F0F0F0F, (v1.z >> 4) & 0x0F0F0F0F,
                                      (v1.w >> 4) & 0x0F0F0F0F);
            q0a = h ? u0 : l0;
            q0b = h ? l0 : u0;
            q1a = h ? u1 : l1;
            q1b = h ? l1 : u1;
        } else {
            const int4 *p0 = reinterpret_cast<const int4 *>(w0 + b * QK),
                       *p1 = reinterpret_cast<const int4 *>(w1 + b * QK);
            q0a = p0[h];
            q0b = p0[h ^ 1];
            q1a = p1[h];
            q1b = p1[h ^ 1];
        }
        const float sc0 = s0[b], sc1 = s1[b];
        const float mn0 = mins ? n0[b] : 0.0f, mn1 = mins ? n1[b] : 0.0f;
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
            const int4 *px = reinterpret_cast<const int4 *>(xs + (size_t)tok[tt] * K + b * QK);
            const int4 xa = px[h], xb = px[h ^ 1];
            const float dx = xds[tok[tt] * nblk + b];
            int xsum = 0;
            if (mins) xsum = dp4a4(make_int4(0x01010101, 0x01010101, 0x01010101, 0x01010101), xa) +
                             dp4a4(make_int4(0x01010101, 0x01010101, 0x01010101, 0x01010101), xb);
            const int is0 = dp4a4(q0a, xa) + dp4a4(q0b, xb);
            const int is1 = dp4a4(q1a, xa) + dp4a4(q1b, xb);
            acc[0][tt] = fmaf(sc0 * dx, (float)is0, acc[0][tt]);
            if (mins) acc[0][tt] = fmaf(-(mn0 * dx), (float)xsum, acc[0][tt]);
            acc[1][tt] = fmaf(sc1 * dx, (float)is1, acc[1][tt]);
            if (mins) acc[1][tt] = fmaf(-(mn1 * dx), (float)xsum, acc[1][tt]);
            if (DBG && b == dbg_block) {
                dbg[0][tt] = is0;
                dbg[1][tt] = is1;
            }
        }
    }
}

// The warp sums of NV values (a power of two, 2..32) per lane, with the additions of warp_sum: at
// offset o every lane adds its own partial and lane (l ^ o)'s, so each sum is warp_sum's bit for
// bit.  At each of the first log2(NV) offsets (16, 8, ...) a lane keeps only half of its values
// (the lower half where bit o of its index is clear, the upper where set) and sends the other half,
// so NV - 1 shuffles do what NV warp_sums do with 5 NV.  Returns the full sum of value
// lane / (32 / NV), held by the 32 / NV lanes that share that quotient.
// One offset O of reduce_lanes with N values still per lane (compile-time throughout, so the
// values stay in registers).
template <int N, int O>
__device__ __forceinline__ void reduce_lanes_step(float *v, int lane) {
    if constexpr (O > 0) {
        if constexpr (N > 1) {
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float keep = upper ? v[i + N / 2] : v[i];
                const float send = upper ? v[i] : v[i + N / 2];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            reduce_lanes_step<N / 2, O / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            reduce_lanes_step<1, O / 2>(v, lane);
        }
    }
}

template <int NV>
__device__ __forceinline__ float reduce_lanes(float (&v)[NV], int lane) {
    static_assert(NV >= 1 && NV <= 32 && (NV & (NV - 1)) == 0, "a power of two");
    reduce_lanes_step<NV, 16>(v, lane);
    return v[0];
}

// The CSR entries of one work item, one slot per lane (lanes 0-7; other lanes hold dead slots):
// staged activation row (dead slots: row 0), h row / CSR entry, output row and scale.
struct Slot {
    int cnt;    // live slots of the item (<= RG_CHUNK), the same in every lane
    int row;
    int ent;    // gate/up: h row (CSR entry, or token for the shared expert); down: CSR entry; -1 dead
    int orow;   // down: output row
    float osc;  // down: shared-expert scale
};

// Slot tt of the work list's pair p (expert e, chunk ch), as stored in the slot table:
// (staged row, entry, output row, scale bits); dead slots have entry -1 and row 0.
template <int MODE>
__device__ __forceinline__ int4 make_slot(const RingArgs &a, int e, int ch, int tt, int *cnt_out) {
    int s0, s1;
    if (a.is_shared) {
        s0 = 0;
        s1 = a.N;
    } else {
        s0 = a.expStart[e];
        s1 = a.expStart[e + 1];
    }
    const int j0 = s0 + RG_CHUNK * ch;
    const int cnt = max(0, min(RG_CHUNK, s1 - j0));
    *cnt_out = cnt;
    int4 v = make_int4(0, -1, -1, __float_as_int(1.0f));
    if (tt < cnt) {
        const int j = j0 + tt;
        if (a.is_shared) {
            v = make_int4(j, j, j, __float_as_int(MODE == 1 ? a.shexp_scale[j] : 1.0f));
        } else {
            const int t = a.expTokI[j];
            const int sl = MODE == 1 ? a.expTokK[j] : 0;
            if ((unsigned)t < (unsigned)a.N && (unsigned)sl < (unsigned)a.top_k)
                v = make_int4(MODE == 0 ? t : j, j, t * a.top_k + sl, __float_as_int(1.0f));
            else
                atomicOr(a.status, MOE_DEV_BAD_CSR);
        }
    }
    return v;
}

__device__ __forceinline__ Slot load_slot(const int4 *slot_tab, const int *pair_cnt, int p, int lane) {
    Slot sl;
    sl.cnt = pair_cnt[p];
    int4 v = make_int4(0, -1, -1, __float_as_int(1.0f));
    if (lane < RG_CHUNK) v = slot_tab[p * RG_CHUNK + lane];
    sl.row = v.x;
    sl.ent = v.y;
    sl.orow = v.z;
    sl.osc = __int_as_float(v.w);
    return sl;
}

// One stage of one consumer warp: rows cw and cw + 8 of the stage against the item's T slots.
template <int MODE, int T, bool DBG, bool PK>
__device__ __forceinline__ void consume_stage(const RingArgs &a, const uint8_t *st, int cw, int lane, int ob, int s,
                                              const Slot &sl, const int8_t *xs, const float *xds, float *hbuf) {
    const int K = a.K, nblk = K / QK;
    const bool mins = a.m0 != nullptr;
    // stage: rows [16 x rb] (gate/up: 8 gate rows then 8 up rows; rb = K, or K/2 packed), scales
    // [16 x nblk], mins [16 x nblk]; this warp's rows are cw and cw + 8
    const int rb = PK ? K / 2 : K;
    const int8_t *w0 = reinterpret_cast<const int8_t *>(st) + (size_t)cw * rb;
    const int8_t *w1 = w0 + (size_t)8 * rb;
    const float *sc = reinterpret_cast<const float *>(st + (size_t)16 * rb);
    const float *s0 = sc + cw * nblk, *s1 = s0 + 8 * nblk;
    const float *n0 = mins ? s0 + 16 * nblk : nullptr, *n1 = mins ? s1 + 16 * nblk : nullptr;
    int tok[T];
#pragma unroll
    for (int tt = 0; tt < T; ++tt) tok[tt] = __shfl_sync(0xffffffffu, sl.row, tt);
    float acc[2][T];
    int dbg[2][T];
    ring_dot<T, DBG, PK>(w0, w1, s0, s1, n0, n1, K, xs, xds, tok, lane, acc, a.dbg_block, dbg);
    // the 2T sums (row m, slot tt) at index m * T + tt: lane l holds the sum of index l / (16 / T)
    float v[2 * T];
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
        v[tt] = acc[0][tt];
        v[T + tt] = acc[1][tt];
    }
    const float mine = reduce_lanes<2 * T>(v, lane);
    const int idx = lane / (16 / T);
    const int m = idx / T, tt = idx % T;         // m = lane's bit 4
    const bool first = (lane % (16 / T)) == 0;   // one lane of those holding the same sum
    // DBG: slot tt's two isums of block dbg_block, from the lane that owned the block
    int d0 = 0, d1 = 0;
    if (DBG) {
        const int src = a.dbg_block & 31;
#pragma unroll
        for (int u = 0; u < T; ++u) {
            const int g0 = __shfl_sync(0xffffffffu, dbg[0][u], src), g1 = __shfl_sync(0xffffffffu, dbg[1][u], src);
            if (lane == u) {
                d0 = g0;
                d1 = g1;
            }
        }
    }
    const bool live_own = lane < T && lane < sl.cnt && sl.ent >= 0;  // slot `lane`, for the DBG writes
    if (MODE == 0) {
        const int f = ob * QK + s * 8 + cw;  // feature within the expert
        if (DBG && live_own && a.dbg_block >= 0) {
            a.dbg_dots[((size_t)sl.ent * 2 + 0) * a.rows_e + f] = d0;
            a.dbg_dots[((size_t)sl.ent * 2 + 1) * a.rows_e + f] = d1;
        }
        const float up = __shfl_xor_sync(0xffffffffu, mine, 16);  // the same slot's up row sum
        if (m == 0 && first) {
            const float silu = mine / (1.0f + expf(-mine));
            hbuf[tt * QK + s * 8 + cw] = silu * up;
        }
    } else {
        const int c0 = ob * QK + s * 16 + cw;  // output columns c0 and c0 + 8
        if (DBG && live_own && !a.is_shared && a.dbg_block >= 0) {
            a.dbg_dots[(size_t)sl.ent * a.D + c0] = d0;
            a.dbg_dots[(size_t)sl.ent * a.D + c0 + 8] = d1;
        }
        // slot tt's output row, scale and liveness come from lane tt, which holds that slot
        const int orow = __shfl_sync(0xffffffffu, sl.orow, tt);
        const int ent = __shfl_sync(0xffffffffu, sl.ent, tt);
        const float osc = __shfl_sync(0xffffffffu, sl.osc, tt);
        if (first && tt < sl.cnt && ent >= 0 && orow >= 0)
            a.out[(size_t)orow * a.D + c0 + 8 * m] = a.is_shared ? osc * mine : mine;
    }
}

// The bulk copies of stage s of a work item whose first weight row is erow: gate/up 8 gate + 8 up
// rows (with scales, Q4_K mins), down 16 rows, completing on the mbarrier fb.  PK: rows of K/2
// packed bytes.
template <int MODE, bool PK>
__device__ __forceinline__ void issue_stage(const RingArgs &a, size_t erow, int s, uint32_t dst, uint32_t fb) {
    const int nblk = a.K / QK;
    const int K = PK ? a.K / 2 : a.K;  // bytes per weight row
    const bool mins = a.m0 != nullptr;
    const uint32_t sbytes = (uint32_t)(nblk * 4);
    if (MODE == 0) {
        const size_t r0 = erow + (size_t)s * 8;
        const uint32_t qb = (uint32_t)(8 * K), db = 8 * sbytes;
        mbar_expect_tx(fb, 2 * qb + 2 * db * (mins ? 2 : 1));
        bulk_load(dst, a.q0 + r0 * K, qb, fb);
        bulk_load(dst + qb, a.q1 + r0 * K, qb, fb);
        bulk_load(dst + 2 * qb, a.d0 + r0 * nblk, db, fb);
        bulk_load(dst + 2 * qb + db, a.d1 + r0 * nblk, db, fb);
        if (mins) {
            bulk_load(dst + 2 * qb + 2 * db, a.m0 + r0 * nblk, db, fb);
            bulk_load(dst + 2 * qb + 3 * db, a.m1 + r0 * nblk, db, fb);
        }
    } else {
        const size_t r0 = erow + (size_t)s * 16;
        const uint32_t qb = (uint32_t)(16 * K), db = 16 * sbytes;
        mbar_expect_tx(fb, qb + db * (mins ? 2 : 1));
        bulk_load(dst, a.q0 + r0 * K, qb, fb);
        bulk_load(dst + qb, a.d0 + r0 * nblk, db, fb);
        if (mins) bulk_load(dst + qb + db, a.m0 + r0 * nblk, db, fb);
    }
}

// Work list: (expert, chunk of 8 CSR entries) for every non-empty segment, in act[] (count in
// *n_pairs); the expert list comes from a launch before the previous one, so it is complete without
// the dependency wait.  Whole CTA (the consumer threads count the experts).
__device__ __forceinline__ void build_work_list(const RingArgs &a, int *act, int *warp_cnt, int *n_pairs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    {
        int base = 0;
        const int ct = threadIdx.x - 32;  // consumer threads count the experts
        for (int e0 = 0; e0 < (a.is_shared ? 1 : a.nexp); e0 += RG_CW * 32) {
            int nch = 0;
            const int e = e0 + ct;
            if (ct >= 0 && e < (a.is_shared ? 1 : a.nexp)) {
                int s0 = 0, s1 = a.N;
                if (!a.is_shared) {
                    s0 = a.expStart[e];
                    s1 = a.expStart[e + 1];
                    if (!(s0 >= 0 && s1 >= s0 && s1 <= a.N * a.top_k)) {
                        atomicOr(a.status, MOE_DEV_BAD_CSR);
                        s1 = s0 = 0;
                    }
                }
                nch = (s1 - s0 + RG_CHUNK - 1) / RG_CHUNK;
            }
            // block exclusive scan of nch over the consumer threads
            int incl = nch;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (warp >= 1 && lane == 31) warp_cnt[warp - 1] = incl;
            __syncthreads();
            int before = base;
            if (warp >= 1)
                for (int w = 0; w < warp - 1; ++w) before += warp_cnt[w];
            before += incl - nch;
            for (int c = 0; c < nch; ++c)
                if (before + c < a.pairs_max) act[before + c] = e | (c << RG_PAIR_SHIFT);
            for (int w = 0; w < RG_CW; ++w) base += warp_cnt[w];
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            if (base > a.pairs_max) atomicOr(a.status, MOE_DEV_BAD_CSR);  // overlapping segments
            *n_pairs = min(base, a.pairs_max);
        }
    }
}

// One work item of a consumer warp: its stages from the ring (stage counter k over the CTA's run),
// then on gate/up the requantisation by the warp that completes the item.  Returns false when a
// wait gave up.
template <int MODE, bool DBG, bool PK>
__device__ __forceinline__ bool consume_item(const RingArgs &a, int it, int ii, int &k, int S, int slot_bytes,
                                             const uint8_t *ring, uint64_t *full_bar, uint64_t *empty_bar,
                                             volatile int *abort_flag, const int4 *slot_tab, const int *pair_cnt,
                                             int *item_done, const int8_t *xs, const float *xds, float *hbuf, int cw,
                                             int lane) {
    const int nob = a.rows_e / QK;
    const int spi = MODE == 0 ? QK / 8 : QK / 16;  // stages per item
    const int ob = it % nob;
    const Slot sl = load_slot(slot_tab, pair_cnt, it / nob, lane);
    const int T = sl.cnt <= 1 ? 1 : sl.cnt <= 2 ? 2 : sl.cnt <= 4 ? 4 : 8;
    float *hb = hbuf + (ii % RG_HBUF) * RG_CHUNK * QK;
    for (int s = 0; s < spi; ++s, ++k) {
        const int slot = k % S;
        bool ok = mbar_wait(smem_u32(&full_bar[slot]), (k / S) & 1, abort_flag, a.status, RG_WAIT_NS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        const uint8_t *st = ring + (size_t)slot * slot_bytes;
        if (T == 1) consume_stage<MODE, 1, DBG, PK>(a, st, cw, lane, ob, s, sl, xs, xds, hb);
        else if (T == 2) consume_stage<MODE, 2, DBG, PK>(a, st, cw, lane, ob, s, sl, xs, xds, hb);
        else if (T == 4) consume_stage<MODE, 4, DBG, PK>(a, st, cw, lane, ob, s, sl, xs, xds, hb);
        else consume_stage<MODE, 8, DBG, PK>(a, st, cw, lane, ob, s, sl, xs, xds, hb);
        __syncwarp();
        if (MODE == 0 && s == spi - 1) {
            // the warp that completes the item requantises its 32 features per slot (the buffer is
            // reused three items later, after every warp has moved past this one)
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&item_done[ii % RG_HBUF], 1) == RG_CW - 1;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                if (lane == 0) item_done[ii % RG_HBUF] = 0;
                for (int tt = 0; tt < sl.cnt; ++tt) {
                    float d16f;
                    const int q = q8_quantize_lane(hb[tt * QK + lane], &d16f);
                    const int j = __shfl_sync(0xffffffffu, sl.ent, tt);
                    if (j >= 0) {
                        a.h_q[(size_t)j * a.rows_e + ob * QK + lane] = (int8_t)q;
                        if (lane == 0) a.h_d[(size_t)j * (a.rows_e / QK) + ob] = d16f;
                    }
                }
            }
        }
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
    }
    return true;
}

template <int MODE, bool DBG, bool PK>
__global__ void __launch_bounds__(RG_THREADS, 2)
matvec_ring_kernel(const RingArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[RG_MAX_STAGES], empty_bar[RG_MAX_STAGES];
    __shared__ int warp_cnt[RG_CW];
    __shared__ int n_pairs;
    __shared__ int item_done[RG_HBUF];
    __shared__ __align__(8) uint64_t x_bar;  // the staged activation rows have landed
    __shared__ volatile int abort_flag;

    const int K = a.K, nblk = K / QK;
    const int S = a.stages;
    uint8_t *ring = smem;
    int8_t *xs = reinterpret_cast<int8_t *>(smem + (size_t)S * a.stage_bytes);
    float *xds = reinterpret_cast<float *>(xs + (size_t)a.n_xrows * K);
    float *hbuf = xds + (size_t)a.n_xrows * nblk;        // [RG_HBUF][RG_CHUNK][32]
    int *act = reinterpret_cast<int *>(hbuf + RG_HBUF * RG_CHUNK * QK);               // [pairs_max]
    int4 *slot_tab = reinterpret_cast<int4 *>(act + ((a.pairs_max + 3) & ~3));         // [pairs_max][8]
    int *pair_cnt = reinterpret_cast<int *>(slot_tab + (size_t)a.pairs_max * RG_CHUNK);  // [pairs_max]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the launch that follows (down after gate/up, the combine after down) may be scheduled now:
    // it waits on the device for this one's output before reading it
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), RG_CW);
        }
        mbar_init(smem_u32(&x_bar), 1);
        for (int i = 0; i < RG_HBUF; ++i) item_done[i] = 0;
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    build_work_list(a, act, warp_cnt, &n_pairs);
    __syncthreads();
    const int nob = a.rows_e / QK;                    // 32-row output blocks per expert
    const int spi = MODE == 0 ? QK / 8 : QK / 16;     // stages per item
    const int n_items = n_pairs * nob;

    if (warp == 0) {
        // ------------------------------------------------------------ producer ---
        if (lane == 0) {
            uint32_t issued = 0, last_par = 0;
            int k = 0;
            bool ok = true, staged = false;
            // the batch's activation rows, once the ring is full: for the down launch they are the
            // previous launch's output, so the weights stream first
            auto stage_x = [&]() {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                const uint32_t xb = (uint32_t)(a.n_xrows * K), db = (uint32_t)(a.n_xrows * nblk * 4);
                mbar_expect_tx(smem_u32(&x_bar), xb + db);
                bulk_load(smem_u32(xs), a.xq, xb, smem_u32(&x_bar));
                bulk_load(smem_u32(xds), a.xd, db, smem_u32(&x_bar));
                staged = true;
            };
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const int e = act[it / nob] & ((1 << RG_PAIR_SHIFT) - 1), ob = it % nob;
                const size_t erow = (size_t)(a.is_shared ? 0 : e) * a.rows_e + (size_t)ob * QK;
                for (int s = 0; s < spi; ++s, ++k) {
                    const int slot = k % S;
                    if (k == S && !staged) stage_x();
                    if (k >= S && !mbar_wait(smem_u32(&empty_bar[slot]), ((k / S) - 1) & 1, &abort_flag, a.status,
                                             RG_WAIT_NS)) {
                        ok = false;
                        break;
                    }
                    issue_stage<MODE, PK>(a, erow, s, smem_u32(ring + (size_t)slot * a.stage_bytes),
                                      smem_u32(&full_bar[slot]));
                    issued |= 1u << slot;
                    last_par = (last_par & ~(1u << slot)) | ((uint32_t)((k / S) & 1) << slot);
                }
            }
            if (!staged && ok && (int)blockIdx.x < n_items) stage_x();
            // every CTA waits for the previous launch before it exits, so this launch's completion
            // implies that one's (the next launch relies on it through its own wait)
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // copies in flight land before the CTA exits (only an aborted run leaves any)
            if (staged) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try(smem_u32(&x_bar), 0) && globaltimer() - t0 < RG_WAIT_NS) {
                }
            }
            for (int s = 0; s < S; ++s)
                if (issued >> s & 1) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try(smem_u32(&full_bar[s]), last_par >> s & 1) && globaltimer() - t0 < RG_WAIT_NS) {
                    }
                }
        }
    } else {
        // ------------------------------------------------------------ consumers ---
        const int cw = warp - 1;
        // slot table of the work list (the CSR comes from a launch before the previous one)
        for (int i = threadIdx.x - 32; i < n_pairs * RG_CHUNK; i += RG_CW * 32) {
            const int p = i / RG_CHUNK, tt = i % RG_CHUNK;
            const int pr = act[p];
            int cnt;
            slot_tab[i] = make_slot<MODE>(a, pr & ((1 << RG_PAIR_SHIFT) - 1), pr >> RG_PAIR_SHIFT, tt, &cnt);
            if (tt == 0) pair_cnt[p] = cnt;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(RG_CW * 32) : "memory");
        int k = 0, ii = 0;
        bool ok = true;
        if ((int)blockIdx.x < n_items) {
            ok = mbar_wait(smem_u32(&x_bar), 0, &abort_flag, a.status, RG_WAIT_NS);
            ok = __all_sync(0xffffffffu, ok);
        }
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++ii)
            ok = consume_item<MODE, DBG, PK>(a, it, ii, k, S, a.stage_bytes, ring, full_bar, empty_bar, &abort_flag,
                                         slot_tab, pair_cnt, item_done, xs, xds, hbuf, cw, lane);
    }
    __syncthreads();
}


}  // namespace

// Ring geometry of one launch, or ok = false when the launch does not fit it (the register-loading
// kernels then serve it).  Two CTAs per SM when the staged rows leave room for two stages in half
// of the SM's shared memory, else one.
struct RingPlan {
    bool ok;
    int stages, stage_bytes, pairs_max;
    size_t smem;
};
static RingPlan ring_plan(int mode, int K, int rows_e, int n_xrows, int nexp, int entries, bool mins, bool pk) {
    RingPlan p{};
    if (K % 128 != 0 || rows_e % QK != 0 || nexp >= (1 << RG_PAIR_SHIFT)) return p;
    const int nblk = K / QK;
    const int srows = mode == 0 ? 16 : 16;  // rows per stage (gate/up: 8 of each matrix)
    p.stage_bytes = srows * (pk ? K / 2 : K) + srows * nblk * 4 * (mins ? 2 : 1);
    p.pairs_max = nexp + (entries + RG_CHUNK - 1) / RG_CHUNK;
    const size_t fixed = (size_t)n_xrows * K + (size_t)n_xrows * nblk * 4 + RG_HBUF * RG_CHUNK * QK * 4 +
                         (size_t)((p.pairs_max + 3) & ~3) * 4 + (size_t)p.pairs_max * (RG_CHUNK * 16 + 4) + 128;
    const size_t half = 110 * 1024, whole = 220 * 1024;
    size_t budget = fixed + 2 * (size_t)p.stage_bytes <= half ? half : whole;
    if (fixed + 2 * (size_t)p.stage_bytes > budget) return p;
    p.stages = (int)std::min<size_t>(RG_MAX_STAGES, (budget - fixed) / p.stage_bytes);
    p.smem = fixed + (size_t)p.stages * p.stage_bytes;
    p.ok = true;
    return p;
}

static int ring_grid(const void *kernel, size_t smem, int max_items) {
    const int n = device_sm_count();
    int per_sm = 0;
    if (n <= 0 || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, RG_THREADS, smem) != cudaSuccess ||
        per_sm <= 0)
        return -1;
    return std::max(1, std::min(n * per_sm, max_items));
}

template <int MODE, bool DBG, bool PK>
static int run_ring_k(const RingArgs &a, const RingPlan &pl, int max_items, cudaStream_t s, bool early) {
    static SmemOptIn configured;
    const void *k = (const void *)matvec_ring_kernel<MODE, DBG, PK>;
    if (int rc = ensure_dynamic_smem(k, pl.smem, &configured)) return rc;
    const int grid = ring_grid(k, pl.smem, max_items);
    if (grid < 0) return MOE_ERR_CUDA;
    if (early) return launch_early(matvec_ring_kernel<MODE, DBG, PK>, dim3(grid), dim3(RG_THREADS), pl.smem, s, a);
    matvec_ring_kernel<MODE, DBG, PK><<<grid, RG_THREADS, pl.smem, s>>>(a);
    return launch_status();
}

template <int MODE>
static int run_ring(const RingArgs &a, const RingPlan &pl, int max_items, cudaStream_t s, bool early, bool dbg,
                    bool pk) {
    if (pk)
        return dbg ? run_ring_k<MODE, true, true>(a, pl, max_items, s, early)
                   : run_ring_k<MODE, false, true>(a, pl, max_items, s, early);
    return dbg ? run_ring_k<MODE, true, false>(a, pl, max_items, s, early)
               : run_ring_k<MODE, false, false>(a, pl, max_items, s, early);
}

bool matvec_ring_eligible(int N, int K, int rows_e, int n_xrows, int nexp, int entries, bool mins, const void *xq,
                          const void *xd, const WeightSet &set) {
    // bulk copies: 16-byte aligned addresses (the spans' sizes are multiples of 16 once K % 128 == 0)
    const void *ptrs[] = {xq, xd, set.gate_q, set.up_q, set.down_q, set.gate_d, set.up_d, set.down_d,
                          set.gate_m, set.up_m, set.down_m, set.gate_p, set.up_p, set.down_p};
    for (const void *q : ptrs)
        if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return false;
    return N <= RG_CHUNK && ring_plan(0, K, rows_e, n_xrows, nexp, entries, mins, set.gate_p != nullptr).ok;
}

int launch_matvec_ring_gate_up(const WeightSet &set, int D, int F, int nexp, bool is_shared, const int8_t *x_q,
                               const float *x_d, const int32_t *expStart, const int32_t *expTokI, int N, int top_k,
                               int8_t *h_q, float *h_d, int32_t *dbg_dots, int dbg_block, unsigned *status,
                               cudaStream_t s) {
    const bool mins = set.gate_m != nullptr, pk = set.gate_p != nullptr;
    const RingPlan pl = ring_plan(0, D, F, N, nexp, is_shared ? N : N * top_k, mins, pk);
    if (!pl.ok) return MOE_ERR_UNSUPPORTED_SHAPE;
    RingArgs a{};
    a.q0 = pk ? reinterpret_cast<const int8_t *>(set.gate_p) : set.gate_q;
    a.q1 = pk ? reinterpret_cast<const int8_t *>(set.up_p) : set.up_q;
    a.d0 = set.gate_d;
    a.d1 = set.up_d;
    a.m0 = set.gate_m;
    a.m1 = set.up_m;
    a.K = D;
    a.rows_e = F;
    a.nexp = nexp;
    a.is_shared = is_shared ? 1 : 0;
    a.xq = x_q;
    a.xd = x_d;
    a.n_xrows = N;
    a.expStart = expStart;
    a.expTokI = expTokI;
    a.N = N;
    a.top_k = top_k;
    a.h_q = h_q;
    a.h_d = h_d;
    a.D = D;
    a.dbg_dots = dbg_dots;
    a.dbg_block = dbg_block;
    a.status = status;
    a.stages = pl.stages;
    a.stage_bytes = pl.stage_bytes;
    a.pairs_max = pl.pairs_max;
    return run_ring<0>(a, pl, pl.pairs_max * (F / QK), s, false, dbg_dots != nullptr, pk);
}

int launch_matvec_ring_down(const WeightSet &set, int D, int F, int nexp, bool is_shared, const int8_t *h_q,
                            const float *h_d, const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                            int N, int top_k, const float *shexp_scale, float *out, unsigned *status, cudaStream_t s,
                            bool early, int32_t *dbg_dots, int dbg_block) {
    const bool mins = set.down_m != nullptr, pk = set.down_p != nullptr;
    const int rows = is_shared ? N : N * top_k;
    const RingPlan pl = ring_plan(1, F, D, rows, nexp, rows, mins, pk);
    if (!pl.ok) return MOE_ERR_UNSUPPORTED_SHAPE;
    RingArgs a{};
    a.q0 = pk ? reinterpret_cast<const int8_t *>(set.down_p) : set.down_q;
    a.d0 = set.down_d;
    a.m0 = set.down_m;
    a.K = F;
    a.rows_e = D;
    a.nexp = nexp;
    a.is_shared = is_shared ? 1 : 0;
    a.xq = h_q;
    a.xd = h_d;
    a.n_xrows = rows;
    a.expStart = expStart;
    a.expTokI = expTokI;
    a.expTokK = expTokK;
    a.N = N;
    a.top_k = top_k;
    a.shexp_scale = shexp_scale;
    a.out = out;
    a.D = D;
    a.dbg_dots = dbg_dots;
    a.dbg_block = dbg_block;
    a.status = status;
    a.stages = pl.stages;
    a.stage_bytes = pl.stage_bytes;
    a.pairs_max = pl.pairs_max;
    return run_ring<1>(a, pl, pl.pairs_max * (D / QK), s, early, dbg_dots != nullptr, pk);
}


}  // namespace moe
