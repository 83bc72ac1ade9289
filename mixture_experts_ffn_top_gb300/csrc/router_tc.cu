// router_tc.cu -- the router of a prefill batch on the 5th-generation tensor cores, with the
// Q8_1 quantisation of the hidden rows and the per-token softmax / top-k in the same launch
// ("Carnice prefill toward llama.cpp 676 t/s", #388: breakdown table "router" row -- matvec +
// softmax + top-k + shexp-gate -- and "Remaining levers" item 1, which moves it onto the GPU).
//
// logits = hidden . routerW^T is a dense fp32 contraction (N x D by D x E).  The tensor cores read
// fp32 operands as tf32 (10 explicit mantissa bits), so every operand x is split into hi = x with
// its low 13 mantissa bits cleared and lo = (x - hi) cut the same way (x - hi is exact in fp32), and
// each K step issues three kind::tf32 MMAs, hi*hi + hi*lo + lo*hi, into one fp32 accumulator in
// tensor memory (N = E <= 256): every product is exact and the dropped lo*lo term and the cut of lo
// are below 2^-20 of |x*w|, so the logits carry fp32-level error (the fp32 SIMT router's within
// its tolerance of the oracle).  The shared gate g_t = x_t . w_sg (one more column) is formed on
// the CUDA cores by the threads that already hold x_t's values (fp32 fused multiply-adds).
//
// Grid: one thread-block cluster of KS CTAs per 128-token tile; CTA r of a cluster takes the K
// range [r, r + 1) * D / KS.  Per 32-wide K block the producer loads the token tile [128 x 32] and
// the router tile [E x 32] by TMA into a ring as deep as shared memory allows (stages of 48-96 KB);
// two groups of eight converter warps take alternate K blocks: they quantise the token rows (each
// 32-wide row is one Q8_1 block: the same rule as the SIMT router, so x_q and x_d are identical),
// accumulate the gate dot and split both tiles into hi / lo in place; one thread issues the MMAs.
// At the end every CTA leaves its partial logits [128 x (E + 1)] in shared memory, the cluster
// meets at a barrier, and CTA r sums the KS partials of its 128 / KS tokens in split order through
// distributed shared memory and routes them (route_token, the SIMT router's arithmetic).  No
// partial leaves the chip and no second launch is needed.
//
// Every mbarrier wait is bounded (MOE_DEV_TIMEOUT; every role then drains out, waits bounded for
// its copies and MMAs, and still meets the cluster barriers, which every thread reaches).
#include <cuda.h>

#include <algorithm>

#include "moe_internal.cuh"
#include "tc_glue.cuh"
#include "topk_token.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int RT_M = 128;                        // tokens per tile (MMA M)
constexpr int RT_MAX_N = 256;                    // router rows (experts) per tile: the MMA's N
constexpr int RT_MAX_STAGES = 6;
constexpr int RT_CONV_WARPS = 8;                 // per converter group: two threads per tile row
constexpr int RT_THREADS = 32 * (2 + 2 * RT_CONV_WARPS);  // warp 0 TMA, warp 1 MMA + TMEM, 2-17 convert
                                                          // (two groups, alternate K blocks; 2-5 drain), all route
constexpr int RT_A = RT_M * 128;                 // token tile: 128 rows x 32 fp32
constexpr int RT_SMEM_MAX = 220 * 1024;          // dynamic shared memory of one CTA at most (the
                                                 // static barriers and gate partials fit beside it)
constexpr int RT_TMEM_COLS = 256;
constexpr int RT_MAX_KS = 8;
constexpr unsigned long long RT_WAIT_NS = 2000000000ull;
// Shared memory of a launch: the stage ring (stage = token tile hi + lo, router tile hi + lo, as many
// stages as fit, at most RT_MAX_STAGES), reused after the main loop for the partial logits
// [128][E + 1] and the summed logits of this CTA's tokens [128 / KS][E + 1]; the gate slice of the
// CTA's K range stays apart.
// The MMA's N: E rounded up to a multiple of 16 (the router tile's extra rows are zero).
__host__ __device__ constexpr int rt_nmma(int E) { return (E + 15) & ~15; }
__host__ __device__ constexpr int rt_stage_bytes(int E) { return 2 * RT_A + 2 * rt_nmma(E) * 128; }
__host__ __device__ constexpr int rt_gate_bytes(int D) { return D * 4; }
__host__ __device__ inline int rt_stages(int E, int D) {
    const int s = (RT_SMEM_MAX - 1024 - rt_gate_bytes(D)) / rt_stage_bytes(E);
    return s < RT_MAX_STAGES ? s : RT_MAX_STAGES;
}
__host__ __device__ inline int rt_tail_bytes(int E, int ks) {
    return (RT_M * (E + 1) + 32 + (RT_M / ks) * (E + 1) + 32 + E) * 4;
}

struct RtMaps {
    CUtensorMap x, w;  // hidden [N][D], routerW [E][D] (boxes of 32 fp32)
};
struct RtParams {
    int N, D, E, ks, kb_per, top_k, norm, has_gate, stages;
    const float *gate_w;  // the shared gate vector [D] (has_gate)
    int *tile_counts;     // nullable: per token tile, how many of its routing entries chose each expert
                          // ([tiles][E], then [tiles] zero flags: the bucketing kernel's count table)
    int8_t *x_q;
    float *x_d;
    int32_t *topk_idx;
    float *topk_w;
    float *shexp_scale;
    float *logits_out;
    unsigned *status;
};

// kind::tf32 instruction descriptor: D fp32, A and B tf32, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_tf32(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// One warp reads 32 TMEM lanes x 16 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// A float of CTA `rank`'s shared memory at this CTA's address local_addr.  Not volatile: the loads
// of one logit's partials may all be in flight at once (they follow the cluster barrier, an asm
// with a memory clobber, which they cannot move above).
__device__ __forceinline__ float ld_cluster(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
    return v;
}
__device__ __forceinline__ uint32_t tf32_hi_bits(uint32_t u) { return u & 0xffffe000u; }
// Asks L2 for one TMA box of the map at (x, y): a hint with no completion to wait for.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Splits the half h of a 128-byte row of 32 fp32 (its 16-byte chunks 4h .. 4h + 3, swizzled) into
// hi (in place) and lo.
__device__ __forceinline__ void split_half(uint8_t *hi_row, uint8_t *lo_row, const float4 (&v)[4], int sw, int h) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int off = ((4 * h + j) ^ sw) << 4;
        const float x[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t hb[4], lb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hb[i] = tf32_hi_bits(__float_as_uint(x[i]));
            lb[i] = tf32_hi_bits(__float_as_uint(__fsub_rn(x[i], __uint_as_float(hb[i]))));
        }
        *reinterpret_cast<uint4 *>(hi_row + off) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
        *reinterpret_cast<uint4 *>(lo_row + off) = make_uint4(lb[0], lb[1], lb[2], lb[3]);
    }
}

template <int EPL>
__global__ void __launch_bounds__(RT_THREADS, 1)
router_tc_kernel(const __grid_constant__ RtMaps maps, const RtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t full_bar[RT_MAX_STAGES], conv_bar[RT_MAX_STAGES], empty_bar[RT_MAX_STAGES];
    __shared__ __align__(8) uint64_t acc_bar, done_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    __shared__ float gpart[2][RT_M][2];  // the shared gate's partial dots: [group][row][half]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_rank();
    const int tile = blockIdx.y;
    const int t0 = tile * RT_M;
    const int kb0 = rank * p.kb_per;
    const int nblk = p.D / QK;
    const int S = p.stages;
    const int SB = rt_stage_bytes(p.E);      // stage: [A hi][A lo][B hi][B lo]
    const int NM = rt_nmma(p.E);
    const int B_BYTES = NM * 128;  // a router tile on chip: NM rows of 32 fp32, E of them loaded
    float *gw = reinterpret_cast<float *>(smem + S * SB);  // gate weights of this K range

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&conv_bar[s]), RT_CONV_WARPS);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&acc_bar), 1);
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the shared gate's slice of this K range (a weight: it does not depend on the previous launch)
    if (p.has_gate)
        for (int i = threadIdx.x; i < p.kb_per * QK; i += RT_THREADS) gw[i] = p.gate_w[kb0 * QK + i];
    if (warp == 0 && lane == 0) {
        prefetch_map(&maps.x);
        prefetch_map(&maps.w);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(RT_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (p.E < NM) {
        // the router tile's rows E .. NM-1 (hi and lo) are zero in every stage: no copy writes them
        for (int st = 0; st < S; ++st) {
            float *bh = reinterpret_cast<float *>(smem + st * SB + 2 * RT_A);
            for (int i = threadIdx.x; i < (NM - p.E) * 32; i += RT_THREADS) {
                bh[p.E * 32 + i] = 0.0f;
                bh[NM * 32 + p.E * 32 + i] = 0.0f;
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tensor core reads them
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer ---
        if (lane == 0) {
            // the router rows of this K range beyond the ring's first fill do not depend on the
            // previous launch: ask L2 for them (hidden may be that launch's output: a chain of layers)
            for (int i = S; i < p.kb_per; ++i) tma_prefetch_2d(&maps.w, (kb0 + i) * QK, 0);
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t issued = 0, last_par = 0;
            for (int i = 0; i < p.kb_per; ++i) {
                const int s = i % S;
                if (i >= S && !mbar_wait(smem_u32(&empty_bar[s]), ((i / S) - 1) & 1, &abort_flag, p.status, RT_WAIT_NS))
                    break;
                uint8_t *st = smem + s * SB;
                const uint32_t fb = smem_u32(&full_bar[s]);
                const int k0 = (kb0 + i) * QK;
                mbar_expect_tx(fb, RT_A + p.E * 128);
                tma_load_2d(smem_u32(st), &maps.x, k0, t0, fb);
                tma_load_2d(smem_u32(st + 2 * RT_A), &maps.w, k0, 0, fb);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | ((uint32_t)((i / S) & 1) << s);
            }
            for (int s = 0; s < S; ++s)
                if (issued >> s & 1) {
                    const uint64_t tw = globaltimer();
                    while (!mbar_try(smem_u32(&full_bar[s]), last_par >> s & 1) && globaltimer() - tw < RT_WAIT_NS) {
                    }
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA ---
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(NM);
            bool ok = true;
            int i = 0;
            for (; i < p.kb_per; ++i) {
                const int s = i % S;
                ok = mbar_wait(smem_u32(&conv_bar[s]), (i / S) & 1, &abort_flag, p.status, RT_WAIT_NS);
                if (!ok) break;
                tc_fence_after();
                // descriptors of the four tiles; K step k starts 32 bytes further (2 in the
                // descriptor's 16-byte address field)
                const uint64_t ah = smem_desc_sw128(smem_u32(smem + s * SB));
                const uint64_t al = ah + (RT_A >> 4), bh = ah + ((2 * RT_A) >> 4), bl = bh + (B_BYTES >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // K = 8 tf32 (32 bytes) per MMA
                    mma_tf32(tmem, ah + 2 * k, bh + 2 * k, idesc, (i | k) != 0);
                    mma_tf32(tmem, ah + 2 * k, bl + 2 * k, idesc, 1);
                    mma_tf32(tmem, al + 2 * k, bh + 2 * k, idesc, 1);
                }
                mma_commit(smem_u32(&empty_bar[s]));
            }
            (void)ok;  // an abort has raised abort_flag: the drain skips the accumulator
            mma_commit(smem_u32(&acc_bar));
            // every MMA issued has completed once this commit arrives
            mma_commit(smem_u32(&done_bar));
            const uint64_t tw = globaltimer();
            while (!mbar_try(smem_u32(&done_bar), 0) && globaltimer() - tw < RT_WAIT_NS) {
            }
        }
    } else {
        // ------------------------------------------------- convert, then drain ---
        // two groups of eight warps take alternate K blocks; in a group, two threads per tile row:
        // thread (r, h) takes the 16-byte chunks 4h .. 4h + 3 of token row r (its Q8_1, its hi / lo
        // split, and its shared-gate dot on the CUDA cores) and of router rows r and r + 128 (< E)
        const int grp = (warp - 2) / RT_CONV_WARPS;
        const int ci = threadIdx.x - 64 - grp * RT_CONV_WARPS * 32;
        const int r = ci >> 1, h = ci & 1;
        const int t = t0 + r;
        const int sw = r & 7;  // 128-byte swizzle: chunk j of row r sits at chunk j ^ (r % 8)
        float gacc = 0.0f;     // shared-gate dot of this row's half over this group's K blocks
        bool ok = true;
        for (int i = grp; i < p.kb_per; i += 2) {
            const int s = i % S;
            ok = mbar_wait(smem_u32(&full_bar[s]), (i / S) & 1, &abort_flag, p.status, RT_WAIT_NS);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            uint8_t *st = smem + s * SB;
            uint32_t qw[4];
            float d16;
            {
                uint8_t *row = st + r * 128;
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const float4 *>(row + (((4 * h + j) ^ sw) << 4));
                // Q8_1 of this token's block kb0 + i (the rule of the SIMT router); the row's
                // maximum from both halves
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v[j].x)), fmaxf(fabsf(v[j].y), fabsf(v[j].z))), fabsf(v[j].w));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                const float d = __fdiv_rn(amax, 127.0f);
                const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int q0 = (int)roundf(__fmul_rn(v[j].x, id)), q1 = (int)roundf(__fmul_rn(v[j].y, id));
                    const int q2 = (int)roundf(__fmul_rn(v[j].z, id)), q3 = (int)roundf(__fmul_rn(v[j].w, id));
                    qw[j] = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) | ((uint32_t)(q2 & 0xff) << 16) |
                            ((uint32_t)(q3 & 0xff) << 24);
                }
                d16 = __half2float(__float2half_rn(d));
                if (p.has_gate) {
                    // K positions 16h .. 16h + 15 of this block, in order
                    const float *g = gw + i * QK + 16 * h;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        gacc = fmaf(v[j].x, g[4 * j + 0], gacc);
                        gacc = fmaf(v[j].y, g[4 * j + 1], gacc);
                        gacc = fmaf(v[j].z, g[4 * j + 2], gacc);
                        gacc = fmaf(v[j].w, g[4 * j + 3], gacc);
                    }
                }
                split_half(row, st + RT_A + r * 128, v, sw, h);
            }
#pragma unroll
            for (int rb = r; rb < r + RT_M + 1; rb += RT_M) {  // router rows r and r + 128
                if (rb >= p.E) break;
                uint8_t *row = st + 2 * RT_A + rb * 128;
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const float4 *>(row + (((4 * h + j) ^ sw) << 4));
                split_half(row, st + 2 * RT_A + B_BYTES + rb * 128, v, sw, h);
            }
            // the tensor core reads these through the async proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&conv_bar[s]));
            // the Q8_1 codes and scale leave after the hand-over (the proxy fence need not wait for them)
            if (t < p.N) {
                const int kb = kb0 + i;
                *reinterpret_cast<int4 *>(p.x_q + (size_t)t * p.D + (size_t)kb * QK + 16 * h) =
                    make_int4((int)qw[0], (int)qw[1], (int)qw[2], (int)qw[3]);
                if (h == 0) p.x_d[(size_t)t * nblk + kb] = d16;
            }
        }
        gpart[grp][r][h] = gacc;
        // partial logits of this K range: warps 2-5, one TMEM lane quarter each -> shared [128][E + 1],
        // column E the shared gate's partial (the four partial dots of the row in a fixed order)
        if (warp < 6) {
            if (ok) ok = mbar_wait(smem_u32(&acc_bar), 0, &abort_flag, p.status, RT_WAIT_NS);
            ok = __all_sync(0xffffffffu, ok) && !abort_flag;
            if (ok) {
                tc_fence_after();
                const int q = warp & 3;
                const int rr = q * 32 + lane;
                float *P = reinterpret_cast<float *>(smem);
                for (int c0 = 0; c0 < p.E; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < p.E) P[rr * (p.E + 1) + c0 + j] = __uint_as_float(v[j]);
                }
            }
        }
    }
    __syncthreads();  // the gate partials of both groups are in place
    if (warp >= 2 && warp < 6 && p.has_gate && !abort_flag) {
        const int rr = (warp & 3) * 32 + lane;
        reinterpret_cast<float *>(smem)[rr * (p.E + 1) + p.E] =
            __fadd_rn(__fadd_rn(gpart[0][rr][0], gpart[0][rr][1]), __fadd_rn(gpart[1][rr][0], gpart[1][rr][1]));
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // every CTA's partials are in its shared memory
    // ----------------------------------------------- reduce across the cluster and route ---
    // this CTA's 128 / KS tokens: their partial rows from every CTA of the cluster, summed in split
    // order into local shared memory (all loads of a thread in flight together), then one warp per
    // token routes from there
    const int per = RT_M / p.ks;
    const int ext = p.E + (p.has_gate ? 1 : 0);
    const int stride = p.E + 1;
    float *Lsum = reinterpret_cast<float *>(smem) + ((RT_M * stride + 31) & ~31);  // [per][ext]
    if (!abort_flag) {
        const uint32_t pbase = smem_u32(smem);
        for (int i = threadIdx.x; i < per * ext; i += RT_THREADS) {
            const int tr = rank * per + i / ext, e = i % ext;
            const uint32_t a = pbase + (uint32_t)((tr * stride + e) * 4);
            float part[RT_MAX_KS];
#pragma unroll
            for (int q = 0; q < RT_MAX_KS; ++q) part[q] = q < p.ks ? ld_cluster(a, q) : 0.0f;
            float v = part[0];
#pragma unroll
            for (int q = 1; q < RT_MAX_KS; ++q)
                if (q < p.ks) v = __fadd_rn(v, part[q]);
            Lsum[i] = v;
        }
    }
    __syncthreads();
    if (!abort_flag) {
        for (int tl = warp; tl < per; tl += RT_THREADS / 32) {
            const int t = t0 + rank * per + tl;
            if (t >= p.N) break;
            const float *row = Lsum + tl * ext;
            auto logit = [&](int e) { return row[e]; };
            auto gate = [&]() { return row[p.E]; };
            route_token<EPL>(logit, gate, p.E, p.top_k, p.norm, t, lane, p.topk_idx, p.topk_w,
                             p.has_gate ? p.shexp_scale : nullptr, p.logits_out);
        }
    }
    if (p.tile_counts != nullptr) {
        // this tile's expert histogram (the bucketing kernel's count table row): every CTA counts
        // the entries of its own tokens, CTA 0 of the cluster adds the KS counts
        int *hist = reinterpret_cast<int *>(Lsum + ((per * ext + 31) & ~31));
        for (int e = threadIdx.x; e < p.E; e += RT_THREADS) hist[e] = 0;
        __syncthreads();  // the routing's stores (this CTA's) are visible to it past the barrier
        const int tb = t0 + rank * per, te = min(p.N, tb + per);
        for (int i = threadIdx.x; i < (te - tb) * p.top_k; i += RT_THREADS) {
            const int e = p.topk_idx[(size_t)tb * p.top_k + i];
            if ((unsigned)e < (unsigned)p.E) atomicAdd(&hist[e], 1);
        }
    }
    cluster_sync();  // no CTA leaves while another still reads its partials (or its counts)
    if (p.tile_counts != nullptr) {
        if (rank == 0) {
            int *hist = reinterpret_cast<int *>(Lsum + ((per * ext + 31) & ~31));
            const uint32_t hb = smem_u32(hist);
            for (int e = threadIdx.x; e < p.E; e += RT_THREADS) {
                int c = 0;
                for (int q = 0; q < p.ks; ++q) c += __float_as_int(ld_cluster(hb + 4 * e, q));
                p.tile_counts[(size_t)tile * p.E + e] = c;
            }
            if (threadIdx.x == 0) p.tile_counts[(size_t)gridDim.y * p.E + tile] = 0;  // no bad entries
        }
        cluster_sync();  // CTA 0 has read every CTA's counts
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(RT_TMEM_COLS)
                     : "memory");
    }
}

// The K split (= cluster size) of a launch: the largest of 8, 4, 2, 1 that divides D/32 and lets
// every token tile's cluster be resident at once (the device's limit on active clusters of that
// size, queried once per device); when none does, the largest that divides D/32.  0 when the
// device cannot hold even one cluster (nothing is launched then).
template <int EPL>
int pick_ks(int tiles, int D) {
    static int maxc[MAX_DEVICES][RT_MAX_KS + 1];  // 0 unknown, else active clusters + 1
    const int dev = current_device();
    if (dev < 0) return 0;
    int best = 0;
    for (int ks = RT_MAX_KS; ks >= 1; ks >>= 1) {
        if ((D / QK) % ks != 0) continue;
        if (maxc[dev][ks] == 0) {
            cudaLaunchConfig_t q{};
            q.gridDim = dim3(ks, 1);
            q.blockDim = dim3(RT_THREADS);
            q.dynamicSmemBytes = RT_SMEM_MAX;  // every launch's size or less
            cudaLaunchAttribute ca[1];
            ca[0].id = cudaLaunchAttributeClusterDimension;
            ca[0].val.clusterDim.x = ks;
            ca[0].val.clusterDim.y = 1;
            ca[0].val.clusterDim.z = 1;
            q.attrs = ca;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, (const void *)router_tc_kernel<EPL>, &q) != cudaSuccess) n = 0;
            cudaGetLastError();
            maxc[dev][ks] = n + 1;
        }
        const int n = maxc[dev][ks] - 1;
        if (n <= 0) continue;
        if (best == 0) best = ks;          // fallback: the largest that divides and fits at all
        if (tiles <= n) return ks;         // one wave
    }
    return best;
}

// MOE_ERR_UNSUPPORTED_SHAPE (nothing launched) when the device cannot hold one cluster.
template <int EPL>
int launch_tc(const RtMaps &maps, RtParams p, int tiles, cudaStream_t s, bool early) {
    static SmemOptIn configured;
    if (int rc = ensure_dynamic_smem((const void *)router_tc_kernel<EPL>, RT_SMEM_MAX, &configured)) return rc;
    p.ks = pick_ks<EPL>(tiles, p.D);
    if (p.ks == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    p.kb_per = p.D / QK / p.ks;
    p.stages = rt_stages(p.E, p.D);
    const size_t ring = (size_t)p.stages * rt_stage_bytes(p.E) + rt_gate_bytes(p.D);
    const size_t smem = 1024 + std::max(ring, (size_t)rt_tail_bytes(p.E, p.ks));
    if (p.stages < 2 || smem > (size_t)RT_SMEM_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.ks, tiles);
    cfg.blockDim = dim3(RT_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 2 : 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, router_tc_kernel<EPL>, maps, p));
}

}  // namespace

bool router_tc_eligible(int N, int D, int E, bool has_gate, const float *hidden, const float *routerW,
                        const float *shexp_gate) {
    const uintptr_t al = reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(routerW) |
                         (has_gate ? reinterpret_cast<uintptr_t>(shexp_gate) : 0);
    return N > 8 && E % 8 == 0 && E >= 8 && E <= RT_MAX_N && D % QK == 0 && al % 16 == 0 && rt_stages(E, D) >= 2;
}

int launch_router_tc(const float *hidden, const float *routerW, const float *shexp_gate, int N, int D, int E,
                     int top_k, int norm, int32_t *topk_idx, float *topk_w, float *shexp_scale, int8_t *x_q,
                     float *x_d, float *logits_out, unsigned *status, cudaStream_t s, bool early, int *tile_counts) {
    RtMaps maps;
    RtParams p{};
    p.N = N;
    p.D = D;
    p.E = E;
    p.has_gate = shexp_gate != nullptr;
    p.gate_w = shexp_gate;
    p.top_k = top_k;
    p.norm = norm;
    p.x_q = x_q;
    p.x_d = x_d;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.shexp_scale = shexp_scale;
    p.logits_out = logits_out;
    p.status = status;
    p.tile_counts = tile_counts;
    if (!encode_fp32_sw128_2d(&maps.x, hidden, N, D, RT_M) || !encode_fp32_sw128_2d(&maps.w, routerW, E, D, E))
        return MOE_ERR_CUDA;
    const int tiles = (N + RT_M - 1) / RT_M;
    if (E <= 32) return launch_tc<1>(maps, p, tiles, s, early);
    if (E <= 64) return launch_tc<2>(maps, p, tiles, s, early);
    if (E <= 128) return launch_tc<4>(maps, p, tiles, s, early);
    return launch_tc<8>(maps, p, tiles, s, early);
}

}  // namespace moe
