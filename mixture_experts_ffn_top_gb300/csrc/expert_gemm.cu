// expert_gemm.cu -- grouped expert GEMM on the 5th-generation tensor cores.
//
// One persistent launch covers every expert's CSR segment (the grouped /
// segmented GEMM of "Carnice prefill toward llama.cpp 676 t/s", #388, lever
// 3, replacing one launch per expert; gather -> GEMM-N -> scatter of "batched
// int8-MMQ trunk prefill gated off for MoE", #406, "The work" item 2).
//
// Arithmetic.  The Q8_0 x Q8_1 dot of a weight row and an activation row is
// sum_b d_w[b] * d_x[b] * isum_b with isum_b the int32 dot of block b's quants.
// tcgen05 has no int8 MMA on sm_103a, but every int8 quant (|q| <= 127) is an
// exact fp16 value, every product (<= 16129) and every 32-term block sum
// (<= 516128 < 2^24) is exact in the fp32 accumulator.  So a kind::f16 MMA
// over exactly one 32-wide block, started from zero, yields isum_b exactly.
// Each block therefore gets its own accumulator in tensor memory (TMEM); the
// drain warps read it (tcgen05.ld), scale it by d_w (per TMEM lane = weight
// row) * d_x (per column = token) and accumulate in registers.
//
// Roles (512 threads, one CTA per SM, persistent over work items):
//   warp 0      TMA producer: per stage (64 K = 2 blocks) the weight tile
//               [128 rows x 64] fp16 and the token tile [nb rows x 64] fp16
//               (nb = 16/32/64/96, the smallest box that holds the tile's
//               rows) into the 5-slot tile ring, both tiles' block scales into
//               the 8-slot scale ring, one mbarrier per stage.
//   warp 1      TMEM owner and MMA issuer: 2 x (M128 x N x K16) per block into
//               one of 5 TMEM accumulators of 96 columns; one commit per stage
//               both releases the tile-ring slot and tells the drain the stage's
//               accumulators are complete.  It starts a
//               stage when the orchestrator's stage count (a shared word it
//               polls) says so.
//   warps 2-13  drain, 3 per SM sub-partition: warp w reads TMEM lanes
//               32*(w%4).. (the hardware's lane-quarter rule) and token
//               columns 32*((w-2)/4) + [0, 32).  Per stage one wait for the
//               second block's commit, both TMEM loads, the two slots handed
//               back, then the scale math of both blocks on packed f32x2 math.
//               At the end of an item the fp32 accumulators go to a shared
//               hand-off buffer.
//   warp 14     orchestrator: waits for a stage's copies and for the drain to
//               hand back the TMEM slots the stage will write, then publishes
//               the stage count to the MMA warp.
//   warp 15     epilogue: finishes each item from the hand-off buffer while the
//               drain moves on.  Gate/up tiles hold 64 gate rows and the 64 up
//               rows of the same features (weights repacked that way): one lane
//               per (token column, 32-feature block) forms h = SiLU(g) * u,
//               requantises it to Q8_1 and stores 32 fp16 codes; down tiles
//               store fp32 rows to partials[t*top_k + slot] (or s_t * y to the
//               shared expert's output).
// Every wait on an mbarrier is bounded (a few seconds); on expiry the CTA sets
// MOE_DEV_TIMEOUT in the status word, every role drains out, in-flight copies
// and MMAs are waited for (bounded) and TMEM is freed before returning.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "moe_internal.cuh"
#include "tc_glue.cuh"
#include "gemm_common.cuh"

namespace moe {

namespace {

using namespace tc;
using namespace gemm;

constexpr int G_DRAIN_WARPS = 12;                 // 3 per SM sub-partition (128 registers each)
constexpr int G_ORCH_WARP = 2 + G_DRAIN_WARPS;    // warp that tells the MMA warp when a stage may go
constexpr int G_EPI_WARP = 3 + G_DRAIN_WARPS;     // warp that finishes each item from the hand-off buffer
constexpr int G_THREADS = 128 + 32 * G_DRAIN_WARPS; // producer, MMA, drain warps, orchestrator, epilogue
constexpr int G_STAGES = 5;                        // weight + token tile ring (TMA -> MMA)
constexpr int G_SSTAGES = G_STAGES + 3;            // block-scale ring (TMA -> drain), one slot per stage
constexpr int G_TMEM_BUFS = 5;                     // per-block accumulators in TMEM
constexpr int G_BUF_COLS = TILE_N;                 // 96 fp32 columns per accumulator
constexpr int G_TMEM_COLS = 512;
constexpr int STAGE_A = 16384;                     // 128 weight rows x 128 B (64 fp16 = 2 blocks)
constexpr int STAGE_B = TILE_N * 128;              // up to 96 token rows x 128 B
constexpr int STAGE_BYTES = STAGE_A + STAGE_B;
constexpr int SSTAGE_BYTES = 2048;                 // [2][128] weight scales + [2][nb] token scales
// Q4_K: + [2][128] weight mins (at 2048) + [2][nb] token code sums times scale (at 3072)
__host__ __device__ constexpr int sstage_bytes(int wf) { return wf ? 4096 : SSTAGE_BYTES; }
constexpr int HAND_STRIDE = 132;                   // floats per token column of the hand-off buffer (128 rows + pad)
constexpr int HAND_BYTES = TILE_N * HAND_STRIDE * 4;
constexpr int BAR_BYTES = 512;
constexpr int EPI_BYTES = TILE_N * 8;                // the epilogue warp's output rows and scales
__host__ __device__ constexpr int g_smem(int wf) {
    return 1024 + G_STAGES * STAGE_BYTES + G_SSTAGES * sstage_bytes(wf) + HAND_BYTES + BAR_BYTES + EPI_BYTES;
}
static_assert(g_smem(1) <= 227 * 1024, "shared memory budget");
static_assert(G_TMEM_BUFS * G_BUF_COLS <= G_TMEM_COLS, "TMEM ring exceeds the allocation");
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
// Scale slot reuse needs no barrier of its own.  The producer loads stage L once the MMAs of stage
// L - G_STAGES completed; those were issued only after the drain handed back the TMEM slots they
// write, last used by the first block of stage L - G_STAGES - 2, and every drain warp hands those
// back only after finishing the scale math of stage L - G_STAGES - 3.  Slot L % G_SSTAGES was last
// used by stage L - G_SSTAGES, so G_SSTAGES >= G_STAGES + 3 keeps it unread by then.
static_assert(G_SSTAGES >= G_STAGES + 3, "scale slots could be overwritten while still read");
static_assert(G_TMEM_BUFS == 5, "the argument above assumes stage t's blocks reuse the slots of blocks 2t-5, 2t-4");
// --------------------------------------------------------------- kernel ---

// MODE 0: gate/up (fused SiLU * up, Q8_1 requant); 1: down (scatter).
// DUMP: also store the raw int32 block dots of block p.dbg_block (the debug entry points; a
// separate instantiation keeps the hot loop lean).
// WF: weight format (0 Q8_0, 1 Q4_K: the weight is d*sc*q - dmin*m per 32-block, so each block
// also subtracts (dmin*m) * (d_x * sum of the block's activation codes)).
template <int MODE, bool DUMP, int WF>
__global__ void __launch_bounds__(G_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned start for the swizzled tiles, kept as an offset from the shared array so
    // the compiler still knows every derived pointer is shared memory (plain LDS/STS, not generic)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sring = smem + G_STAGES * STAGE_BYTES;
    // hand-off buffer: an item's accumulators, token column c at hand[c * HAND_STRIDE + row]
    constexpr int SSB = sstage_bytes(WF);
    float *hand = reinterpret_cast<float *>(sring + G_SSTAGES * SSB);
    uint8_t *bars = reinterpret_cast<uint8_t *>(hand) + HAND_BYTES;
    int *epi_row = reinterpret_cast<int *>(bars + BAR_BYTES);  // [TILE_N] output row per column
    float *epi_scale = reinterpret_cast<float *>(epi_row + TILE_N);  // [TILE_N] shared-expert scale
    const uint32_t bar_base = smem_u32(bars);
    int nb_ = 0;
    auto next_bar = [&](int n) {
        const uint32_t b = bar_base + 8 * nb_;
        nb_ += n;
        return b;
    };
    const uint32_t full0 = next_bar(G_STAGES), empty0 = next_bar(G_STAGES);
    const uint32_t tempty0 = next_bar(G_TMEM_BUFS);
    const uint32_t hfull = next_bar(1), hempty = next_bar(1);
    const uint32_t done_bar = next_bar(1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 8 * nb_);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *stages_ready = reinterpret_cast<int *>(tmem_slot + 2);  // orchestrator -> MMA warp

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);   // the copies' arrival (tiles and scales)
            mbar_init(empty0 + 8 * s, 1);  // the stage's MMAs are complete (one commit per stage)
        }
        for (int b = 0; b < G_TMEM_BUFS; ++b) mbar_init(tempty0 + 8 * b, G_DRAIN_WARPS);
        mbar_init(hfull, G_DRAIN_WARPS);  // every drain warp has stored its columns
        mbar_init(hempty, 1);             // the epilogue warp is done with the buffer
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        *stages_ready = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&maps.a_r);
        prefetch_map(&maps.sa_r);
        prefetch_map(&maps.a_s);
        prefetch_map(&maps.sa_s);
        for (int i = 0; i < 4; ++i) {
            prefetch_map(&maps.b[i]);
            prefetch_map(&maps.sb[i]);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(G_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int n_tiles = p.plan->n_tiles;
    int n_rtiles = p.plan->pad;  // routed tiles come first
    n_tiles = min(max(n_tiles, 0), p.tiles_max);
    n_rtiles = min(max(n_rtiles, 0), n_tiles);
    const int n_items = total_items(p, n_tiles, n_rtiles);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int stage = 0, sstage = 0;
            uint32_t phase = 0;
            // per slot: was it ever filled, and the parity of its last fill (bit masks)
            uint32_t issued = 0, last_parity = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok && !p.starve; it += gridDim.x) {
                const Item x = item_at(p, it, n_rtiles);
                const CUtensorMap *ma = x.shared ? &maps.a_s : &maps.a_r;
                const CUtensorMap *msa = x.shared ? &maps.sa_s : &maps.sa_r;
                const int arow = (x.shared ? 0 : x.expert * p.rows_r) + x.mt * 128;
                const int sarow = x.shared ? 0 : x.expert * p.sblk_r;
                for (int ks = 0; ks < x.K / 64; ++ks) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + stage * STAGE_BYTES;
                    uint8_t *ss = sring + sstage * SSB;
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, STAGE_A + x.nb * 128 + (WF ? 2 : 1) * (1024 + 2 * x.nb * 4));
                    tma_load_2d(smem_u32(st), ma, ks * 64, arow, fb);
                    tma_load_2d(smem_u32(st + STAGE_A), &maps.b[x.bi], ks * 64, x.row0, fb);
                    tma_load_2d(smem_u32(ss), msa, x.mt * 128, sarow + 2 * ks, fb);
                    tma_load_2d(smem_u32(ss + 1024), &maps.sb[x.bi], x.row0, 2 * ks, fb);
                    if (WF) {
                        tma_load_2d(smem_u32(ss + 2048), x.shared ? &maps.sm_s : &maps.sm_r, x.mt * 128,
                                    sarow + 2 * ks, fb);
                        tma_load_2d(smem_u32(ss + 3072), &maps.sx[x.bi], x.row0, 2 * ks, fb);
                    }
                    issued |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == G_STAGES) stage = 0, phase ^= 1;
                    if (++sstage == G_SSTAGES) sstage = 0;
                }
            }
            // copies still in flight must land before the CTA can exit
            for (int s = 0; s < G_STAGES; ++s)
                if (issued >> s & 1) {
                    uint64_t t0 = globaltimer();
                    while (!mbar_try(full0 + 8 * s, last_parity >> s & 1) && globaltimer() - t0 < WAIT_LIMIT_NS) {
                    }
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            int stage = 0, buf = 0, mt = 0;  // mt: stages issued over the run
            bool ok = true;
            bool any = false;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const Item x = item_at(p, it, n_rtiles);
                const uint32_t idesc = idesc_f16((x.nrows + 15) & ~15);
                for (int ks = 0; ks < x.K / 64 && ok; ++ks) {
                    // A plain shared-memory poll: an mbarrier wait in the thread that issues the
                    // MMAs stalls it for a few hundred cycles, a shared load for tens.
                    if (ld_acquire_shared(stages_ready) <= mt) {
                        uint64_t t0 = 0;
                        for (uint32_t n = 1; ld_acquire_shared(stages_ready) <= mt; ++n) {
                            if ((n & 255) == 0) {
                                if (*abort_flag) { ok = false; break; }
                                if (t0 == 0) t0 = globaltimer();
                                else if (globaltimer() - t0 > p.wait_ns) {
                                    *abort_flag = 1;
                                    atomicOr(p.status, MOE_DEV_TIMEOUT);
                                    ok = false;
                                    break;
                                }
                            }
                        }
                        if (!ok) break;
                    }
                    ++mt;
                    tc_fence_after();  // the stage's data has landed and its two TMEM slots are free
                    const uint32_t a0 = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t b0 = a0 + STAGE_A;
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t d = tmem_base + buf * G_BUF_COLS;
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint32_t off = half * 64 + kk * 32;  // bytes along K inside the swizzle atom
                            mma_f16(d, smem_desc_sw128(a0 + off), smem_desc_sw128(b0 + off), idesc, kk);
                        }
                        any = true;
                        if (++buf == G_TMEM_BUFS) buf = 0;
                    }
                    // one commit per stage: it tells the drain that both blocks' accumulators are
                    // complete and the producer that the tile slot is free (a thread's commits are
                    // retired at most about one per 330 cycles, so a commit per block would bound
                    // the whole kernel)
                    mma_commit(empty0 + 8 * stage);
                    if (++stage == G_STAGES) stage = 0;
                }
            }
            if (any) {
                // every issued MMA has completed once this commit arrives
                mma_commit(done_bar);
                uint64_t t0 = globaltimer();
                while (!mbar_try(done_bar, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
    } else if (warp == G_ORCH_WARP) {
        // ---------------------------------------------------- orchestrator ---
        // Per stage: wait until its tiles and scales have landed and the drain has handed back
        // the TMEM slots of its two blocks, then publish the stage count to the MMA warp.  The
        // slots of blocks 2t and 2t+1 were last used by blocks 2t-5 (stage t-3) and 2t-4 (stage
        // t-2); every drain warp hands back stage t-3 before stage t-2, so the second slot's
        // barrier alone tells that both are free.
        if (lane == 0) {
            int stage = 0, t = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const Item x = item_at(p, it, n_rtiles);
                for (int ks = 0; ks < x.K / 64 && ok; ++ks) {
                    ok = mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, p.wait_ns);
                    const int j = 2 * t + 1;  // second block of the stage, counted over the run
                    if (ok && j >= G_TMEM_BUFS)
                        ok = mbar_wait(tempty0 + 8 * (j % G_TMEM_BUFS), ((j / G_TMEM_BUFS) - 1) & 1, abort_flag,
                                       p.status, p.wait_ns);
                    if (!ok) break;
                    st_release_shared(stages_ready, ++t);
                    if (++stage == G_STAGES) stage = 0, phase ^= 1;
                }
            }
        }
    } else if (warp == G_EPI_WARP) {
        // -------------------------------------------------------- epilogue ---
        uint32_t hphase = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item x = item_at(p, it, n_rtiles);
            // down: output row (and shared-expert scale) of columns lane, lane + 32, lane + 64,
            // loaded before the wait so they land while the drain works on the item
            int orow[3] = {-1, -1, -1};
            float oscale[3] = {1.0f, 1.0f, 1.0f};
            if (MODE == 1) {
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int col = lane + 32 * j;
                    if (col < x.nrows) {
                        if (x.shared) {
                            orow[j] = x.entry0 + col;  // shared-expert rows map row i to token i
                            oscale[j] = p.shexp_scale[orow[j]];
                        } else {
                            orow[j] = p.rowinfo[x.row0 + col].y;
                        }
                    }
                }
            }
            ok = mbar_wait(hfull, hphase, abort_flag, p.status, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (MODE == 0) {
                // rows 0-63 hold gate, rows 64-127 up, of features mt*64 + (row & 63).  One lane
                // per (token column, 32-feature block): SiLU(gate) * up of the block's 32 features,
                // then the Q8_1 rule on them, 32 fp16 codes stored as one 64-byte run.
                for (int fb = 0; fb < 2; ++fb) {
                    for (int col = lane; col < x.nrows; col += 32) {
                        const float *gcol = hand + col * HAND_STRIDE + 32 * fb;
                        const float *ucol = gcol + 64;
                        float hv[32];
                        float amax = 0.0f;
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4) {
                            const float4 g = *reinterpret_cast<const float4 *>(gcol + 4 * i4);
                            const float4 u = *reinterpret_cast<const float4 *>(ucol + 4 * i4);
                            hv[4 * i4 + 0] = swiglu(g.x, u.x);
                            hv[4 * i4 + 1] = swiglu(g.y, u.y);
                            hv[4 * i4 + 2] = swiglu(g.z, u.z);
                            hv[4 * i4 + 3] = swiglu(g.w, u.w);
#pragma unroll
                            for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(hv[4 * i4 + k]));
                        }
                        const float d = __fdiv_rn(amax, 127.0f);
                        const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
                        const int prow = x.row0 + col;
                        const int f0 = x.mt * 64 + 32 * fb;
                        const float d16 = __half2float(__float2half_rn(d));
                        p.h_dT[(size_t)(f0 >> 5) * p.rows_max + prow] = d16;
                        __align__(16) __half2 hq[16];
                        int qsum = 0;  // the block's code sum (the down GEMM's Q4_K min term)
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int q0 = (int)roundf(__fmul_rn(hv[2 * i], id));
                            const int q1 = (int)roundf(__fmul_rn(hv[2 * i + 1], id));
                            qsum += q0 + q1;
                            hq[i] = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
                        }
                        if (WF) p.h_sT[(size_t)(f0 >> 5) * p.rows_max + prow] = d16 * (float)qsum;
                        int4 *dst = reinterpret_cast<int4 *>(p.h16 + (size_t)prow * p.Fmax + f0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = reinterpret_cast<const int4 *>(hq)[i];
                    }
                }
            } else {
                // one token column at a time: its 128 output features, 4 per lane, one 512-byte row;
                // four columns in flight per step
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int col = lane + 32 * j;
                    if (col < TILE_N) {
                        epi_row[col] = orow[j];
                        epi_scale[col] = oscale[j];
                    }
                }
                __syncwarp();
                float *__restrict__ dstb = x.shared ? p.shared_out : p.partials;
                // the combine reads these rows next: ask L2 to keep them over the streamed weights
                const uint64_t keep = l2_evict_last_policy();
                for (int col = 0; col < x.nrows; col += 4) {
                    float4 v[4];
                    int o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c = min(col + u, TILE_N - 1);
                        o[u] = col + u < x.nrows ? epi_row[c] : -1;
                        v[u] = *reinterpret_cast<const float4 *>(hand + c * HAND_STRIDE + 4 * lane);
                        if (x.shared) {
                            const float sc = epi_scale[c];
                            v[u] = make_float4(sc * v[u].x, sc * v[u].y, sc * v[u].z, sc * v[u].w);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (o[u] >= 0) st_evict_last(dstb + (size_t)o[u] * p.D + x.mt * 128 + 4 * lane, v[u], keep);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(hempty);
            hphase ^= 1;
        }
    } else {
        // ------------------------------------------------------- drain ---
        const int q = warp & 3;              // TMEM lane quarter (= SM sub-partition) of this warp
        const int grp = (warp - 2) >> 2;     // column group: token columns 32*grp + [0, 32)
        const int r = q * 32 + lane;         // row of the 128-row weight tile
        int sstage = 0, buf = 0, dstage = 0;
        uint32_t tphase = 0, hphase = 0, dphase = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item x = item_at(p, it, n_rtiles);
            // this warp's columns: 32*grp + [0, 32) of the token tile; acc[m] = columns 2m, 2m+1
            const int c0 = 32 * grp;
            const bool active = c0 < x.nrows;  // warp-uniform: whole groups beyond the tile idle
            float2 acc[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = make_float2(0.0f, 0.0f);
            const uint32_t tlane = tmem_base + ((uint32_t)(q * 32) << 16) + c0;
            // Per stage (two K blocks in two TMEM slots): one wait for the stage's commit (it covers
            // both blocks, and the MMA warp only issued them once the stage's tiles and scales had
            // landed), both TMEM loads, then the slots go back before the math, which interleaves
            // the two blocks.  The drain never falls two phases behind a stage barrier: the MMAs of
            // stage t + G_STAGES need TMEM slots it hands back only after stage t + 2.
            const int nst = x.K / 64;
            uint32_t v0[32], v1[32];
            for (int ks = 0; ks < nst && ok; ++ks) {
                const int s0 = buf;
                int s1 = buf + 1;
                uint32_t ph1 = tphase;
                if (s1 == G_TMEM_BUFS) s1 = 0, ph1 ^= 1;
                ok = mbar_wait(empty0 + 8 * dstage, dphase, abort_flag, p.status, p.wait_ns);
                if (++dstage == G_STAGES) dstage = 0, dphase ^= 1;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (active) {
                    tmem_ld32(tlane + s0 * G_BUF_COLS, v0);
                    tmem_ld32(tlane + s1 * G_BUF_COLS, v1);
                }
                if (active) {
                    tmem_wait_ld();
                    tmem_reg_fence32(v0);
                    tmem_reg_fence32(v1);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(tempty0 + 8 * s0);
                    mbar_arrive(tempty0 + 8 * s1);
                }
                buf = s1 + 1;
                tphase = ph1;
                if (buf == G_TMEM_BUFS) buf = 0, tphase ^= 1;
                if (active) {
                    const float *SA = reinterpret_cast<const float *>(sring + sstage * SSB);
                    const float *SB = SA + 256;
                    if (DUMP && x.shared == 0 && (2 * ks == p.dbg_block || 2 * ks + 1 == p.dbg_block)) {
                        const uint32_t *v = (2 * ks == p.dbg_block) ? v0 : v1;
                        for (int j = 0; j < 32 && c0 + j < x.nrows; ++j) {
                            const size_t e = (size_t)(x.entry0 + c0 + j);
                            if (MODE == 0)
                                p.dbg_dots[(e * 2 + (r < 64 ? 0 : 1)) * p.F + x.mt * 64 + (r & 63)] =
                                    (int32_t)__uint_as_float(v[j]);
                            else
                                p.dbg_dots[e * p.D + x.mt * 128 + r] = (int32_t)__uint_as_float(v[j]);
                        }
                    }
                    const float dwa = SA[r], dwb = SA[128 + r];
                    const float2 dw2a = make_float2(dwa, dwa), dw2b = make_float2(dwb, dwb);
                    const float4 *sa4 = reinterpret_cast<const float4 *>(SB + c0);
                    const float4 *sb4 = reinterpret_cast<const float4 *>(SB + x.nb + c0);
                    // Q4_K: minus the mins of the two blocks (weight rows) and the code sums times scale
                    // (token columns), both staged behind the scales
                    const float *SMn = SA + 512, *SX = SA + 768;
                    const float2 nma = WF ? make_float2(-SMn[r], -SMn[r]) : make_float2(0.f, 0.f);
                    const float2 nmb = WF ? make_float2(-SMn[128 + r], -SMn[128 + r]) : make_float2(0.f, 0.f);
                    const float4 *xa4 = reinterpret_cast<const float4 *>(SX + c0);
                    const float4 *xb4 = reinterpret_cast<const float4 *>(SX + x.nb + c0);
#pragma unroll
                    for (int g4 = 0; g4 < 8; ++g4) {
                        // token scales of columns 4*g4 .. 4*g4+3 for the two blocks (broadcast loads)
                        const float4 ta = sa4[g4], tb = sb4[g4];
                        const float2 a01 = __fmul2_rn(make_float2(ta.x, ta.y), dw2a);
                        const float2 a23 = __fmul2_rn(make_float2(ta.z, ta.w), dw2a);
                        const float2 b01 = __fmul2_rn(make_float2(tb.x, tb.y), dw2b);
                        const float2 b23 = __fmul2_rn(make_float2(tb.z, tb.w), dw2b);
                        float2 u = __ffma2_rn(make_float2(__uint_as_float(v0[4 * g4]), __uint_as_float(v0[4 * g4 + 1])),
                                              a01, acc[2 * g4]);
                        float2 w = __ffma2_rn(
                            make_float2(__uint_as_float(v0[4 * g4 + 2]), __uint_as_float(v0[4 * g4 + 3])), a23,
                            acc[2 * g4 + 1]);
                        if (WF) {
                            const float4 xa = xa4[g4];
                            u = __ffma2_rn(make_float2(xa.x, xa.y), nma, u);
                            w = __ffma2_rn(make_float2(xa.z, xa.w), nma, w);
                        }
                        u = __ffma2_rn(make_float2(__uint_as_float(v1[4 * g4]), __uint_as_float(v1[4 * g4 + 1])), b01, u);
                        w = __ffma2_rn(make_float2(__uint_as_float(v1[4 * g4 + 2]), __uint_as_float(v1[4 * g4 + 3])), b23,
                                       w);
                        if (WF) {
                            const float4 xb = xb4[g4];
                            u = __ffma2_rn(make_float2(xb.x, xb.y), nmb, u);
                            w = __ffma2_rn(make_float2(xb.z, xb.w), nmb, w);
                        }
                        acc[2 * g4] = u;
                        acc[2 * g4 + 1] = w;
                    }
                }
                if (++sstage == G_SSTAGES) sstage = 0;
            }
            tmem_wait_ld();  // no TMEM load outlives the loop, even when it was cut short
            if (!ok) break;
            // ------------------------------------------------------ hand-off ---
            // the epilogue warp finishes the item from shared memory while this warp moves on
            ok = mbar_wait(hempty, hphase ^ 1, abort_flag, p.status, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (active) {
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    hand[(c0 + 2 * m) * HAND_STRIDE + r] = acc[m].x;
                    hand[(c0 + 2 * m + 1) * HAND_STRIDE + r] = acc[m].y;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(hfull);
            hphase ^= 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(G_TMEM_COLS)
                     : "memory");
}

// ------------------------------------------------ planning and gathering ---
// One CTA: padded segment starts (16-row aligned), token tiles of <= tile_n rows
// per segment (routed experts first, then the shared expert's N rows), and for
// every padded row its source token, output row and CSR entry.
__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t *__restrict__ expStart, const int32_t *__restrict__ expTokI,
            const int32_t *__restrict__ expTokK, int N, int top_k, int E, int with_shared, int rows_max,
            int tiles_max, int tile_n, PlanHeader *hdr, int32_t *gstart_out, TileDesc *tiles, int4 *rowinfo,
            unsigned *status) {
    __shared__ int cnt[MAX_E + 1], gst[MAX_E + 2], tst[MAX_E + 2];
    __shared__ int bad;
    const int tid = threadIdx.x;
    const int total = N * top_k;
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int a = expStart[e], b = expStart[e + 1];
        if (a < 0 || b < a || b > total) bad = 1;
        cnt[e] = b - a;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            atomicOr(status, MOE_DEV_BAD_CSR);
            hdr->n_tiles = 0;
            hdr->n_rows = 0;
            hdr->shared_row0 = -1;
            hdr->pad = 0;
        }
        return;
    }
    if (tid == 0) {
        // serial scans over <= 1025 segments: negligible next to the GEMMs
        int g = 0, t = 0;
        for (int e = 0; e < E; ++e) {
            gst[e] = g;
            tst[e] = t;
            g += (cnt[e] + SEG_ALIGN - 1) / SEG_ALIGN * SEG_ALIGN;
            t += (cnt[e] + tile_n - 1) / tile_n;
        }
        gst[E] = g;
        tst[E] = t;
        const int ns = with_shared ? N : 0;
        gst[E + 1] = g + (ns + SEG_ALIGN - 1) / SEG_ALIGN * SEG_ALIGN;
        tst[E + 1] = t + (ns + tile_n - 1) / tile_n;
        hdr->n_tiles = min(tst[E + 1], tiles_max);
        hdr->n_rows = min(gst[E + 1], rows_max);
        hdr->shared_row0 = with_shared ? g : -1;
        hdr->pad = tst[E];  // routed tiles
    }
    __syncthreads();
    for (int e = tid; e <= E + 1; e += blockDim.x) gstart_out[e] = gst[e];
    // tiles
    for (int e = tid; e <= E; e += blockDim.x) {
        const bool sh = (e == E);
        if (sh && !with_shared) continue;
        const int n = sh ? N : cnt[e];
        for (int i = 0; i * tile_n < n; ++i) {
            const int ti = tst[e] + i;
            if (ti >= tiles_max) break;
            TileDesc td;
            td.row0 = gst[e] + i * tile_n;
            td.nrows = min(tile_n, n - i * tile_n);
            td.expert = e;
            td.entry0 = (sh ? 0 : expStart[e]) + i * tile_n;
            tiles[ti] = td;
        }
    }
    // rows: .x source token, .y output row (t*top_k + slot, or t for the shared expert), .z CSR entry
    const int nrows = min(gst[E + 1], rows_max);
    for (int prow = tid; prow < nrows; prow += blockDim.x) {
        int lo = 0, hi = E + 1;  // find e with gst[e] <= prow < gst[e+1]
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (gst[mid] <= prow) lo = mid;
            else hi = mid;
        }
        const int e = lo;
        const int i = prow - gst[e];
        int4 ri = make_int4(-1, -1, -1, 0);
        if (e < E) {
            if (i < cnt[e]) {
                const int j = expStart[e] + i;
                const int t = expTokI[j];
                const int s = expTokK ? expTokK[j] : 0;
                if ((unsigned)t < (unsigned)N && (unsigned)s < (unsigned)top_k) {
                    ri = make_int4(t, t * top_k + s, j, 0);
                } else {
                    atomicOr(status, MOE_DEV_BAD_CSR);
                }
            }
        } else if (with_shared && i < N) {
            ri = make_int4(i, i, -1, 0);
        }
        rowinfo[prow] = ri;
    }
}

// Gather the Q8_1 rows of x into the padded segment order as exact fp16
// integers, and their block scales transposed ([D/32][rows]).  A CTA owns
// GATHER_ROWS padded rows (one wave of CTAs for the OLMoE shape); a warp takes
// two of them.  Each lane turns 8 int8 codes into 8 fp16 values per step, so a
// warp reads 256 contiguous bytes and writes 512; all of a row pair's loads are
// issued before the first store.  Pad rows are zero.
constexpr int GATHER_ROWS = 16;
constexpr int GATHER_UNR = 8;
// 4 signed bytes -> 4 fp16 integers: the byte b + 128 goes into the mantissa of 1024
// (0x6400 | (b ^ 0x80) is the fp16 value 1152 + b), then 1152 is subtracted; exact for
// every int8, since fp16 spaces the integers of [1024, 2048) one apart.
__device__ __forceinline__ uint2 i8x4_to_h16x4(uint32_t v) {
    const uint32_t u = v ^ 0x80808080u;
    const uint32_t lo = __byte_perm(u, 0x64646464u, 0x5140);  // bytes 0, 1 over 0x64 high halves
    const uint32_t hi = __byte_perm(u, 0x64646464u, 0x7362);  // bytes 2, 3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    const __half2 a = __hsub2(*reinterpret_cast<const __half2 *>(&lo), bias);
    const __half2 b = __hsub2(*reinterpret_cast<const __half2 *>(&hi), bias);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
}

__global__ void __launch_bounds__(256)
gather_kernel(const int8_t *__restrict__ x_q, const float *__restrict__ x_d, int D, const PlanHeader *hdr,
              const int4 *__restrict__ rowinfo, int rows_max, __half *__restrict__ xg16, float *__restrict__ xg_dT,
              float *__restrict__ xg_sT) {
    __shared__ int src[GATHER_ROWS];
    const int row0 = blockIdx.x * GATHER_ROWS;
    const int nrows = hdr->n_rows;
    if (row0 >= nrows) return;
    if (threadIdx.x < GATHER_ROWS) {
        const int prow = row0 + threadIdx.x;
        src[threadIdx.x] = prow < nrows ? rowinfo[prow].x : -1;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n8 = D / 8;  // 8-code pieces per row
    const int ra = 2 * warp, rb = 2 * warp + 1;
    const int ta = row0 + ra < nrows ? src[ra] : -2, tb = row0 + rb < nrows ? src[rb] : -2;  // -2: past the rows
    for (int c0 = lane; c0 < n8; c0 += 32 * GATHER_UNR) {
        uint2 va[GATHER_UNR], vb[GATHER_UNR];
#pragma unroll
        for (int u = 0; u < GATHER_UNR; ++u) {
            const int c = c0 + 32 * u;
            va[u] = (ta >= 0 && c < n8) ? reinterpret_cast<const uint2 *>(x_q + (size_t)ta * D)[c] : make_uint2(0, 0);
            vb[u] = (tb >= 0 && c < n8) ? reinterpret_cast<const uint2 *>(x_q + (size_t)tb * D)[c] : make_uint2(0, 0);
        }
#pragma unroll
        for (int u = 0; u < GATHER_UNR; ++u) {
            const int c = c0 + 32 * u;
            if (c >= n8) break;
            if (ta != -2) {
                const uint2 a = i8x4_to_h16x4(va[u].x), b = i8x4_to_h16x4(va[u].y);
                reinterpret_cast<uint4 *>(xg16 + (size_t)(row0 + ra) * D)[c] = make_uint4(a.x, a.y, b.x, b.y);
            }
            if (tb != -2) {
                const uint2 a = i8x4_to_h16x4(vb[u].x), b = i8x4_to_h16x4(vb[u].y);
                reinterpret_cast<uint4 *>(xg16 + (size_t)(row0 + rb) * D)[c] = make_uint4(a.x, a.y, b.x, b.y);
            }
        }
    }
    // scales: 16 consecutive rows of one block per half warp (64-byte runs of xg_dT)
    const int nblk = D / QK;
    const int rr = threadIdx.x & (GATHER_ROWS - 1);
    const int prow = row0 + rr;
    const int t = src[rr];
    for (int b = threadIdx.x / GATHER_ROWS; b < nblk; b += 256 / GATHER_ROWS) {
        const bool live = t >= 0 && prow < nrows;
        const float d = live ? x_d[(size_t)t * nblk + b] : 0.0f;
        if (prow < rows_max) xg_dT[(size_t)b * rows_max + prow] = d;
        if (xg_sT != nullptr && prow < rows_max) {  // Q4_K weights: the block's code sum times its scale
            int sum = 0;
            if (live) {
                const int4 *src = reinterpret_cast<const int4 *>(x_q + (size_t)t * D + (size_t)b * QK);
                const int4 a = src[0], c = src[1];
                sum = __dp4a(a.x, 0x01010101, __dp4a(a.y, 0x01010101, __dp4a(a.z, 0x01010101, __dp4a(a.w, 0x01010101, 0))));
                sum = __dp4a(c.x, 0x01010101, __dp4a(c.y, 0x01010101, __dp4a(c.z, 0x01010101, __dp4a(c.w, 0x01010101, sum))));
            }
            xg_sT[(size_t)b * rows_max + prow] = d * (float)sum;
        }
    }
}
static_assert(2 * (256 / 32) == GATHER_ROWS, "two rows per warp");

// h (fp16 codes + transposed scales, padded order) -> int8 + fp32 scales in CSR entry order.
__global__ void h16_to_q8_kernel(const __half *__restrict__ h16, const float *__restrict__ h_dT, int F, int Fmax,
                                 int rows_max, const PlanHeader *hdr, const int4 *__restrict__ rowinfo,
                                 int8_t *__restrict__ h_q, float *__restrict__ h_d) {
    const int prow = blockIdx.x;
    if (prow >= hdr->n_rows) return;
    const int j = rowinfo[prow].z;
    if (j < 0) return;
    for (int f = threadIdx.x; f < F; f += blockDim.x) {
        h_q[(size_t)j * F + f] = (int8_t)__half2int_rn(h16[(size_t)prow * Fmax + f]);
        if ((f & 31) == 0) h_d[(size_t)j * (F / QK) + f / QK] = h_dT[(size_t)(f / QK) * rows_max + prow];
    }
}

// int8 + fp32 scales in CSR entry order -> fp16 codes + transposed scales in padded order.
__global__ void q8_to_h16_kernel(const int8_t *__restrict__ h_q, const float *__restrict__ h_d, int F, int Fmax,
                                 int rows_max, const PlanHeader *hdr, const int4 *__restrict__ rowinfo,
                                 __half *__restrict__ h16, float *__restrict__ h_dT, float *__restrict__ h_sT) {
    const int prow = blockIdx.x;
    if (prow >= hdr->n_rows) return;
    const int j = rowinfo[prow].z;
    for (int f = threadIdx.x; f < F; f += blockDim.x) {
        const int v = j >= 0 ? h_q[(size_t)j * F + f] : 0;
        h16[(size_t)prow * Fmax + f] = __int2half_rn(v);
        if ((f & 31) == 0) {
            const float d = j >= 0 ? h_d[(size_t)j * (F / QK) + f / QK] : 0.0f;
            h_dT[(size_t)(f / QK) * rows_max + prow] = d;
            if (h_sT != nullptr) {  // Q4_K weights: the block's code sum times its scale
                int sum = 0;
                for (int i = 0; i < QK && j >= 0; ++i) sum += h_q[(size_t)j * F + f + i];
                h_sT[(size_t)(f / QK) * rows_max + prow] = d * (float)sum;
            }
        }
    }
}

// ----------------------------------------------------- tensor map encode ---
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
    });
    return fn;
}

// 2D row-major tensor [rows][cols] of fp16 (swizzled 64-wide boxes) or fp32 (plain boxes).
bool encode_2d(CUtensorMap *m, const void *base, bool fp16, uint64_t rows, uint64_t cols, uint32_t box_cols,
               uint32_t box_rows) {
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const size_t es = fp16 ? 2 : 4;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * es};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    fp16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct WeightMaps {
    CUtensorMap gu_r, gu_dT_r, dn_r, dn_dT_r;
    CUtensorMap gu_s, gu_dT_s, dn_s, dn_dT_s;
    CUtensorMap gu_mT_r, dn_mT_r, gu_mT_s, dn_mT_s;  // Q4_K mins, as the scales
};

// One instantiation per (mode, dump, weight format), each with its own dynamic shared memory size.
template <int MODE, bool DUMP, int WF>
int run_gemm(const GemmMaps &maps, const GemmParams &p, int num_sms, cudaStream_t s) {
    static SmemOptIn configured;
    if (int rc = ensure_dynamic_smem((const void *)grouped_gemm_kernel<MODE, DUMP, WF>, g_smem(WF), &configured))
        return rc;
    grouped_gemm_kernel<MODE, DUMP, WF><<<num_sms, G_THREADS, g_smem(WF), s>>>(maps, p);
    return launch_status();
}

int launch_gemm(int mode, const moe_weights_s *w, int N, int top_k, bool with_shared, void *ws, const WsLayout &L,
                float *partials, float *shared_out, const float *shexp_scale, int32_t *dbg_dots, int dbg_block,
                cudaStream_t s, unsigned long long wait_ns = WAIT_LIMIT_NS, int starve = 0) {
    const WeightMaps *wm = static_cast<const WeightMaps *>(w->tmaps);
    if (!wm) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int D = w->D, F = w->F, Fs = w->Fs, Fmax = std::max(F, Fs);
    GemmMaps maps;
    GemmParams p{};
    const int wf = w->wfmt == MOE_WFMT_Q4_K ? 1 : 0;
    if (mode == 0) {
        maps.a_r = wm->gu_r;
        maps.sa_r = wm->gu_dT_r;
        maps.a_s = Fs ? wm->gu_s : wm->gu_r;
        maps.sa_s = Fs ? wm->gu_dT_s : wm->gu_dT_r;
        if (wf) {
            maps.sm_r = wm->gu_mT_r;
            maps.sm_s = Fs ? wm->gu_mT_s : wm->gu_mT_r;
        }
        p.K_r = D;
        p.K_s = D;
        p.MT_r = 2 * F / 128;
        p.MT_s = Fs ? 2 * Fs / 128 : 1;
        p.rows_r = 2 * F;
        p.rows_s = 2 * Fs;
        p.sblk_r = D / QK;
        p.sblk_s = D / QK;
    } else {
        maps.a_r = wm->dn_r;
        maps.sa_r = wm->dn_dT_r;
        maps.a_s = Fs ? wm->dn_s : wm->dn_r;
        maps.sa_s = Fs ? wm->dn_dT_s : wm->dn_dT_r;
        if (wf) {
            maps.sm_r = wm->dn_mT_r;
            maps.sm_s = Fs ? wm->dn_mT_s : wm->dn_mT_r;
        }
        p.K_r = F;
        p.K_s = Fs ? Fs : F;
        p.MT_r = D / 128;
        p.MT_s = D / 128;
        p.rows_r = D;
        p.rows_s = D;
        p.sblk_r = F / QK;
        p.sblk_s = Fs / QK;
    }
    // token-side maps over the workspace (per call: the workspace is the caller's)
    const int rows = L.rows_max;
    void *bdata = mode == 0 ? (void *)ws_ptr<__half>(ws, L.xg16) : (void *)ws_ptr<__half>(ws, L.h16);
    void *bscale = mode == 0 ? (void *)ws_ptr<float>(ws, L.xg_dT) : (void *)ws_ptr<float>(ws, L.h_dT);
    void *bsum = mode == 0 ? (void *)ws_ptr<float>(ws, L.xg_sT) : (void *)ws_ptr<float>(ws, L.h_sT);
    const int kcols = mode == 0 ? D : Fmax;
    for (int i = 0; i < 4; ++i) {
        const uint32_t nb = i < 3 ? (16u << i) : (uint32_t)TILE_N;  // box heights 16/32/64/96
        if (!encode_2d(&maps.b[i], bdata, true, rows, kcols, 64, nb)) return MOE_ERR_CUDA;
        if (!encode_2d(&maps.sb[i], bscale, false, kcols / QK, rows, nb, 2)) return MOE_ERR_CUDA;
        if (wf && !encode_2d(&maps.sx[i], bsum, false, kcols / QK, rows, nb, 2)) return MOE_ERR_CUDA;
    }
    p.E = w->E;
    p.D = D;
    p.F = F;
    p.Fs = Fs;
    p.Fmax = Fmax;
    p.top_k = top_k;
    p.N = N;
    p.rows_max = rows;
    p.tiles_max = L.tiles_max;
    p.plan = ws_ptr<PlanHeader>(ws, L.plan);
    p.tiles = ws_ptr<TileDesc>(ws, L.tiles);
    p.rowinfo = ws_ptr<int4>(ws, L.rowinfo);
    p.h16 = ws_ptr<__half>(ws, L.h16);
    p.h_dT = ws_ptr<float>(ws, L.h_dT);
    p.h_sT = ws_ptr<float>(ws, L.h_sT);
    p.partials = partials;
    p.shared_out = shared_out;
    p.shexp_scale = shexp_scale;
    p.dbg_dots = dbg_dots;
    p.dbg_block = dbg_block;
    p.status = reinterpret_cast<unsigned *>(ws);
    p.wait_ns = wait_ns;
    p.starve = starve;
    (void)with_shared;
    const bool dump = dbg_dots != nullptr;
    const int num_sms = device_sm_count();
    if (num_sms <= 0) return MOE_ERR_CUDA;
    if (mode == 0)
        return dump ? (wf ? run_gemm<0, true, 1>(maps, p, num_sms, s) : run_gemm<0, true, 0>(maps, p, num_sms, s))
                    : (wf ? run_gemm<0, false, 1>(maps, p, num_sms, s) : run_gemm<0, false, 0>(maps, p, num_sms, s));
    return dump ? (wf ? run_gemm<1, true, 1>(maps, p, num_sms, s) : run_gemm<1, true, 0>(maps, p, num_sms, s))
                : (wf ? run_gemm<1, false, 1>(maps, p, num_sms, s) : run_gemm<1, false, 0>(maps, p, num_sms, s));
}

}  // namespace

bool tensor_path_supported(const moe_weights_s *w) { return w && w->tensor_ok && w->tmaps != nullptr; }

bool encode_fp32_sw128_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int prepare_tensor_maps(moe_weights_s *w) {
    if (!encode_fn()) return MOE_OK;  // no driver entry point: the tensor path stays off
    WeightMaps *m = new WeightMaps();
    const int E = w->E, D = w->D, F = w->F, Fs = w->Fs;
    bool ok = encode_2d(&m->gu_r, w->routed.gu16, true, (uint64_t)E * 2 * F, D, 64, 128) &&
              encode_2d(&m->gu_dT_r, w->routed.gu_dT, false, (uint64_t)E * (D / QK), 2 * F, 128, 2) &&
              encode_2d(&m->dn_r, w->routed.dn16, true, (uint64_t)E * D, F, 64, 128) &&
              encode_2d(&m->dn_dT_r, w->routed.dn_dT, false, (uint64_t)E * (F / QK), D, 128, 2);
    if (ok && Fs)
        ok = encode_2d(&m->gu_s, w->shared.gu16, true, (uint64_t)2 * Fs, D, 64, 128) &&
             encode_2d(&m->gu_dT_s, w->shared.gu_dT, false, (uint64_t)(D / QK), 2 * Fs, 128, 2) &&
             encode_2d(&m->dn_s, w->shared.dn16, true, (uint64_t)D, Fs, 64, 128) &&
             encode_2d(&m->dn_dT_s, w->shared.dn_dT, false, (uint64_t)(Fs / QK), D, 128, 2);
    if (ok && w->wfmt == MOE_WFMT_Q4_K) {
        ok = encode_2d(&m->gu_mT_r, w->routed.gu_mT, false, (uint64_t)E * (D / QK), 2 * F, 128, 2) &&
             encode_2d(&m->dn_mT_r, w->routed.dn_mT, false, (uint64_t)E * (F / QK), D, 128, 2);
        if (ok && Fs)
            ok = encode_2d(&m->gu_mT_s, w->shared.gu_mT, false, (uint64_t)(D / QK), 2 * Fs, 128, 2) &&
                 encode_2d(&m->dn_mT_s, w->shared.dn_mT, false, (uint64_t)(Fs / QK), D, 128, 2);
    }
    if (!ok) {
        delete m;
        return MOE_OK;  // tensor path unavailable; the matvec path still serves every call
    }
    w->tmaps = m;
    return MOE_OK;
}

void free_tensor_maps(moe_weights_s *w) {
    delete static_cast<WeightMaps *>(w->tmaps);
    w->tmaps = nullptr;
}

int launch_plan_and_gather(const moe_weights_s *w, const int8_t *x_q, const float *x_d, const int32_t *expStart,
                           const int32_t *expTokI, const int32_t *expTokK, int N, int top_k, bool with_shared,
                           void *ws, const WsLayout &L, cudaStream_t s, bool plan_ready) {
    PlanHeader *hdr = ws_ptr<PlanHeader>(ws, L.plan);
    int32_t *gst = reinterpret_cast<int32_t *>(hdr + 1);
    int rc = MOE_OK;
    if (!plan_ready) {
        plan_kernel<<<1, 1024, 0, s>>>(expStart, expTokI, expTokK, N, top_k, w->E, with_shared ? 1 : 0, L.rows_max,
                                       L.tiles_max, plan_tile_rows(w), hdr, gst, ws_ptr<TileDesc>(ws, L.tiles),
                                       ws_ptr<int4>(ws, L.rowinfo), reinterpret_cast<unsigned *>(ws));
        rc = launch_status();
    }
    if (rc || x_q == nullptr) return rc;
    gather_kernel<<<(L.rows_max + GATHER_ROWS - 1) / GATHER_ROWS, 256, 0, s>>>(
        x_q, x_d, w->D, hdr, ws_ptr<int4>(ws, L.rowinfo), L.rows_max, ws_ptr<__half>(ws, L.xg16),
        ws_ptr<float>(ws, L.xg_dT), w->wfmt == MOE_WFMT_Q4_K ? ws_ptr<float>(ws, L.xg_sT) : nullptr);
    return launch_status();
}

int launch_gemm_gate_up(const moe_weights_s *w, int N, int top_k, bool with_shared, void *ws, const WsLayout &L,
                        int32_t *dbg_dots, int dbg_block, cudaStream_t s) {
    return launch_gemm(0, w, N, top_k, with_shared, ws, L, nullptr, nullptr, nullptr, dbg_dots, dbg_block, s);
}

int launch_gemm_gate_up_starved(const moe_weights_s *w, int N, int top_k, void *ws, const WsLayout &L,
                                unsigned long long wait_ns, cudaStream_t s) {
    return launch_gemm(0, w, N, top_k, false, ws, L, nullptr, nullptr, nullptr, nullptr, -1, s, wait_ns, 1);
}

int launch_gemm_down(const moe_weights_s *w, int N, int top_k, bool with_shared, const float *shexp_scale,
                     float *partials, float *shared_out, void *ws, const WsLayout &L, cudaStream_t s,
                     int32_t *dbg_dots, int dbg_block) {
    return launch_gemm(1, w, N, top_k, with_shared, ws, L, partials, shared_out, shexp_scale, dbg_dots, dbg_block,
                       s);
}

int launch_h16_to_q8(const moe_weights_s *w, int N, int top_k, void *ws, const WsLayout &L, int8_t *h_q, float *h_d,
                     cudaStream_t s) {
    (void)N;
    (void)top_k;
    const int Fmax = std::max(w->F, w->Fs);
    h16_to_q8_kernel<<<L.rows_max, 256, 0, s>>>(ws_ptr<__half>(ws, L.h16), ws_ptr<float>(ws, L.h_dT), w->F, Fmax,
                                                L.rows_max, ws_ptr<PlanHeader>(ws, L.plan),
                                                ws_ptr<int4>(ws, L.rowinfo), h_q, h_d);
    return launch_status();
}

int launch_q8_to_h16(const moe_weights_s *w, int N, int top_k, void *ws, const WsLayout &L, const int8_t *h_q,
                     const float *h_d, cudaStream_t s) {
    (void)N;
    (void)top_k;
    const int Fmax = std::max(w->F, w->Fs);
    q8_to_h16_kernel<<<L.rows_max, 256, 0, s>>>(h_q, h_d, w->F, Fmax, L.rows_max, ws_ptr<PlanHeader>(ws, L.plan),
                                                ws_ptr<int4>(ws, L.rowinfo), ws_ptr<__half>(ws, L.h16),
                                                ws_ptr<float>(ws, L.h_dT),
                                                w->wfmt == MOE_WFMT_Q4_K ? ws_ptr<float>(ws, L.h_sT) : nullptr);
    return launch_status();
}

}  // namespace moe
