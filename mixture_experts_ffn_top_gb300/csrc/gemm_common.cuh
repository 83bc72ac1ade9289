// gemm_common.cuh -- parameters and work-item schedule of the tensor-core expert GEMM (gate/up
// and down, every weight format).  A work item is one 128-row
// weight tile of one expert against one token tile of that expert's CSR segment; items are
// numbered routed tiles first (MT_r row tiles each), then the shared expert's tiles.
#pragma once

#include <cuda.h>

#include "moe_internal.cuh"

namespace moe {
namespace gemm {

constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s: any healthy wait is microseconds

struct GemmMaps {
    CUtensorMap a_r, sa_r, a_s, sa_s;  // weights + weight scales, routed / shared
    CUtensorMap b[4], sb[4];           // tokens + token scales, box heights 16/32/64/96
    CUtensorMap sm_r, sm_s;            // Q4_K: weight mins, routed / shared
    CUtensorMap sx[4];                 // Q4_K: token code sums times scale, box heights as sb
};

struct GemmParams {
    int K_r, K_s;      // reduction length of routed / shared tiles
    int MT_r, MT_s;    // 128-row weight tiles per token tile, routed / shared
    int rows_r, rows_s;  // weight rows per expert in the A tensor map (2F or D), routed / shared
    int sblk_r, sblk_s;  // scale rows per expert in the SA map (K/32)
    int E, D, F, Fs, Fmax, top_k, N, rows_max, tiles_max;
    const PlanHeader *plan;
    const TileDesc *tiles;
    const int4 *rowinfo;
    __half *h16;       // gate/up output (fp16 integer codes), row stride Fmax
    float *h_dT;       // [Fmax/32][rows_max]
    float *h_sT;       // Q4_K: [Fmax/32][rows_max] code sum of each h block times its scale
    float *partials;
    float *shared_out;
    const float *shexp_scale;
    int32_t *dbg_dots;
    int dbg_block;
    unsigned *status;
    unsigned long long wait_ns;  // limit of every mbarrier wait
    int starve;                  // failure-detection check: the producer issues no copy
};

// ------------------------------------------------------------ schedule ---
struct Item {
    int tile, mt, shared, K, nrows, row0, expert, entry0, nb, bi;
};
__device__ __forceinline__ int total_items(const GemmParams &p, int n_tiles, int n_rtiles) {
    return n_rtiles * p.MT_r + (n_tiles - n_rtiles) * p.MT_s;
}
// The token-side tensor maps have box heights 16/32/64/96; bi picks the smallest box that holds
// the tile's rows.
__device__ __forceinline__ Item item_at(const GemmParams &p, int it, int n_rtiles) {
    Item x;
    if (it < n_rtiles * p.MT_r) {
        x.tile = it / p.MT_r;
        x.mt = it - x.tile * p.MT_r;
        x.shared = 0;
        x.K = p.K_r;
    } else {
        int i2 = it - n_rtiles * p.MT_r;
        x.tile = n_rtiles + i2 / p.MT_s;
        x.mt = i2 % p.MT_s;
        x.shared = 1;
        x.K = p.K_s;
    }
    const TileDesc td = p.tiles[x.tile];
    x.nrows = td.nrows;
    x.row0 = td.row0;
    x.expert = td.expert;
    x.entry0 = td.entry0;
    x.bi = x.nrows <= 16 ? 0 : x.nrows <= 32 ? 1 : x.nrows <= 64 ? 2 : 3;
    x.nb = x.bi < 3 ? (16 << x.bi) : TILE_N;
    return x;
}


// SiLU(g) * u with the fast exponential and division (the result is requantised to 8 bits)
__device__ __forceinline__ float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

}  // namespace gemm
}  // namespace moe
