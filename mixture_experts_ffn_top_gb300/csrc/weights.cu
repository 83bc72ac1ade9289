// weights.cu -- one-time repack of the caller's Q8_0 (or Q4_K, Q3_K) expert tensors into the
// library-owned layouts the kernels read (load time, not on the hot path).
//
// GGUF Q8_0 stores each 32-block as 34 bytes (fp16 scale + 32 int8), which
// leaves the quants misaligned for vector loads and interleaves them with the
// scales.  Following the SoA repack idea of the pages' int8 MMQ work (#406
// references: "split-K + better-tiled int8 MMQ GEMM ... (SoA repack)"), the
// repack splits every matrix into
//   - int8 quants [rows][K] (16-byte aligned rows) and fp32 scales [rows][K/32]
//     (the fp16 scale widened exactly), read by the matvec path;
//   - for the tensor-core path: the quants again as exact fp16 integers
//     (integers up to 2048 are exact in fp16), gate and up interleaved per 128-row tile
//     (rows 0-63 gate f0..f0+63, rows 64-127 up f0..f0+63) so one MMA tile
//     yields gate and up of the same 64 features; scales transposed to
//     [K/32][rows] so a TMA box of 128 rows x 2 blocks is one copy.
#include <algorithm>

#include "moe_internal.cuh"

#include <vector>

namespace moe {

namespace {

// Stores one decoded 32-block (codes vals, scale) of row r of matrix m (mr = m * rows + r) into
// the matvec layout (q, d: int8 row-major, fp32 [rows][nblk]) and the tensor-core layout (h16
// exact fp16 codes, gate/up interleaved per 128-row tile; dT scales [nblk][rows_out]).
__device__ __forceinline__ void store_block(const int8_t *vals, float scale, int64_t mr, int b, int m, int r,
                                            int rows, int nblk, int8_t *__restrict__ q, float *__restrict__ d,
                                            __half *__restrict__ h16, float *__restrict__ dT, int interleave_gu,
                                            int up_half) {
    const int K = nblk * QK;
    if (q != nullptr) {
        int4 *dst = reinterpret_cast<int4 *>(q + mr * K + (int64_t)b * QK);
        dst[0] = *reinterpret_cast<const int4 *>(vals);
        dst[1] = *reinterpret_cast<const int4 *>(vals + 16);
        d[mr * nblk + b] = scale;
    }
    if (h16 != nullptr) {
        // row inside the tensor-core operand of this matrix
        int64_t rr = r;
        int64_t rows_out = rows;
        if (interleave_gu) {  // gate/up pair: [2*rows] rows, 64-row halves per 128-row tile
            rows_out = 2 * (int64_t)rows;
            rr = (int64_t)(r / 64) * 128 + (up_half ? 64 : 0) + (r % 64);
        }
        __half *dst = h16 + ((int64_t)m * rows_out + rr) * K + (int64_t)b * QK;
#pragma unroll
        for (int j = 0; j < QK; j += 2)
            *reinterpret_cast<__half2 *>(dst + j) = __halves2half2(__int2half_rn(vals[j]), __int2half_rn(vals[j + 1]));
        dT[((int64_t)m * nblk + b) * rows_out + rr] = scale;
    }
}

// Position of the block in the tensor-core operand's transposed scale array, for extra
// per-block arrays laid out like dT (the Q4_K mins).
__device__ __forceinline__ int64_t dT_index(int64_t m, int b, int r, int rows, int nblk, int interleave_gu,
                                            int up_half) {
    int64_t rr = r, rows_out = rows;
    if (interleave_gu) {
        rows_out = 2 * (int64_t)rows;
        rr = (int64_t)(r / 64) * 128 + (up_half ? 64 : 0) + (r % 64);
    }
    return (m * nblk + b) * rows_out + rr;
}

// One thread per 32-block.  src: [nmat][rows][nblk] AoS blocks.
__global__ void repack_kernel(const uint8_t *__restrict__ src, int nmat, int rows, int nblk,
                              int8_t *__restrict__ q, float *__restrict__ d, __half *__restrict__ h16,
                              float *__restrict__ dT, int interleave_gu, int up_half) {
    const int64_t total = (int64_t)nmat * rows * nblk;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t mr = i / nblk;  // matrix * rows + row
        const int b = (int)(i - mr * nblk);
        const int m = (int)(mr / rows);
        const int r = (int)(mr - (int64_t)m * rows);
        const uint8_t *blk = src + i * Q8_0_BYTES;
        const float df = __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
        alignas(16) int8_t vals[QK];
#pragma unroll
        for (int j = 0; j < QK; ++j) vals[j] = (int8_t)blk[2 + j];
        store_block(vals, df, mr, b, m, r, rows, nblk, q, d, h16, dT, interleave_gu, up_half);
    }
}

// Q4_K rows (K/256 super-blocks of 144 bytes each) into the same layouts: quants 0..15 as int8
// (and exact fp16), per-32-block scale d*sc_j and min dmin*m_j as fp32 (both exact: 11-bit
// fp16 times a 6-bit integer).  One thread per 32-wide sub-block.
__global__ void repack_q4k_kernel(const uint8_t *__restrict__ src, int nmat, int rows, int nblk,
                                  int8_t *__restrict__ q, float *__restrict__ d, float *__restrict__ mn,
                                  __half *__restrict__ h16, float *__restrict__ dT, float *__restrict__ mT,
                                  int interleave_gu, int up_half, uint8_t *__restrict__ packed) {
    const int64_t total = (int64_t)nmat * rows * nblk;
    const int64_t row_bytes = (int64_t)(nblk / 8) * Q4_K_BYTES;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t mr = i / nblk;  // matrix * rows + row
        const int b = (int)(i - mr * nblk);
        const int m = (int)(mr / rows);
        const int r = (int)(mr - (int64_t)m * rows);
        const int j = b & 7;  // sub-block inside its super-block
        const uint8_t *blk = src + mr * row_bytes + (int64_t)(b >> 3) * Q4_K_BYTES;
        const float dd = __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(blk[2] | (blk[3] << 8))));
        const uint8_t *s12 = blk + 4;
        int sc, mm;
        if (j < 4) {
            sc = s12[j] & 63;
            mm = s12[j + 4] & 63;
        } else {
            sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
            mm = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
        }
        const float scale = dd * (float)sc, minv = dmin * (float)mm;
        const uint8_t *qs = blk + 16 + 32 * (j >> 1);
        alignas(16) int8_t vals[QK];
#pragma unroll
        for (int l = 0; l < QK; ++l) vals[l] = (int8_t)((j & 1) ? (qs[l] >> 4) : (qs[l] & 15));
        store_block(vals, scale, mr, b, m, r, rows, nblk, q, d, h16, dT, interleave_gu, up_half);
        if (q != nullptr) mn[mr * nblk + b] = minv;
        if (packed != nullptr) {  // byte l: q[l] low nibble, q[l + 16] high nibble
            alignas(16) uint8_t pk[16];
#pragma unroll
            for (int l = 0; l < 16; ++l) pk[l] = (uint8_t)(vals[l] | (vals[l + 16] << 4));
            *reinterpret_cast<int4 *>(packed + (mr * nblk + b) * 16) = *reinterpret_cast<const int4 *>(pk);
        }
        if (h16 != nullptr) mT[dT_index(m, b, r, rows, nblk, interleave_gu, up_half)] = minv;
    }
}

// Q3_K rows (K/256 super-blocks of 110 bytes each) into the Q8_0 layouts.  Value i of a
// super-block is d * s_j * q_i with q_i in [-4, 3] and one signed 6-bit scale s_j per 16 values;
// the kernels work per 32-wide block with one scale, so the repack folds s_j into the codes.
// s_j * q_i spans [-124, 128], one past int8; its negation c_i = -s_j * q_i spans [-128, 124],
// so the codes are stored negated with the block scale -d (exact: the signs cancel in every
// product the kernels form).  One thread per 32-wide block b (sub-blocks 2b', 2b'+1 of its
// super-block, b' = b mod 8):
//   high bit of value 32b' + l: bit b' of byte l;
//   low two bits: bits 2*(b' mod 4) of byte 32 + 32*(b' / 4) + l;
//   6-bit scale field of sub-block j: low 4 bits from nibble j / 8 of byte 96 + j mod 8, high
//   2 bits from bits 2*(j / 4) of byte 104 + j mod 4; s_j = field - 32; fp16 d at byte 108.
__global__ void repack_q3k_kernel(const uint8_t *__restrict__ src, int nmat, int rows, int nblk,
                                  int8_t *__restrict__ q, float *__restrict__ d, __half *__restrict__ h16,
                                  float *__restrict__ dT, int interleave_gu, int up_half) {
    const int64_t total = (int64_t)nmat * rows * nblk;
    const int64_t row_bytes = (int64_t)(nblk / 8) * Q3_K_BYTES;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t mr = i / nblk;  // matrix * rows + row
        const int b = (int)(i - mr * nblk);
        const int m = (int)(mr / rows);
        const int r = (int)(mr - (int64_t)m * rows);
        const int bb = b & 7;  // 32-wide block inside its super-block
        const uint8_t *blk = src + mr * row_bytes + (int64_t)(b >> 3) * Q3_K_BYTES;
        const float dd = __half2float(__ushort_as_half((unsigned short)(blk[108] | (blk[109] << 8))));
        int s[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * bb + h;
            const int lo = (blk[96 + (j & 7)] >> (4 * (j >> 3))) & 15;
            const int hi = (blk[104 + (j & 3)] >> (2 * (j >> 2))) & 3;
            s[h] = (lo | (hi << 4)) - 32;
        }
        const uint8_t *qs = blk + 32 + 32 * (bb >> 2);
        const int shift = 2 * (bb & 3);
        alignas(16) int8_t vals[QK];
#pragma unroll
        for (int l = 0; l < QK; ++l) {
            const int low = (qs[l] >> shift) & 3;
            const int qv = ((blk[l] >> bb) & 1) ? low : low - 4;
            vals[l] = (int8_t)(-s[l >> 4] * qv);
        }
        store_block(vals, -dd, mr, b, m, r, rows, nblk, q, d, h16, dT, interleave_gu, up_half);
    }
}

int repack(int wfmt, const void *src, int nmat, int rows, int K, int8_t *q, float *d, float *mn, __half *h16,
           float *dT, float *mT, uint8_t *packed, int interleave, int up_half, cudaStream_t s) {
    int64_t total = (int64_t)nmat * rows * (K / QK);
    if (total == 0) return MOE_OK;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)std::max(1, device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (wfmt == MOE_WFMT_Q4_K)
        repack_q4k_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(src), nmat, rows, K / QK, q, d,
                                                           mn, h16, dT, mT, interleave, up_half, packed);
    else if (wfmt == MOE_WFMT_Q3_K)
        repack_q3k_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(src), nmat, rows, K / QK, q, d,
                                                           h16, dT, interleave, up_half);
    else
        repack_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(src), nmat, rows, K / QK, q, d,
                                                       h16, dT, interleave, up_half);
    return launch_status();
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Sizes of one weight set's arrays; carve == true assigns pointers from base.
static size_t layout_set(WeightSet &ws, int nexp, int D, int F, bool tensor, int wfmt, char *base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align256(bytes);
        return base ? base + o : nullptr;
    };
    const size_t gu = (size_t)nexp * F * D, dn = (size_t)nexp * D * F;
    ws.F = F;
    ws.rows_gu = 2 * F;
    ws.gate_q = (int8_t *)take(gu);
    ws.up_q = (int8_t *)take(gu);
    ws.gate_d = (float *)take(gu / QK * sizeof(float));
    ws.up_d = (float *)take(gu / QK * sizeof(float));
    ws.down_q = (int8_t *)take(dn);
    ws.down_d = (float *)take(dn / QK * sizeof(float));
    const bool mins = wfmt == MOE_WFMT_Q4_K;
    if (mins) {
        ws.gate_m = (float *)take(gu / QK * sizeof(float));
        ws.up_m = (float *)take(gu / QK * sizeof(float));
        ws.down_m = (float *)take(dn / QK * sizeof(float));
        ws.gate_p = (uint8_t *)take(gu / 2);
        ws.up_p = (uint8_t *)take(gu / 2);
        ws.down_p = (uint8_t *)take(dn / 2);
    }
    if (tensor) {
        ws.gu16 = (__half *)take(2 * gu * sizeof(__half));
        ws.gu_dT = (float *)take(2 * gu / QK * sizeof(float));
        ws.dn16 = (__half *)take(dn * sizeof(__half));
        ws.dn_dT = (float *)take(dn / QK * sizeof(float));
        if (mins) {
            ws.gu_mT = (float *)take(2 * gu / QK * sizeof(float));
            ws.dn_mT = (float *)take(dn / QK * sizeof(float));
        }
    }
    return off;
}

int repack_weights(moe_weights_s *w, const void *gate, const void *up, const void *down, const void *sh_gate,
                   const void *sh_up, const void *sh_down, cudaStream_t s) {
    const int E = w->E, D = w->D, F = w->F, Fs = w->Fs;
    const bool tensor = w->tensor_ok;
    const int wf = w->wfmt;
    size_t r_bytes = layout_set(w->routed, E, D, F, tensor, wf, nullptr);
    size_t s_bytes = Fs ? layout_set(w->shared, 1, D, Fs, tensor, wf, nullptr) : 0;
    char *arena = nullptr;
    if (cudaMalloc(&arena, r_bytes + s_bytes) != cudaSuccess) return MOE_ERR_CUDA;
    w->bytes = r_bytes + s_bytes;
    layout_set(w->routed, E, D, F, tensor, wf, arena);
    if (Fs) layout_set(w->shared, 1, D, Fs, tensor, wf, arena + r_bytes);
    // the arena start doubles as the handle's allocation
    w->routed_arena_ = arena;
    auto sets = [&](WeightSet &ws, int nexp, int Fx, const void *g, const void *u, const void *dn) {
        int rc = repack(wf, g, nexp, Fx, D, ws.gate_q, ws.gate_d, ws.gate_m, ws.gu16, ws.gu_dT, ws.gu_mT, ws.gate_p, 1,
                        0, s);
        if (!rc)
            rc = repack(wf, u, nexp, Fx, D, ws.up_q, ws.up_d, ws.up_m, ws.gu16, ws.gu_dT, ws.gu_mT, ws.up_p, 1, 1, s);
        if (!rc)
            rc = repack(wf, dn, nexp, D, Fx, ws.down_q, ws.down_d, ws.down_m, ws.dn16, ws.dn_dT, ws.dn_mT, ws.down_p, 0,
                        0, s);
        return rc;
    };
    int rc = sets(w->routed, E, F, gate, up, down);
    if (!rc && Fs) rc = sets(w->shared, 1, Fs, sh_gate, sh_up, sh_down);
    if (!rc) rc = cuda_status(cudaStreamSynchronize(s));
    return rc;
}

void free_weights(moe_weights_s *w) {
    if (w->routed_arena_) cudaFree(w->routed_arena_);
    w->routed_arena_ = nullptr;
}

}  // namespace moe
