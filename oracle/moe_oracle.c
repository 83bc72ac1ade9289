/*
 * moe_oracle.c -- plain CPU oracle for the batched routed-MoE FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm use it.  It shares no code, header, table or
 * helper with the CUDA library (mixture_experts_ffn_top_gb300/csrc).
 *
 * What it computes follows the four SharpInference issue pages:
 *   - "Carnice prefill toward llama.cpp 676 t/s" (#388), the per-token
 *     breakdown table (router row: matvec + softmax + top-k + shexp-gate) and
 *     "Remaining levers" item 1 (router matvec norm[N x embDim] x
 *     routerW[numExperts x embDim], the expStart/expTokI/expTokK CSR);
 *   - "full-offload MoE decode ~3.4x behind llama.cpp" (#408), "Hypothesis"
 *     (64 experts / 8 active, norm_topk_prob=false) and lever 2 (Q8_1
 *     activations, int8 dot products);
 *   - "batched int8-MMQ trunk prefill gated off for MoE" (#406), "The work"
 *     item 2 (gather tokens per expert -> per-expert GEMM-N -> scatter) and
 *     the references list (Q8_0 MMQ);
 *   - issue #129 (batched weighted scatter-reduce), intro and "Scope": the
 *     unweighted down-partials are reduced per token in top-k slot order
 *     k = 0..na-1 with the per-(token,slot) weights (Clear, AddScaledInPlace
 *     per k, then AddInPlace(shared)).
 *
 * Precision: every reduction whose precision the pages leave open is done
 * in double and rounded to fp32 once.  Two steps are fp32 by definition:
 *   - the Q8_0/Q8_1 block quantiser (the GGUF block formats are defined with
 *     an fp32 scale computation, an fp16 stored scale and roundf);
 *   - the combine, which must reproduce an fp32 host reduce bit for bit in a
 *     fixed order; AddScaledInPlace is read as a fused multiply-add.
 * Build with -ffp-contract=off (and never -ffast-math) so that the compiler
 * fuses nothing the code does not fuse explicitly.
 *
 * Parity pins: see tests/test_oracle_*.py.  Every function below is pinned
 * against an independent fact (a closed form, brute force, a library routine
 * on a special case, or a hand-computed fixture).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32         /* elements per Q8 block */
#define Q8_0_BYTES 34 /* fp16 scale + 32 int8 quants */

/* ------------------------------------------------------------------------
 * IEEE 754 binary16 conversions, written from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).
 * ---------------------------------------------------------------------- */
float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    float v;
    if (ex == 0)
        v = ldexpf((float)frac, -24); /* subnormal: frac * 2^-24 */
    else if (ex == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + frac), ex - 25); /* (1.frac) * 2^(ex-15) */
    return sign ? -v : v;
}

/* Round to nearest, ties to even. */
uint16_t oracle_float_to_half(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    float a = fabsf(f);
    if (isnan(f))
        return 0x7e00;
    if (a >= 65520.0f) /* halfway between 65504 and 2^16 rounds to even: inf */
        return sign | 0x7c00;
    if (a < 0x1p-14f) {
        /* subnormal range: units of 2^-24; a result of 1024 is the smallest
         * normal number and encodes correctly as exponent 1, fraction 0 */
        float r = rintf(a * 0x1p24f);
        return sign | (uint16_t)r;
    }
    int e2;
    frexpf(a, &e2);   /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;   /* a in [2^E, 2^(E+1)) */
    float r = rintf(ldexpf(a, 10 - E)); /* in [1024, 2048] */
    uint32_t bits = ((uint32_t)(E + 15) << 10) + ((uint32_t)r - 1024u);
    return sign | (uint16_t)bits; /* r == 2048 carries into the exponent */
}

/* ------------------------------------------------------------------------
 * Q8 block quantiser (GGUF Q8_0 / Q8_1 rule), fp32 arithmetic:
 *   amax = max |x_i|; d = amax / 127; id = d != 0 ? 1/d : 0;
 *   q_i = roundf(x_i * id)  (half away from zero);
 *   stored scale = fp16(d) (RNE); Q8_1 also stores fp16(d * sum_i q_i).
 * Quants are computed from the fp32 d; dequantisation uses the fp16 d.
 * The pages name these formats ("Q8_0 MMQ", "Q8_1 / dp4a expert matvec")
 * without restating them; this is the standard definition.
 * ---------------------------------------------------------------------- */
void oracle_quantize_q8_1(const float *x, int64_t nblocks, int8_t *q, uint16_t *d16, uint16_t *s16)
{
    for (int64_t b = 0; b < nblocks; ++b) {
        const float *xb = x + b * QK;
        float amax = 0.0f;
        for (int i = 0; i < QK; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax)
                amax = a;
        }
        float d = amax / 127.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        int sum = 0;
        for (int i = 0; i < QK; ++i) {
            float v = xb[i] * id;
            int qi = (int)roundf(v);
            q[b * QK + i] = (int8_t)qi;
            sum += qi;
        }
        d16[b] = oracle_float_to_half(d);
        if (s16)
            s16[b] = oracle_float_to_half(d * (float)sum);
    }
}

/* ------------------------------------------------------------------------
 * Router (#388 breakdown table, "router" row; levers item 1):
 *   logits[t,e] = sum_d x[t,d] * W_r[e,d], d ascending, in double, -> fp32.
 * The shared-expert gate logit g_t = sum_d x[t,d] * w_sg[d] is the same
 * computation with one row (E = 1).
 * ---------------------------------------------------------------------- */
void oracle_router_logits(const float *x, const float *W, int64_t N, int D, int E, float *logits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < N; ++t) {
        const float *xt = x + t * D;
        for (int e = 0; e < E; ++e) {
            const float *we = W + (int64_t)e * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)xt[d] * (double)we[d];
            logits[t * E + e] = (float)acc;
        }
    }
}

/* ------------------------------------------------------------------------
 * Softmax over all E experts, then top-k (#388 router row "softmax + top-k";
 * #408 "Hypothesis": norm_topk_prob).
 *   m = max_e l_e;  p_e = exp(l_e - m) / sum_e' exp(l_e' - m)   (double)
 *   slots 0..k-1 = experts in order of decreasing logit, ties broken to the
 *   lower expert index (selection on the logit is selection on p, since exp
 *   is increasing, without exp-rounding ties);
 *   w[t,s] = p_sel            when norm_topk_prob = 0,
 *          = p_sel / sum_sel p when norm_topk_prob = 1;   rounded to fp32.
 * p_out (nullable) receives fp32(p) for every expert.
 * ---------------------------------------------------------------------- */
void oracle_softmax_topk(const float *logits, int64_t N, int E, int k, int norm,
                         int32_t *idx, float *w, float *p_out)
{
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        unsigned char *taken = (unsigned char *)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < N; ++t) {
            const float *l = logits + t * E;
            double m = -INFINITY;
            for (int e = 0; e < E; ++e)
                if ((double)l[e] > m)
                    m = (double)l[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) {
                p[e] = exp((double)l[e] - m);
                z += p[e];
            }
            for (int e = 0; e < E; ++e) {
                p[e] = p[e] / z;
                if (p_out)
                    p_out[t * E + e] = (float)p[e];
            }
            memset(taken, 0, (size_t)E);
            double psel = 0.0;
            for (int s = 0; s < k; ++s) {
                int best = -1;
                for (int e = 0; e < E; ++e)
                    if (!taken[e] && (best < 0 || l[e] > l[best]))
                        best = e; /* strict '>' keeps the lower index on ties */
                taken[best] = 1;
                idx[t * k + s] = best;
                psel += p[best];
            }
            for (int s = 0; s < k; ++s) {
                double ps = p[idx[t * k + s]];
                w[t * k + s] = (float)(norm ? ps / psel : ps);
            }
        }
        free(p);
        free(taken);
    }
}

/* Shared-expert gate scale s_t = sigmoid(g_t) (#388 router row "shexp-gate"). */
void oracle_sigmoid(const float *g, int64_t N, float *s)
{
    for (int64_t t = 0; t < N; ++t)
        s[t] = (float)(1.0 / (1.0 + exp(-(double)g[t])));
}

/* ------------------------------------------------------------------------
 * Expert bucketing into a CSR (#388 levers item 1: expStart/expTokI/expTokK).
 * A counting sort of the N*k (token, slot) pairs by expert:
 *   cnt[e] = #{(t,s) : idx[t,s] = e};  expStart = exclusive scan of cnt;
 *   entries are filled in order t = 0..N-1, s = 0..k-1, so each segment is
 *   ascending in t.  expTokI[j] = t, expTokK[j] = s.
 * Returns 0, or -1 on an expert index out of range, or -2 when a token
 * selects the same expert twice.
 * ---------------------------------------------------------------------- */
int oracle_bucket(const int32_t *idx, int64_t N, int k, int E,
                  int32_t *expStart, int32_t *expTokI, int32_t *expTokK)
{
    int64_t *fill = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    for (int64_t t = 0; t < N; ++t)
        for (int s = 0; s < k; ++s) {
            int e = idx[t * k + s];
            if (e < 0 || e >= E) {
                free(fill);
                return -1;
            }
            for (int s2 = 0; s2 < s; ++s2)
                if (idx[t * k + s2] == e) {
                    free(fill);
                    return -2;
                }
            fill[e + 1] += 1;
        }
    for (int e = 0; e < E; ++e)
        fill[e + 1] += fill[e];
    for (int e = 0; e <= E; ++e)
        expStart[e] = (int32_t)fill[e];
    for (int64_t t = 0; t < N; ++t)
        for (int s = 0; s < k; ++s) {
            int e = idx[t * k + s];
            int64_t j = fill[e]++;
            expTokI[j] = (int32_t)t;
            expTokK[j] = s;
        }
    free(fill);
    return 0;
}

/* ------------------------------------------------------------------------
 * Q8_0 x Q8_1 row dot, per 32-block (#406 references: Q8_0 MMQ; #408 lever 2:
 * Q8_1 activations, int8 dot products):
 *   isum_b = sum_{i in b} qw_i * qa_i   (exact int32)
 *   result = sum_b fp16(dw_b) * fp16(da_b) * isum_b, accumulated in double
 * (each block term is exact in double: 11 + 11 + 20 significant bits).
 * w_row points at the row's first Q8_0 block (34 bytes each: fp16 d, 32 q).
 * ---------------------------------------------------------------------- */
static inline int32_t block_isum(const int8_t *a, const int8_t *b)
{
    int32_t s = 0;
    for (int i = 0; i < QK; ++i)
        s += (int32_t)a[i] * (int32_t)b[i];
    return s;
}

static inline uint16_t load_u16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8)); /* little-endian fp16 field */
}

static double q8_row_dot(const uint8_t *w_row, const int8_t *aq, const uint16_t *ad16, int nblk)
{
    double acc = 0.0;
    for (int b = 0; b < nblk; ++b) {
        const uint8_t *blk = w_row + (size_t)b * Q8_0_BYTES;
        int32_t isum = block_isum((const int8_t *)(blk + 2), aq + b * QK);
        acc += (double)oracle_half_to_float(load_u16(blk)) *
               (double)oracle_half_to_float(ad16[b]) * (double)isum;
    }
    return acc;
}

/* int32 block dots of one weight row against one activation row: the
 * bit-exact quantity of the GEMM (exported for the block-dot pins). */
void oracle_block_dots(const uint8_t *w_row, const int8_t *aq, int nblk, int32_t *out)
{
    for (int b = 0; b < nblk; ++b)
        out[b] = block_isum((const int8_t *)(w_row + (size_t)b * Q8_0_BYTES + 2), aq + b * QK);
}

/* The int32 dot of block `block` for every CSR entry j and every weight row r of
 * the entry's expert, Q8_0 weights: out[j][r] = sum over the block's 32 values of
 * q_w[e][r] * q_a[row of j].  W is [E][rows][K/32 blocks of 34 bytes]; the
 * activation row of entry j is act[sel[j]] (sel = expTokI: token rows of x_q) or
 * act[j] when sel is NULL (h_q, stored in entry order).  Entries are independent,
 * so they are split across threads; each dot is one serial integer sum. */
void oracle_block_dots_csr(const uint8_t *W, int E, int rows, int K, const int8_t *act,
                           const int32_t *expStart, const int32_t *sel, int block, int32_t *out)
{
    const int nblk = K / QK;
    const size_t rbytes = (size_t)nblk * Q8_0_BYTES;
    const int64_t n = expStart[E];
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t j = 0; j < n; ++j) {
        int e = 0;
        while (e + 1 < E && expStart[e + 1] <= j) ++e;
        const int64_t a = sel ? (int64_t)sel[j] : j;
        const int8_t *x = act + a * (int64_t)K + (int64_t)block * QK;
        for (int r = 0; r < rows; ++r) {
            const uint8_t *blk = W + ((size_t)e * rows + r) * rbytes + (size_t)block * Q8_0_BYTES;
            out[j * rows + r] = block_isum((const int8_t *)(blk + 2), x);
        }
    }
}

/* ------------------------------------------------------------------------
 * Q4_K weights (the K-quant the pages' MMQ work names next to Q8_0: #406
 * references "Q8_0/Q4_K MMQ"; its layout is the GGUF one, which the pages do
 * not spell out).  A super-block of QK_K = 256 values is 144 bytes: fp16 d,
 * fp16 dmin, 12 bytes holding eight 6-bit sub-block scales sc_j and mins m_j,
 * 128 bytes of 4-bit quants q in [0, 15].  Value i of sub-block j:
 *   w = d * sc_j * q_i - dmin * m_j.
 * Packing of the 12 bytes: for j < 4, sc_j and m_j are the low 6 bits of
 * bytes j and j + 4; for j >= 4, the low (high) nibble of byte j + 4 gives
 * the low 4 bits of sc_j (m_j) and the top 2 bits of byte j - 4 (byte j) its
 * high 2 bits.  Quants: the 64 values of sub-blocks 2g and 2g + 1 share 32
 * bytes, sub-block 2g in the low nibbles, 2g + 1 in the high ones.
 * Dot with a Q8_1 row, per 32-wide sub-block b (exact int32 isum_b as for
 * Q8_0, plus the activation's code sum xsum_b for the min term):
 *   result = sum_b fp16(da_b) * (d * sc_b * isum_b - dmin * m_b * xsum_b)
 * accumulated in double (each term is exact in double).
 * ---------------------------------------------------------------------- */
#define QK_K 256
#define Q4_K_BYTES 144
enum { FMT_Q8_0 = 0, FMT_Q4_K = 1 };

static void q4_k_scale_min(const uint8_t *s12, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s12[j] & 63;
        *m = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
        *m = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

static void q4_k_quants(const uint8_t *qs, int j, int8_t *q)
{
    const uint8_t *p = qs + 32 * (j / 2);
    for (int l = 0; l < QK; ++l)
        q[l] = (int8_t)((j & 1) ? (p[l] >> 4) : (p[l] & 15));
}

static double q4_k_row_dot(const uint8_t *w_row, const int8_t *aq, const uint16_t *ad16, int K)
{
    double acc = 0.0;
    for (int sb = 0; sb < K / QK_K; ++sb) {
        const uint8_t *blk = w_row + (size_t)sb * Q4_K_BYTES;
        double d = oracle_half_to_float(load_u16(blk));
        double dmin = oracle_half_to_float(load_u16(blk + 2));
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            int8_t q[QK];
            q4_k_scale_min(blk + 4, j, &sc, &m);
            q4_k_quants(blk + 16, j, q);
            int b = sb * 8 + j;
            int32_t isum = block_isum(q, aq + b * QK);
            int32_t xsum = 0;
            for (int l = 0; l < QK; ++l)
                xsum += aq[b * QK + l];
            acc += (double)oracle_half_to_float(ad16[b]) * (d * sc * (double)isum - dmin * m * (double)xsum);
        }
    }
    return acc;
}

/* Dequantised Q4_K row (K values, each rounded once to fp32), for the pins. */
void oracle_q4_k_dequant(const uint8_t *w_row, int K, float *out)
{
    for (int sb = 0; sb < K / QK_K; ++sb) {
        const uint8_t *blk = w_row + (size_t)sb * Q4_K_BYTES;
        double d = oracle_half_to_float(load_u16(blk));
        double dmin = oracle_half_to_float(load_u16(blk + 2));
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            int8_t q[QK];
            q4_k_scale_min(blk + 4, j, &sc, &m);
            q4_k_quants(blk + 16, j, q);
            for (int l = 0; l < QK; ++l)
                out[sb * QK_K + j * QK + l] = (float)(d * sc * q[l] - dmin * m);
        }
    }
}

/* int32 block dots of a Q4_K row (quants 0..15) against an activation row. */
void oracle_block_dots_q4_k(const uint8_t *w_row, const int8_t *aq, int K, int32_t *out)
{
    for (int sb = 0; sb < K / QK_K; ++sb)
        for (int j = 0; j < 8; ++j) {
            int8_t q[QK];
            q4_k_quants(w_row + (size_t)sb * Q4_K_BYTES + 16, j, q);
            out[sb * 8 + j] = block_isum(q, aq + (sb * 8 + j) * QK);
        }
}

/* ------------------------------------------------------------------------
 * Q3_K weights (the Carnice prefill page, #388 "Key references", names a
 * Q3_K GPU expert kernel and Q3_K x Q8 CPU dots: the routed experts of that
 * model are Q3_K; the layout is the GGUF one, which the pages do not spell
 * out).  A super-block of QK_K = 256 values is 110 bytes:
 *   bytes   0..31  hmask: bit (i / 32) of byte (i % 32) is value i's high bit h_i;
 *   bytes  32..95  qs: bits 2*((i % 128) / 32) .. +1 of byte 32*(i / 128) + i % 32
 *                  are value i's low two bits l_i;
 *   bytes  96..107 sixteen 6-bit scales, one per 16-wide sub-block j = i / 16:
 *                  low 4 bits = nibble (j / 8) of byte j % 8, high 2 bits =
 *                  bits 2*(j / 4) .. +1 of byte 8 + j % 4; s_j = that - 32;
 *   bytes 108..109 fp16 d.
 * q_i = l_i - 4 when h_i is clear, l_i when it is set (q in [-4, 3]), and
 *   w_i = d * s_j * q_i.
 * Dot with a Q8_1 row, per 32-wide activation block b (sub-blocks 2b, 2b+1):
 *   result = sum_b fp16(da_b) * d * (s_2b * isum_2b + s_2b+1 * isum_2b+1)
 * with isum_j the exact int32 dot of sub-block j's q with the activation
 * codes; accumulated in double (each term is exact in double).
 * ---------------------------------------------------------------------- */
#define Q3_K_BYTES 110
enum { FMT_Q3_K = 2 };

static int q3_k_scale(const uint8_t *blk, int j)
{
    const uint8_t *s12 = blk + 96;
    int lo = (s12[j % 8] >> (4 * (j / 8))) & 15;
    int hi = (s12[8 + j % 4] >> (2 * (j / 4))) & 3;
    return (lo | (hi << 4)) - 32;
}

static int q3_k_quant(const uint8_t *blk, int i)
{
    int l = (blk[32 + 32 * (i / 128) + i % 32] >> (2 * ((i % 128) / 32))) & 3;
    int h = (blk[i % 32] >> (i / 32)) & 1;
    return h ? l : l - 4;
}

/* sum over 32-wide block b of one super-block: s_j-weighted int dots (exact). */
static int64_t q3_k_block_sisum(const uint8_t *blk, int b, const int8_t *aq_sb)
{
    int64_t sisum = 0;
    for (int half = 0; half < 2; ++half) {
        int j = 2 * b + half;
        int32_t isum = 0;
        for (int l = 0; l < 16; ++l)
            isum += q3_k_quant(blk, 16 * j + l) * (int32_t)aq_sb[16 * j + l];
        sisum += (int64_t)q3_k_scale(blk, j) * isum;
    }
    return sisum;
}

static double q3_k_row_dot(const uint8_t *w_row, const int8_t *aq, const uint16_t *ad16, int K)
{
    double acc = 0.0;
    for (int sb = 0; sb < K / QK_K; ++sb) {
        const uint8_t *blk = w_row + (size_t)sb * Q3_K_BYTES;
        double d = oracle_half_to_float(load_u16(blk + 108));
        for (int b = 0; b < 8; ++b) {
            int64_t sisum = q3_k_block_sisum(blk, b, aq + sb * QK_K);
            acc += (double)oracle_half_to_float(ad16[sb * 8 + b]) * d * (double)sisum;
        }
    }
    return acc;
}

/* Dequantised Q3_K row (K values, each rounded once to fp32), for the pins. */
void oracle_q3_k_dequant(const uint8_t *w_row, int K, float *out)
{
    for (int sb = 0; sb < K / QK_K; ++sb) {
        const uint8_t *blk = w_row + (size_t)sb * Q3_K_BYTES;
        double d = oracle_half_to_float(load_u16(blk + 108));
        for (int i = 0; i < QK_K; ++i)
            out[sb * QK_K + i] = (float)(d * q3_k_scale(blk, i / 16) * q3_k_quant(blk, i));
    }
}

/* Per 32-wide block of a Q3_K row: s_2b * isum_2b + s_2b+1 * isum_2b+1 (int32). */
void oracle_block_dots_q3_k(const uint8_t *w_row, const int8_t *aq, int K, int32_t *out)
{
    for (int sb = 0; sb < K / QK_K; ++sb)
        for (int b = 0; b < 8; ++b)
            out[sb * 8 + b] = (int32_t)q3_k_block_sisum(w_row + (size_t)sb * Q3_K_BYTES, b, aq + sb * QK_K);
}

static size_t row_bytes(int fmt, int K)
{
    if (fmt == FMT_Q4_K)
        return (size_t)(K / QK_K) * Q4_K_BYTES;
    if (fmt == FMT_Q3_K)
        return (size_t)(K / QK_K) * Q3_K_BYTES;
    return (size_t)(K / QK) * Q8_0_BYTES;
}

static double row_dot(int fmt, const uint8_t *w_row, const int8_t *aq, const uint16_t *ad16, int K)
{
    if (fmt == FMT_Q4_K)
        return q4_k_row_dot(w_row, aq, ad16, K);
    if (fmt == FMT_Q3_K)
        return q3_k_row_dot(w_row, aq, ad16, K);
    return q8_row_dot(w_row, aq, ad16, K / QK);
}

/* ------------------------------------------------------------------------
 * SwiGLU expert, gate/up half, for one activation row (#129 intro: the
 * routed-expert gate/up/down GEMMs; #406 "The work" item 2):
 *   g_r = <W_g[r], x_q>,  u_r = <W_u[r], x_q>   (q8_row_dot, double)
 *   h_r = fp32( SiLU(g_r) * u_r ),  SiLU(z) = z / (1 + exp(-z))
 * then h -> Q8_1 (oracle_quantize_q8_1).  Optional g/u outputs (double).
 * Wg, Wu: [F rows][D/32 blocks] Q8_0.
 * ---------------------------------------------------------------------- */
static void expert_gate_up_row(int fmt, const uint8_t *Wg, const uint8_t *Wu, int D, int F,
                               const int8_t *xq, const uint16_t *xd16,
                               float *h, int8_t *hq, uint16_t *hd16, double *g_out, double *u_out)
{
    size_t rb = row_bytes(fmt, D);
    for (int r = 0; r < F; ++r) {
        double g = row_dot(fmt, Wg + r * rb, xq, xd16, D);
        double u = row_dot(fmt, Wu + r * rb, xq, xd16, D);
        if (g_out)
            g_out[r] = g;
        if (u_out)
            u_out[r] = u;
        h[r] = (float)((g / (1.0 + exp(-g))) * u);
    }
    oracle_quantize_q8_1(h, F / QK, hq, hd16, NULL);
}

/* Down half: y_c = <W_d[c], h_q> in double, c = 0..D-1.  Wd: [D] rows of K = F. */
static void expert_down_row(int fmt, const uint8_t *Wd, int D, int F, const int8_t *hq, const uint16_t *hd16,
                            double *y)
{
    size_t rb = row_bytes(fmt, F);
    for (int c = 0; c < D; ++c)
        y[c] = row_dot(fmt, Wd + c * rb, hq, hd16, F);
}

/* Exported single-row pieces, for the pins (fmt: 0 Q8_0, 1 Q4_K, 2 Q3_K). */
void oracle_expert_gate_up_fmt(int fmt, const uint8_t *Wg, const uint8_t *Wu, int D, int F,
                               const int8_t *xq, const uint16_t *xd16,
                               float *h, int8_t *hq, uint16_t *hd16, double *g, double *u)
{
    expert_gate_up_row(fmt, Wg, Wu, D, F, xq, xd16, h, hq, hd16, g, u);
}

void oracle_expert_down_fmt(int fmt, const uint8_t *Wd, int D, int F, const int8_t *hq, const uint16_t *hd16,
                            double *y)
{
    expert_down_row(fmt, Wd, D, F, hq, hd16, y);
}

/* ------------------------------------------------------------------------
 * Grouped expert FFN over the CSR (#406 "The work" item 2: gather tokens per
 * expert -> per-expert GEMM-N -> scatter).  For every entry j of expert e's
 * segment, token t = expTokI[j], slot s = expTokK[j]:
 *   h_q[j]                   = Q8_1(SiLU(W_g[e] x_q[t]) * (W_u[e] x_q[t]))
 *   partials[t*k + s, 0..D)  = fp32(W_d[e] h_q[j])         (unweighted)
 * gate/up: [E][F][D/32] Q8_0; down: [E][D][F/32] Q8_0.
 * hq/hd16 (nullable) receive the segment-ordered requantised activations.
 * ---------------------------------------------------------------------- */
void oracle_grouped_ffn_fmt(int fmt, const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                            int E, int D, int F, const int8_t *xq, const uint16_t *xd16,
                            const int32_t *expStart, const int32_t *expTokI, const int32_t *expTokK,
                            int k, float *partials, int8_t *hq_out, uint16_t *hd16_out)
{
    size_t gu_bytes = (size_t)F * row_bytes(fmt, D); /* one expert's gate (or up) */
    size_t dn_bytes = (size_t)D * row_bytes(fmt, F);
    int64_t total = expStart[E];
#pragma omp parallel
    {
        float *h = (float *)malloc(sizeof(float) * (size_t)F);
        int8_t *hq = (int8_t *)malloc((size_t)F);
        uint16_t *hd = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(F / QK));
        double *y = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t j = 0; j < total; ++j) {
            int e = 0;
            while (expStart[e + 1] <= j) /* segment owning entry j */
                ++e;
            int64_t t = expTokI[j];
            int s = expTokK[j];
            expert_gate_up_row(fmt, gate + e * gu_bytes, up + e * gu_bytes, D, F,
                               xq + t * D, xd16 + t * (D / QK), h, hq, hd, NULL, NULL);
            if (hq_out) {
                memcpy(hq_out + j * F, hq, (size_t)F);
                memcpy(hd16_out + j * (F / QK), hd, sizeof(uint16_t) * (size_t)(F / QK));
            }
            expert_down_row(fmt, down + e * dn_bytes, D, F, hq, hd, y);
            float *dst = partials + (t * k + s) * (int64_t)D;
            for (int c = 0; c < D; ++c)
                dst[c] = (float)y[c];
        }
        free(h);
        free(hq);
        free(hd);
        free(y);
    }
}

/* ------------------------------------------------------------------------
 * Shared expert over all N tokens, scaled by its gate (#129 "Scope": the
 * optionally batched Phase 1 shared expert; #388 router row: shexp-gate):
 *   S[t,c] = fp32( s_t * y_c ),  y = W_sd Q8_1(SiLU(W_sg x_q[t]) * (W_su x_q[t]))
 * sg/su: [Fs][D/32]; sd: [D][Fs/32].
 * ---------------------------------------------------------------------- */
void oracle_shared_expert_fmt(int fmt, const uint8_t *sg, const uint8_t *su, const uint8_t *sd, int D, int Fs,
                              const int8_t *xq, const uint16_t *xd16, const float *s, int64_t N,
                              float *S, int8_t *hq_out, uint16_t *hd16_out)
{
#pragma omp parallel
    {
        float *h = (float *)malloc(sizeof(float) * (size_t)Fs);
        int8_t *hq = (int8_t *)malloc((size_t)Fs);
        uint16_t *hd = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(Fs / QK));
        double *y = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < N; ++t) {
            expert_gate_up_row(fmt, sg, su, D, Fs, xq + t * D, xd16 + t * (D / QK), h, hq, hd, NULL, NULL);
            if (hq_out) {
                memcpy(hq_out + t * Fs, hq, (size_t)Fs);
                memcpy(hd16_out + t * (Fs / QK), hd, sizeof(uint16_t) * (size_t)(Fs / QK));
            }
            expert_down_row(fmt, sd, D, Fs, hq, hd, y);
            for (int c = 0; c < D; ++c)
                S[t * D + c] = (float)((double)s[t] * y[c]);
        }
        free(h);
        free(hq);
        free(hd);
        free(y);
    }
}

/* ------------------------------------------------------------------------
 * Combine (#129 "Scope"): per token row, Clear, then for k = 0..na-1
 * AddScaledInPlace(acc, partial[t*na + k], w[t,k]) -- one fp32 fused
 * multiply-add per element -- then AddInPlace(shared) when present:
 *   acc = +0.0f; for s: acc = fmaf(w[t,s], partial[t*k+s, c], acc);
 *   if (S) acc = acc + S[t,c];   out[t,c] = acc.
 * ---------------------------------------------------------------------- */
void oracle_combine(const float *partials, const float *w, const float *S, int64_t N, int k, int D,
                    float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < N; ++t)
        for (int c = 0; c < D; ++c) {
            float acc = 0.0f;
            for (int s = 0; s < k; ++s)
                acc = fmaf(w[t * k + s], partials[(t * k + s) * (int64_t)D + c], acc);
            if (S)
                acc = acc + S[t * D + c];
            out[t * D + c] = acc;
        }
}

/* ------------------------------------------------------------------------
 * Combine with the residual add of the pages' host combine ("Carnice prefill
 * toward llama.cpp 676 t/s", #388, "Dead ends": the per-layer combine is
 * (routed + shared*scale) + resid): the combine above, then one more fp32 add
 * of the residual row R[t]:
 *   out[t,c] = (acc + S[t,c]) + R[t,c].
 * ---------------------------------------------------------------------- */
void oracle_combine_residual(const float *partials, const float *w, const float *S, const float *R, int64_t N,
                             int k, int D, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < N; ++t)
        for (int c = 0; c < D; ++c) {
            float acc = 0.0f;
            for (int s = 0; s < k; ++s)
                acc = fmaf(w[t * k + s], partials[(t * k + s) * (int64_t)D + c], acc);
            if (S)
                acc = acc + S[t * D + c];
            acc = acc + R[t * D + c];
            out[t * D + c] = acc;
        }
}

/* ------------------------------------------------------------------------
 * The combine with the residual, then the next layer's input norm.  The pages
 * feed the router a normalised activation ("Carnice prefill toward llama.cpp
 * 676 t/s", #388, "Remaining levers" item 1: norm[N x embDim] x routerW) and
 * chain the layers through the residual stream (item 2: layer L+1's trunk
 * starts with its norm of layer L's combine output); they do not spell the
 * norm out.  Read as RMSNorm with a per-column weight gamma and an epsilon
 * (the norm of the OLMoE and Qwen3-MoE layer families the pages run): per
 * token row t,
 *   out[t,c]    = the combine with residual above (fp32, fixed order);
 *   ms          = (sum over c of out[t,c]^2) / D                  (double)
 *   normed[t,c] = out[t,c] * (1 / sqrt(ms + eps)) * gamma[c]       (double,
 *                 rounded to fp32 once).
 * ---------------------------------------------------------------------- */
void oracle_combine_residual_rmsnorm(const float *partials, const float *w, const float *S, const float *R,
                                     const float *gamma, double eps, int64_t N, int k, int D, float *out,
                                     float *normed)
{
    oracle_combine_residual(partials, w, S, R, N, k, D, out);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < N; ++t) {
        const float *o = out + t * D;
        double ss = 0.0;
        for (int c = 0; c < D; ++c)
            ss += (double)o[c] * (double)o[c];
        double r = 1.0 / sqrt(ss / (double)D + eps);
        for (int c = 0; c < D; ++c)
            normed[t * D + c] = (float)((double)o[c] * r * (double)gamma[c]);
    }
}

/* Threads the OpenMP runtime will use (reported beside oracle timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
