// topk_token.cuh -- routing of one token by one warp: softmax over all E router logits, top-k by
// logit (ties to the lower expert index), the selected probabilities (divided by their sum with
// norm_topk_prob) and the shared-expert gate sigma(g) ("Carnice prefill toward llama.cpp 676 t/s",
// #388, breakdown table "router" row; "full-offload MoE decode", #408, "Hypothesis":
// norm_topk_prob).  Shared by the SIMT and the tensor-core routers, which differ only in how a
// token's logits are formed.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// logit(e): the token's logit of expert e (called once per e < E, by the lane holding e);
// gate(): its shared-gate logit (called by lane 0 when shexp_scale is not NULL).
// EPL = experts per lane (power of two, EPL*32 >= E).  logits_out (nullable): [N][E].
template <int EPL, class Logit, class Gate>
__device__ __forceinline__ void route_token(Logit logit, Gate gate, int E, int top_k, int norm, int t, int lane,
                                            int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                                            float *__restrict__ shexp_scale, float *__restrict__ logits_out) {
    float l[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        int e = lane + 32 * i;
        float v = -INFINITY;
        if (e < E) {
            v = logit(e);
            if (logits_out) logits_out[(size_t)t * E + e] = v;
        }
        l[i] = v;
    }
    if (shexp_scale != nullptr && lane == 0) shexp_scale[t] = __fdiv_rn(1.0f, 1.0f + expf(-gate()));
    // softmax over all E experts
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, l[i]);
    m = warp_max(m);
    float p[EPL];
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        p[i] = (lane + 32 * i < E) ? expf(l[i] - m) : 0.0f;
        z += p[i];
    }
    z = warp_sum(z);
    float psel_sum = 0.0f;
    float my_w = 0.0f;
    if (EPL <= 2) {
        // top-k (top_k <= 32) by rank: expert e's slot is the number of experts before it in the order
        // (logit descending, ties to the lower index); every lane counts for its own experts against
        // all E logits, taken by shuffle (independent steps, no serial argmax rounds)
        int rank[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) rank[i] = 0;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
#pragma unroll
            for (int src = 0; src < 32; ++src) {
                // straight-line code (no branch between the shuffles), so they issue back to back;
                // experts past E hold -inf and count for no one (eo < E masks them)
                const float o = __shfl_sync(0xffffffffu, l[j], src);
                const int eo = src + 32 * j;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    rank[i] += (int)((eo < E) & ((o > l[i]) | ((o == l[i]) & (eo < e))));
                }
            }
        }
        // the selected experts' probabilities, each by the lane holding it
        float pw_own[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            pw_own[i] = (e < E && rank[i] < top_k) ? __fdiv_rn(p[i], z) : 0.0f;
        }
        // slot s: its holder lane gives the expert and its probability; weights summed in slot order
        for (int s = 0; s < top_k; ++s) {
            int has = -1;
            float pv = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && rank[i] == s) {
                    has = e;
                    pv = pw_own[i];
                }
            }
            const unsigned holders = __ballot_sync(0xffffffffu, has >= 0);
            const int src = __ffs(holders) - 1;  // exactly one lane holds slot s
            const int bi = __shfl_sync(0xffffffffu, has, src);
            const float pw = __shfl_sync(0xffffffffu, pv, src);
            psel_sum = __fadd_rn(psel_sum, pw);
            if (lane == s) my_w = pw;
            if (lane == 0) topk_idx[(size_t)t * top_k + s] = bi;
        }
    } else {
        // more than 64 experts: top_k rounds of warp argmax on the logits (the same order, ties to
        // the lower index) cost less than ranks (measured at E = 128); lane s keeps slot s's
        // probability
        for (int s = 0; s < top_k; ++s) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                int e = lane + 32 * i;
                bool cand = e < E && p[i] >= 0.0f;  // p = -1 marks a taken expert
                if (cand && (bi == 0x7fffffff || l[i] > bv || (l[i] == bv && e < bi))) {
                    bv = l[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
                    bv = ov;
                    bi = oi;
                }
            }
            float pw = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == bi) {
                    pw = __fdiv_rn(p[i], z);
                    p[i] = -1.0f;
                }
            pw = __shfl_sync(0xffffffffu, pw, bi & 31);
            psel_sum = __fadd_rn(psel_sum, pw);
            if (lane == s) my_w = pw;
            if (lane == 0) topk_idx[(size_t)t * top_k + s] = bi;
        }
    }
    if (lane < top_k)
        topk_w[(size_t)t * top_k + lane] = norm ? __fdiv_rn(my_w, psel_sum) : my_w;
}

}  // namespace moe
