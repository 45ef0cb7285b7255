// routing.cuh -- per-token routing of a warp: fp32 softmax over the experts,
// top-k and renormalisation (router kernels and the small-batch dispatch).
//
// Follows the routing steps of Qwen3MoeSparseMoeBlock.forward (cnblogs page
// "大模型-qwen3 MoE 详细解读"): softmax over the experts in fp32, torch.topk of
// the probabilities (sorted), and division by their sum when norm_topk_prob.
// Ranking is done on the fp32 logits (the same order as on the
// probabilities, without exp rounding creating ties), descending, ties to
// the lower expert index.
#pragma once

#include "moe_common.cuh"

namespace moe {

// Order-preserving map of a float to uint32 (larger float -> larger key);
// -0 is folded to +0 first, so equal floats give equal keys.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One warp routes one token whose E logits sit in l[] (lane holds experts
// lane, lane+32, ...).  Writes idx/w for the token and, when probs != null,
// the full softmax into probs[0..E).  With bias != null (fp32 [E], a
// selection-only expert bias for auxiliary-loss-free balancing, the DeepSeek
// scheme of the sshipanoo.com page "项目 17：稀疏性的调度艺术", section
// "第四阶段：更先进的路由方案：DeepSeek 的突破") the experts are ranked by the
// fp32 key l + bias while their weights stay the unbiased probabilities.
template <int EPL>
__device__ __forceinline__ void route_token(const float (&l)[EPL], int E, int K, int norm,
                                            const float* bias, int32_t* idx_row, float* w_row,
                                            float* probs) {
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < EPL; ++q)
        if (lane + 32 * q < E) m = fmaxf(m, l[q]);
    m = warp_max(m);
    float ex[EPL];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        ex[q] = (lane + 32 * q < E) ? expf(l[q] - m) : 0.f;
        s += ex[q];
    }
    s = warp_sum(s);
    const float inv_s = 1.0f / s;
    float p[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        p[q] = ex[q] * inv_s;
        if (probs && lane + 32 * q < E) probs[lane + 32 * q] = p[q];
    }
    // K rounds of a warp-wide arg-max: the largest key, then the lowest expert
    // index among the lanes holding it (two redux.sync per round).  The
    // winner's (unbiased) probability is fetched from the lane that holds it.
    uint32_t key[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        key[q] = e < E ? order_key(bias ? l[q] + bias[e] : l[q]) : 0u;
    }
    float wsum = 0.f;
    int my_e = -1;
    float my_p = 0.f;
    for (int k = 0; k < K; ++k) {
        uint32_t bk = 0u;
        int be = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < EPL; ++q)  // experts of a lane come in increasing index
            if (key[q] > bk) {
                bk = key[q];
                be = lane + 32 * q;
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const int we = (int)__reduce_min_sync(0xffffffffu, bk == mk ? (uint32_t)be : 0x7fffffffu);
        float pw = 0.f;
#pragma unroll
        for (int q = 0; q < EPL; ++q)  // taken; the winner's probability
            if (we == lane + 32 * q) {
                key[q] = 0u;
                pw = p[q];
            }
        const float pk = __shfl_sync(0xffffffffu, pw, we & 31);
        wsum += pk;  // same value and order in every lane
        if (lane == k) {
            my_e = we;
            my_p = pk;
        }
    }
    if (lane < K) {
        idx_row[lane] = my_e;
        w_row[lane] = norm ? my_p / wsum : my_p;
    }
}

}  // namespace moe
