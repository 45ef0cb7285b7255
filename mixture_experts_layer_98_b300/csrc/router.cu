// router.cu -- router GEMM fused with fp32 softmax, top-k and renormalisation.
//
// Follows the routing steps of Qwen3MoeSparseMoeBlock.forward (cnblogs page
// "大模型-qwen3 MoE 详细解读"): router_logits = gate(hidden_states) with a
// bias-free Linear, softmax over the experts in fp32, torch.topk of the
// probabilities (sorted), and division by their sum when norm_topk_prob.
//
// Ranking is done on the fp32 logits (the same order as on the probabilities,
// without exp rounding creating ties), descending, ties to the lower expert
// index.  Each CTA also writes, per expert, the sum of the probabilities of its
// tokens (in token order) for the load-balance statistic.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kHC = 32;  // hidden-dimension chunk staged in shared memory

// (value, expert, prob) of the best candidate: larger value first, then the
// lower expert index.
struct Cand {
    float v;
    int e;
    float p;
};

__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
    return a.v > b.v || (a.v == b.v && a.e < b.e);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Cand o;
        o.v = __shfl_xor_sync(0xffffffffu, c.v, off);
        o.e = __shfl_xor_sync(0xffffffffu, c.e, off);
        o.p = __shfl_xor_sync(0xffffffffu, c.p, off);
        if (better(o, c)) c = o;
    }
    return c;
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
// the full softmax into probs[0..E).
template <int EPL>
__device__ __forceinline__ void route_token(const float (&l)[EPL], int E, int K, int norm,
                                            int32_t* idx_row, float* w_row, float* probs) {
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
    uint32_t taken = 0;
    float wsum = 0.f;
    int my_e = -1;
    float my_p = 0.f;
    for (int k = 0; k < K; ++k) {
        Cand c{-INFINITY, 0x7fffffff, 0.f};
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            if (e < E && !(taken & (1u << q))) {
                Cand o{l[q], e, p[q]};
                if (c.e == 0x7fffffff || better(o, c)) c = o;
            }
        }
        c = warp_best(c);
        if ((c.e & 31) == lane) taken |= 1u << (c.e >> 5);
        wsum += c.p;  // same value and order in every lane
        if (lane == k) {
            my_e = c.e;
            my_p = c.p;
        }
    }
    if (lane < K) {
        idx_row[lane] = my_e;
        w_row[lane] = norm ? my_p / wsum : my_p;
    }
}

// x [T,H] bf16, Wr [E,H] bf16 -> logits, idx, w, per-CTA probability sums.
// CTA = 256 threads = 8 token groups of 4 tokens; lane -> experts lane+32q.
template <int EPL>
__global__ void __launch_bounds__(256) router_simt_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wr, int T, int H,
    int E, int K, int norm, float* __restrict__ logits, int32_t* __restrict__ idx,
    float* __restrict__ w, float* __restrict__ p_partial, int32_t* __restrict__ status) {
    extern __shared__ float sm[];
    if (status && blockIdx.x == 0 && threadIdx.x == 0) *status = 0;  // first kernel of a forward
    float* xs = sm;                             // [32][kHC + 1]
    float* wsm = xs + kRouterTokens * (kHC + 1);  // [kHC][E]
    float* ls = wsm + kHC * E;                  // [32][E] logits, then probabilities
    const int tid = threadIdx.x, lane = tid & 31, tg = tid >> 5;
    const int t0 = blockIdx.x * kRouterTokens;

    float acc[4][EPL];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < EPL; ++q) acc[j][q] = 0.f;

    for (int h0 = 0; h0 < H; h0 += kHC) {
        for (int i = tid; i < kRouterTokens * kHC; i += 256) {
            const int t = i / kHC, c = i % kHC;
            xs[t * (kHC + 1) + c] =
                (t0 + t < T) ? __bfloat162float(x[(size_t)(t0 + t) * H + h0 + c]) : 0.f;
        }
        for (int i = tid; i < E * kHC; i += 256) {
            const int e = i / kHC, c = i % kHC;
            wsm[c * E + e] = __bfloat162float(Wr[(size_t)e * H + h0 + c]);
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < kHC; ++c) {
            float xv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) xv[j] = xs[(tg * 4 + j) * (kHC + 1) + c];
#pragma unroll
            for (int q = 0; q < EPL; ++q) {
                const int e = lane + 32 * q;
                const float wv = (e < E) ? wsm[c * E + e] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[j][q] = fmaf(xv[j], wv, acc[j][q]);
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int t = t0 + tg * 4 + j;
        if (t >= T) continue;  // warp-uniform
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            if (e < E && logits) logits[(size_t)t * E + e] = acc[j][q];
        }
        route_token<EPL>(acc[j], E, K, norm, idx + (size_t)t * K, w + (size_t)t * K,
                         ls + (tg * 4 + j) * E);
    }
    __syncthreads();
    if (p_partial) {
        const int nt = min(kRouterTokens, T - t0);
        for (int e = tid; e < E; e += 256) {
            float s = 0.f;
            for (int t = 0; t < nt; ++t) s += ls[t * E + e];
            p_partial[(size_t)blockIdx.x * E + e] = s;
        }
    }
}

// Routing only, from given logits (same per-token code as the fused kernel).
// CTA = 256 threads, one warp per token, kRouterTokens tokens per CTA.
template <int EPL>
__global__ void __launch_bounds__(256) route_from_logits_kernel(
    const float* __restrict__ logits, int T, int E, int K, int norm, int32_t* __restrict__ idx,
    float* __restrict__ w, float* __restrict__ p_partial) {
    __shared__ float ls[kRouterTokens * kMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int t0 = blockIdx.x * kRouterTokens;
    for (int j = wid; j < kRouterTokens; j += 8) {
        const int t = t0 + j;
        if (t >= T) break;
        float l[EPL];
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            l[q] = (e < E) ? logits[(size_t)t * E + e] : -INFINITY;
        }
        route_token<EPL>(l, E, K, norm, idx + (size_t)t * K, w + (size_t)t * K, ls + j * E);
    }
    __syncthreads();
    if (p_partial) {
        const int nt = min(kRouterTokens, T - t0);
        for (int e = tid; e < E; e += 256) {
            float s = 0.f;
            for (int t = 0; t < nt; ++t) s += ls[t * E + e];
            p_partial[(size_t)blockIdx.x * E + e] = s;
        }
    }
}

template <int EPL>
cudaError_t launch_router_t(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                            int norm, float* logits, int32_t* idx, float* w, float* p_partial,
                            int32_t* status, cudaStream_t st) {
    const size_t smem =
        sizeof(float) * (kRouterTokens * (kHC + 1) + kHC * s.E + kRouterTokens * s.E);
    cudaError_t err = cudaFuncSetAttribute(router_simt_kernel<EPL>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    router_simt_kernel<EPL><<<s.nrouter(), 256, smem, st>>>(x, Wr, s.T, s.H, s.E, s.K, norm,
                                                            logits, idx, w, p_partial, status);
    count_launches(1);
    return cudaGetLastError();
}

template <int EPL>
cudaError_t launch_route_t(const float* logits, const Sizes& s, int norm, int32_t* idx, float* w,
                           float* p_partial, cudaStream_t st) {
    route_from_logits_kernel<EPL><<<s.nrouter(), 256, 0, st>>>(logits, s.T, s.E, s.K, norm, idx,
                                                               w, p_partial);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                          int norm, float* logits, int32_t* idx, float* w, float* p_partial,
                          int32_t* status, cudaStream_t st) {
    const int epl = (s.E + 31) / 32;
    if (epl <= 1) return launch_router_t<1>(x, Wr, s, norm, logits, idx, w, p_partial, status, st);
    if (epl <= 2) return launch_router_t<2>(x, Wr, s, norm, logits, idx, w, p_partial, status, st);
    if (epl <= 4) return launch_router_t<4>(x, Wr, s, norm, logits, idx, w, p_partial, status, st);
    return launch_router_t<8>(x, Wr, s, norm, logits, idx, w, p_partial, status, st);
}

cudaError_t launch_route_from_logits(const float* logits, const Sizes& s, int norm, int32_t* idx,
                                     float* w, float* p_partial, cudaStream_t st) {
    const int epl = (s.E + 31) / 32;
    if (epl <= 1) return launch_route_t<1>(logits, s, norm, idx, w, p_partial, st);
    if (epl <= 2) return launch_route_t<2>(logits, s, norm, idx, w, p_partial, st);
    if (epl <= 4) return launch_route_t<4>(logits, s, norm, idx, w, p_partial, st);
    return launch_route_t<8>(logits, s, norm, idx, w, p_partial, st);
}

}  // namespace moe
