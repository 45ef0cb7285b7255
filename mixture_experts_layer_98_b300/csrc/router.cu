// router.cu -- CUDA-core router (decode-sized batches, and E > 128): logits,
// then fp32 softmax, top-k and renormalisation.
//
// Follows the routing steps of Qwen3MoeSparseMoeBlock.forward (cnblogs page
// "大模型-qwen3 MoE 详细解读"): router_logits = gate(hidden_states) with a
// bias-free Linear, softmax over the experts in fp32, torch.topk of the
// probabilities (sorted), and division by their sum when norm_topk_prob.
//
// Ranking is done on the fp32 logits (the same order as on the probabilities,
// without exp rounding creating ties), descending, ties to the lower expert
// index.  The routing CTAs also write, per expert, the sum of the
// probabilities of their tokens (in token order) for the load-balance
// statistic.
#include "moe_common.cuh"
#include "routing.cuh"

namespace moe {

namespace {

constexpr int kSplitWarps = 8;   // experts per logits CTA (one warp each)
constexpr int kSplitTokens = 8;  // tokens per logits CTA (staged in shared memory)

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b, float acc) {
    acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
    acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
    acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
    acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
    acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
    acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
    acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
    acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
    return acc;
}

// logits[t,e] = x[t]·W_router[e] in fp32.  Grid (ceil(T/8), ceil(E/8), nsplit):
// a CTA stages 8 token rows of its slice of H (H/nsplit columns) in shared
// memory and each of its 8 warps streams that slice of one router row with
// 16-byte loads, writing partial logits to parts + z·T·E (slice z).  A single
// token thus spreads the router weights over nsplit·E/8 CTAs with a few loads
// in flight per lane.  The first CTA also zeroes the forward's status words
// (status[0..n_clear)).
__global__ void __launch_bounds__(kSplitWarps * 32) router_logits_split_kernel(
    const __nv_bfloat16* x, const __nv_bfloat16* Wr, int T, int H,
    int E, float* parts, int32_t* status, int n_clear) {
    extern __shared__ uint4 xs[];  // [kSplitTokens][H/nsplit/8]
    pdl_trigger();
    pdl_wait();
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < n_clear; i += blockDim.x) status[i] = 0;
    const int vpr = H / 8;                 // 16-byte vectors per row
    const int vps = vpr / gridDim.z;       // ... per slice
    const int c0 = blockIdx.z * vps;
    const int t0 = blockIdx.x * kSplitTokens;
    const int nt = min(kSplitTokens, T - t0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.y * kSplitWarps + warp;
    const uint4* wr = reinterpret_cast<const uint4*>(Wr) + (size_t)min(e, E - 1) * vpr + c0;
    // the first router-weight vectors of this warp's row are requested before
    // the tokens are staged, so the two memory round trips overlap
    constexpr int kEarly = 4;
    uint4 w_early[kEarly];
#pragma unroll
    for (int j = 0; j < kEarly; ++j) {
        const int c = lane + 32 * j;
        if (c < vps) w_early[j] = wr[c];
    }
    const uint4* xg = reinterpret_cast<const uint4*>(x) + (size_t)t0 * vpr + c0;
    for (int i = threadIdx.x; i < nt * vps; i += blockDim.x) {
        const int m = i / vps, c = i - m * vps;
        xs[i] = xg[(size_t)m * vpr + c];
    }
    __syncthreads();
    if (e >= E) return;
    float acc[kSplitTokens];
#pragma unroll
    for (int m = 0; m < kSplitTokens; ++m) acc[m] = 0.f;
#pragma unroll
    for (int j = 0; j < kEarly; ++j) {
        const int c = lane + 32 * j;
        if (c < vps) {
#pragma unroll
            for (int m = 0; m < kSplitTokens; ++m)
                if (m < nt) acc[m] = dot8_bf16(w_early[j], xs[m * vps + c], acc[m]);
        }
    }
#pragma unroll 4
    for (int c = lane + 32 * kEarly; c < vps; c += 32) {
        const uint4 wv = wr[c];
#pragma unroll
        for (int m = 0; m < kSplitTokens; ++m)
            if (m < nt) acc[m] = dot8_bf16(wv, xs[m * vps + c], acc[m]);
    }
    float* out = parts + (size_t)blockIdx.z * T * E;
#pragma unroll
    for (int m = 0; m < kSplitTokens; ++m) {
        float v = acc[m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == m && m < nt) out[(size_t)(t0 + m) * E + e] = v;
    }
}

// Routing from logits: one warp per token, kRouterTokens tokens (warps) per
// CTA, so a 4096-token batch keeps 4096 warps in flight.  The
// logits are the sum, in slice order, of nparts partial-logit arrays
// (parts + s * part_stride, [T, E] each); logits_out (may be null) receives
// that sum.
template <int EPL>
__global__ void __launch_bounds__(kRouterTokens * 32) route_from_logits_kernel(
    const float* parts, int nparts, size_t part_stride, float* logits_out, int T, int E, int K,
    int norm, const float* bias, int32_t* idx, float* w, float* p_partial) {
    __shared__ float ls[kRouterTokens * kMaxExperts];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int t0 = blockIdx.x * kRouterTokens;
    const int j = wid;  // one warp per token
    const int t = t0 + j;
    if (t < T) {  // warp-uniform
        float l[EPL];
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            if (e < E) {
                // every slice loaded before the first add, summed in slice order
                float pv[kRouterMaxSplits];
#pragma unroll
                for (int sl = 0; sl < kRouterMaxSplits; ++sl)
                    pv[sl] = sl < nparts ? parts[sl * part_stride + (size_t)t * E + e] : 0.f;
                float v = pv[0];
#pragma unroll
                for (int sl = 1; sl < kRouterMaxSplits; ++sl)
                    if (sl < nparts) v += pv[sl];
                l[q] = v;
                if (logits_out) logits_out[(size_t)t * E + e] = v;
            } else {
                l[q] = -INFINITY;
            }
        }
        route_token<EPL>(l, E, K, norm, bias, idx + (size_t)t * K, w + (size_t)t * K, ls + j * E);
    }
    __syncthreads();
    if (p_partial) {
        const int nt = min(kRouterTokens, T - t0);
        for (int e = tid; e < E; e += blockDim.x) {
            float s = 0.f;
            for (int t = 0; t < nt; ++t) s += ls[t * E + e];
            p_partial[(size_t)blockIdx.x * E + e] = s;
        }
    }
}

template <int EPL>
cudaError_t launch_route_t(const float* parts, int nparts, float* logits_out, const Sizes& s,
                           int norm, const float* bias, int32_t* idx, float* w, float* p_partial,
                           cudaStream_t st) {
    cudaError_t e = launch_pdl(route_from_logits_kernel<EPL>, dim3(s.nrouter()),
                               dim3(kRouterTokens * 32), 0, st, parts, nparts, (size_t)s.T * s.E,
                               logits_out, s.T, s.E, s.K, norm, bias, idx, w, p_partial);
    count_launches(1);
    return e;
}

}  // namespace

int router_simt_splits(const Sizes& s) {
    // Slices of H: enough CTAs to cover the SMs about twice (at most
    // kRouterMaxSplits, and H/nsplit a multiple of 8 columns).
    const int tiles = ((s.T + kSplitTokens - 1) / kSplitTokens) *
                      ((s.E + kSplitWarps - 1) / kSplitWarps);
    int nsplit = 1;
    while (nsplit < kRouterMaxSplits && tiles * nsplit < 2 * num_sms() &&
           (s.H / 8) % (2 * nsplit) == 0)
        nsplit *= 2;
    return nsplit;
}

cudaError_t launch_router_logits(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                                 int nsplit, float* parts, int32_t* status, int n_clear,
                                 cudaStream_t st) {
    const int smem = kSplitTokens * (s.H / nsplit) * 2;
    cudaError_t err = ensure_smem((const void*)router_logits_split_kernel, kSplitTokens * s.H * 2);
    if (err != cudaSuccess) return err;
    dim3 grid((s.T + kSplitTokens - 1) / kSplitTokens, (s.E + kSplitWarps - 1) / kSplitWarps,
              nsplit);
    err = launch_pdl(router_logits_split_kernel, grid, dim3(kSplitWarps * 32), smem, st, x, Wr, s.T,
                     s.H, s.E, parts, status, n_clear);
    count_launches(1);
    return err;
}

cudaError_t launch_router(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                          int norm, const float* bias, float* logits, float* parts, int32_t* idx,
                          float* w, float* p_partial, int32_t* status, int n_clear,
                          cudaStream_t st) {
    const int nsplit = router_simt_splits(s);
    cudaError_t err = launch_router_logits(x, Wr, s, nsplit, parts, status, n_clear, st);
    if (err != cudaSuccess) return err;
    return launch_route_from_logits(parts, nsplit, logits, s, norm, bias, idx, w, p_partial, st);
}

cudaError_t launch_route_from_logits(const float* parts, int nparts, float* logits_out,
                                     const Sizes& s, int norm, const float* bias, int32_t* idx,
                                     float* w, float* p_partial, cudaStream_t st) {
    if (nparts < 1 || nparts > kRouterMaxSplits) return cudaErrorInvalidValue;
    const int epl = (s.E + 31) / 32;
    if (epl <= 1)
        return launch_route_t<1>(parts, nparts, logits_out, s, norm, bias, idx, w, p_partial, st);
    if (epl <= 2)
        return launch_route_t<2>(parts, nparts, logits_out, s, norm, bias, idx, w, p_partial, st);
    if (epl <= 4)
        return launch_route_t<4>(parts, nparts, logits_out, s, norm, bias, idx, w, p_partial, st);
    return launch_route_t<8>(parts, nparts, logits_out, s, norm, bias, idx, w, p_partial, st);
}

}  // namespace moe
