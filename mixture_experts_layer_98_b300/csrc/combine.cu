// combine.cu -- gather-reduce of the weighted expert outputs into token order.
//
// Qwen3MoeSparseMoeBlock.forward (cnblogs page "大模型-qwen3 MoE 详细解读")
// accumulates each expert's weighted output with index_add_ into a zeroed
// [tokens, hidden] buffer.  Here each token instead reads its K rows of Y (the
// weighted expert outputs) and sums them in fp32 in k order, then rounds once
// to bf16: no zero-fill, no atomics, and the result does not depend on
// scheduling.  The down-projection kernels store Y token-major ([T, K, H]: the
// pair (t, k) at row t*K + k), so a token's K rows are one contiguous read;
// a pair with inv[t*K + k] < 0 was dropped by an expert capacity and is
// skipped (the pages' capacity: csdn page section "容量因子设计").  With
// y_by_inv, Y is in dispatch order and row inv[t*K + k] is read instead.
// Under a capacity Y is fp32: dropping pairs can leave a token with a few
// large terms that nearly cancel, and a bf16 rounding of each term would then
// be large next to the token's small result.  16-byte loads and stores.
#include "moe_common.cuh"

namespace moe {

namespace {

// The weighted expert outputs as bf16 (8 per 16-byte vector) or, under an
// expert capacity, as fp32 (8 per two 16-byte vectors).
struct YBf16 {
    using Vec = uint4;
    static __device__ __forceinline__ Vec load(const Vec* Y, size_t row, int vpr, int c) {
        return Y[row * vpr + c];
    }
    static __device__ __forceinline__ void add(float (&a)[8], const Vec& v) {
        a[0] += bf16_lo(v.x);
        a[1] += bf16_hi(v.x);
        a[2] += bf16_lo(v.y);
        a[3] += bf16_hi(v.y);
        a[4] += bf16_lo(v.z);
        a[5] += bf16_hi(v.z);
        a[6] += bf16_lo(v.w);
        a[7] += bf16_hi(v.w);
    }
};
struct YF32 {
    struct Vec {
        float4 lo, hi;
    };
    static __device__ __forceinline__ Vec load(const Vec* Y, size_t row, int vpr, int c) {
        return Y[row * vpr + c];
    }
    static __device__ __forceinline__ void add(float (&a)[8], const Vec& v) {
        a[0] += v.lo.x;
        a[1] += v.lo.y;
        a[2] += v.lo.z;
        a[3] += v.lo.w;
        a[4] += v.hi.x;
        a[5] += v.hi.y;
        a[6] += v.hi.z;
        a[7] += v.hi.w;
    }
};

template <typename YT>
__global__ void __launch_bounds__(256) combine_kernel(const typename YT::Vec* Y,
                                                      const int32_t* inv, int y_by_inv,
                                                      int T, int K, int vpr, uint4* out) {
    pdl_trigger();
    pdl_wait();
    const long long total = (long long)T * vpr;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int t = (int)(i / vpr), c = (int)(i % vpr);
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = 0.f;
        // plain (coherent) loads: Y (and inv) are written by earlier kernels of
        // the forward, which may still have been running when this grid
        // launched.  Four rows are loaded before any is added, so four loads
        // are in flight; the sum still runs in k order.
        for (int k0 = 0; k0 < K; k0 += 4) {
            typename YT::Vec v[4];
            bool ok[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = k0 + j;
                ok[j] = k < K;
                if (ok[j]) {
                    const int r = inv ? inv[(size_t)t * K + k] : 0;
                    ok[j] = r >= 0;  // a pair dropped by a capacity adds nothing
                    const size_t row = y_by_inv ? (size_t)r : (size_t)t * K + k;
                    if (ok[j]) v[j] = YT::load(Y, row, vpr, c);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (ok[j]) YT::add(a, v[j]);
        }
        uint4 o;
        o.x = pack_bf16x2(a[0], a[1]);
        o.y = pack_bf16x2(a[2], a[3]);
        o.z = pack_bf16x2(a[4], a[5]);
        o.w = pack_bf16x2(a[6], a[7]);
        out[(size_t)t * vpr + c] = o;
    }
}

}  // namespace

cudaError_t launch_combine(const __nv_bfloat16* Y, const float* Y32, const int32_t* inv,
                           bool y_by_inv, int T, int K, int H, __nv_bfloat16* out,
                           cudaStream_t st) {
    const int vpr = H / 8;
    const long long total = (long long)T * vpr;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t e =
        Y32 ? launch_pdl(combine_kernel<YF32>, dim3((unsigned)blocks), dim3(256), 0, st,
                         reinterpret_cast<const YF32::Vec*>(Y32), inv, (int)y_by_inv, T, K, vpr,
                         reinterpret_cast<uint4*>(out))
            : launch_pdl(combine_kernel<YBf16>, dim3((unsigned)blocks), dim3(256), 0, st,
                         reinterpret_cast<const uint4*>(Y), inv, (int)y_by_inv, T, K, vpr,
                         reinterpret_cast<uint4*>(out));
    count_launches(1);
    return e;
}

}  // namespace moe
