// router_tc.cu -- router GEMM on tcgen05 fused with fp32 softmax, top-k,
// renormalisation and the per-tile probability sums of the load-balance
// statistic.
//
// Routing as in Qwen3MoeSparseMoeBlock.forward (cnblogs page
// "大模型-qwen3 MoE 详细解读"): router_logits = gate(x) (bias-free Linear),
// softmax over all experts in fp32, top-k (sorted), division by the kept sum
// when norm_topk_prob.  Ranking uses the fp32 logits, descending, ties to the
// lower expert index -- the same rule as the SIMT router.
//
// One CTA per 128-token tile (192 threads), E <= 128:
//   warp 0     TMA: x tile 128x64 and the whole router weight tile N x 64
//              (N = E rounded up to 32) per k-block, 4-stage SW128 ring
//   warp 1     owns TMEM (two N-column fp32 buffers) and issues, per k-block,
//              tcgen05.mma M=128 N K=16 x4 into a fresh accumulator
//   warps 2-5  epilogue, one token per thread (its TMEM lane): adds each
//              k-block's partial logits into fp32 registers (round to nearest),
//              then writes the logits, keeps a sorted top-KMAX list while
//              taking the row maximum, computes the exp-sum and the weights, and
//              finally the column sums of the probabilities over the tile; the
//              row is staged in shared memory (reusing the drained stage ring)
//              so these passes run as compact rolled loops, and the column sums
//              are one expert per thread over the rows in order
// Accumulating in TMEM over only 64 products per k-block and summing the
// k-blocks in registers keeps the logits within ~1e-6 relative of the exact
// dot product; one accumulation chain over all of H drifts by ~1e-5 at
// H = 4096, which would eat into the margin that separates genuine near-ties
// in the top-k.
// Waits are bounded as in the expert GEMMs; a timeout writes MOE_ERR_TIMEOUT to
// the status word.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kRM = 128;
constexpr int kRK = 64;
constexpr int kRStages = 4;
constexpr int kRThreads = 192;
constexpr uint64_t kRTimeoutNs = 2000000000ull;
constexpr int kRowPitch = 129;  // floats per staged logits row (odd: conflict-free columns)

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int NCH, int KMAX>
__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, int T, int H, int E, int K,
                     int norm, float* __restrict__ logits, int32_t* __restrict__ idx,
                     float* __restrict__ wout, float* __restrict__ p_partial,
                     int32_t* __restrict__ status) {
    constexpr int N = NCH * 32;
    constexpr int kABytes = kRM * kRK * 2;
    constexpr int kStageBytes = kABytes + N * kRK * 2;
    constexpr uint32_t kTmemCols = 2 * N <= 64 ? 64u : (2 * N <= 128 ? 128u : 256u);
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kRM, N);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[kRStages];
    __shared__ __align__(8) uint64_t empty_bar[kRStages];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_kb = H / kRK;
    const int t0 = blockIdx.x * kRM;

    if (threadIdx.x == 0) {
        if (status && blockIdx.x == 0) *status = 0;  // first kernel of a forward
        for (int s = 0; s < kRStages; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull_bar[b], 1);
            ptx::mbar_init(&tempty_bar[b], 4);
        }
        ptx::mbar_init(&drain_bar, 1);
        abort_s = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&tmem_base_s, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!ptx::mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_s, kRTimeoutNs)) {
                    ok = false;
                    break;
                }
                uint8_t* sA = smem + stage * kStageBytes;
                ptx::mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
                ptx::tma_load_2d(sA, &tmX, &full_bar[stage], kb * kRK, t0);
                ptx::tma_load_2d(sA + kABytes, &tmW, &full_bar[stage], kb * kRK, 0);
                ++issued;
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                atomicExch(status, MOE_ERR_TIMEOUT);
                int dummy = 0;
                const long long first = issued > kRStages ? issued - kRStages : 0;
                for (long long n = first; n < issued; ++n)
                    ptx::mbar_wait_bounded(&full_bar[n % kRStages], (uint32_t)((n / kRStages) & 1),
                                           &dummy, kRTimeoutNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = 0; kb < num_kb; ++kb) {
                const int buf = kb & 1;
                const uint32_t use_phase = (uint32_t)((kb >> 1) & 1);
                if (!ptx::mbar_wait_bounded(&tempty_bar[buf], use_phase ^ 1u, &abort_s,
                                            kRTimeoutNs) ||
                    !ptx::mbar_wait_bounded(&full_bar[stage], phase, &abort_s, kRTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a_addr = ptx::smem_u32(smem + stage * kStageBytes);
                const uint64_t adesc = ptx::desc_sw128_kmajor(a_addr);
                const uint64_t bdesc = ptx::desc_sw128_kmajor(a_addr + kABytes);
                const uint32_t d = tmem_base + (uint32_t)(buf * N);
#pragma unroll
                for (int k = 0; k < kRK / 16; ++k)  // a fresh accumulator per k-block
                    ptx::mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k != 0 ? 1u : 0u);
                ptx::mma_commit(&empty_bar[stage]);
                ptx::mma_commit(&tfull_bar[buf]);
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) atomicExch(status, MOE_ERR_TIMEOUT);
            ptx::mma_commit(&drain_bar);
            int dummy = 0;
            ptx::mbar_wait_bounded(&drain_bar, 0u, &dummy, kRTimeoutNs);
        }
    } else {
        // ---------------- epilogue: one token per thread ----------------
        const int q = warp & 3;   // TMEM lane quadrant
        const int r = q * 32 + lane;
        const int t = t0 + r;
        const bool valid = t < T;
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
        float acc[N];
#pragma unroll
        for (int j = 0; j < N; ++j) acc[j] = 0.f;
        int ok = 1;
        for (int kb = 0; kb < num_kb && ok; ++kb) {
            const int buf = kb & 1;
            if (lane == 0)
                ok = ptx::mbar_wait_bounded(&tfull_bar[buf], (uint32_t)((kb >> 1) & 1), &abort_s,
                                            kRTimeoutNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                uint32_t v[32];
                ptx::tmem_ld32(taddr + (uint32_t)(buf * N + c * 32), v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[c * 32 + j] += __uint_as_float(v[j]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty_bar[buf]);
        }
        // The mainloop is over (every MMA has completed, so the stage buffers are
        // free): park the row in shared memory and run the epilogue passes as
        // rolled loops -- fully unrolled they would be tens of KB of straight-line
        // code executed once, bound by instruction fetch.
        float* rows = reinterpret_cast<float*>(smem);  // [128][kRowPitch]
        float* myrow = rows + r * kRowPitch;
        if (ok) {
#pragma unroll
            for (int j = 0; j < N; ++j) myrow[j] = acc[j];
        }
        __syncwarp();
        if (ok) {
            // logits out, row max, sorted top-KMAX: experts arrive in increasing
            // index, so a new logit equal to the last kept one ranks after it;
            // displaced entries keep the (logit desc, index asc) order as they move
            float tv[KMAX];
            int ti[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                tv[j] = -INFINITY;
                ti[j] = 0x7fffffff;
            }
            float m = -INFINITY;
#pragma unroll 1
            for (int e = 0; e < E; ++e) {
                const float l = myrow[e];
                if (valid && logits) logits[(size_t)t * E + e] = l;
                m = fmaxf(m, l);
                if (l > tv[KMAX - 1]) {
                    float cv = l;
                    int ce = e;
#pragma unroll
                    for (int s2 = 0; s2 < KMAX; ++s2) {
                        if (cv > tv[s2] || (cv == tv[s2] && ce < ti[s2])) {
                            const float fv = tv[s2];
                            const int fe = ti[s2];
                            tv[s2] = cv;
                            ti[s2] = ce;
                            cv = fv;
                            ce = fe;
                        }
                    }
                }
            }
            float ssum = 0.f;
#pragma unroll 1
            for (int e = 0; e < E; ++e) ssum += expf(myrow[e] - m);
            const float inv_s = 1.0f / ssum;
            float wsum = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < K) wsum += expf(tv[j] - m) * inv_s;
            if (valid) {
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < K) {
                        const float pj = expf(tv[j] - m) * inv_s;
                        idx[(size_t)t * K + j] = ti[j];
                        wout[(size_t)t * K + j] = norm ? pj / wsum : pj;
                    }
                }
            }
            // the row now holds this token's probabilities (zero for padding rows)
#pragma unroll 1
            for (int e = 0; e < E; ++e) myrow[e] = valid ? expf(myrow[e] - m) * inv_s : 0.f;
        } else if (lane == 0) {
            atomicExch(status, MOE_ERR_TIMEOUT);
        }
        // every epilogue warp reaches this barrier exactly once, timed out or not
        ptx::tc_fence_before();
        epi_bar();
        if (!abort_s) {
            // column sums: thread e adds expert e's probability over the 128 rows in order
            const int tid = threadIdx.x - 64;  // 0..127
            for (int e = tid; e < E; e += 128) {
                float cs = 0.f;
#pragma unroll 8
                for (int rr = 0; rr < kRM; ++rr) cs += rows[rr * kRowPitch + e];
                p_partial[(size_t)blockIdx.x * E + e] = cs;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

template <int NCH, int KMAX>
cudaError_t launch_router_tc_t(const CUtensorMap& mx, const CUtensorMap& mw, const Sizes& s,
                               int norm, float* logits, int32_t* idx, float* w, float* p_partial,
                               int32_t* status, cudaStream_t st) {
    const int ring = kRStages * (kRM * kRK * 2 + NCH * 32 * kRK * 2);
    const int smem = (ring > kRM * kRowPitch * 4 ? ring : kRM * kRowPitch * 4) + 1024;
    cudaError_t err = ensure_smem((const void*)router_tc_kernel<NCH, KMAX>, smem);
    if (err != cudaSuccess) return err;
    const int grid = (s.T + kRM - 1) / kRM;
    router_tc_kernel<NCH, KMAX><<<grid, kRThreads, smem, st>>>(mx, mw, s.T, s.H, s.E, s.K, norm,
                                                               logits, idx, w, p_partial, status);
    count_launches(1);
    return cudaGetLastError();
}

template <int NCH>
cudaError_t launch_router_tc_k(const CUtensorMap& mx, const CUtensorMap& mw, const Sizes& s,
                               int norm, float* logits, int32_t* idx, float* w, float* p_partial,
                               int32_t* status, cudaStream_t st) {
    if (s.K <= 2)
        return launch_router_tc_t<NCH, 2>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
    if (s.K <= 4)
        return launch_router_tc_t<NCH, 4>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
    if (s.K <= 8)
        return launch_router_tc_t<NCH, 8>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
    return launch_router_tc_t<NCH, 16>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
}

}  // namespace

int router_tc_partials(int T) { return (T + kRM - 1) / kRM; }

bool router_tc_supported(const Sizes& s) { return s.E <= 128; }

cudaError_t launch_router_tc(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                             int norm, float* logits, int32_t* idx, float* w, float* p_partial,
                             int32_t* status, cudaStream_t st) {
    const int nch = (s.E + 31) / 32;
    if (nch > 4) return cudaErrorInvalidValue;
    CUtensorMap mx, mw;
    if (!make_tma_2d(&mx, x, (uint64_t)s.T, (uint64_t)s.H, kRM) ||
        !make_tma_2d(&mw, Wr, (uint64_t)s.E, (uint64_t)s.H, (uint32_t)(nch * 32)))
        return cudaErrorInvalidValue;
    switch (nch) {
        case 1: return launch_router_tc_k<1>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
        case 2: return launch_router_tc_k<2>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
        case 3: return launch_router_tc_k<3>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
        default: return launch_router_tc_k<4>(mx, mw, s, norm, logits, idx, w, p_partial, status, st);
    }
}

}  // namespace moe
