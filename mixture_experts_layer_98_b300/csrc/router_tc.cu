// router_tc.cu -- router GEMM on tcgen05: fp32 logits x·W_routerᵀ for the
// tensor-core path (T >= 128, E <= 128).
//
// Routing as in Qwen3MoeSparseMoeBlock.forward (cnblogs page
// "大模型-qwen3 MoE 详细解读") starts with router_logits = gate(x), a bias-free
// Linear.  This kernel produces those logits; the softmax, top-k and
// renormalisation run in the routing kernel of router.cu, one warp per token
// over many CTAs, which also adds up the partial logits written here.
//
// Grid (ceil(T/128), S): CTA (tile, s) computes the 128 x N partial logits
// (N = E rounded up to 32) of its token tile over the s-th of S equal slices of
// H, so that even T = 4096 gives ~148 CTAs.  192 threads:
//   warp 0     prefetches the tile's x rows and the router weights into L2 as
//              contiguous ranges, then feeds a 4-stage SW128 TMA ring (x tile
//              128x64, router weight tile N x 64 per k-block)
//   warp 1     owns TMEM (four N-column fp32 accumulators) and issues, per
//              k-block, tcgen05.mma M=128 N K=16 x4 into accumulator kb % 4
//   warps 2-5  read the accumulators (one token per thread, its TMEM lane), add
//              them in fp32 in a fixed order, and stage the rows in shared
//              memory; then every warp copies the rows out with coalesced stores
// Four independent accumulation chains, each over a quarter of the slice,
// keep the logits within a few 1e-6 relative of the exact dot product; one
// chain over all of H drifts by ~1e-5 at H = 4096, which would eat into the
// margin that separates genuine near-ties in the top-k.
// Waits are bounded as in the expert GEMMs; a timeout writes MOE_ERR_TIMEOUT to
// the status word.  The first CTA zeroes the forward's status words
// (status[0..n_clear)) after its dependency wait.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kRM = 128;
constexpr int kRK = 64;
constexpr int kRStages = 4;
constexpr int kRThreads = 192;
constexpr uint64_t kRTimeoutNs = 2000000000ull;
constexpr int kRBufs = 4;       // independent TMEM accumulators (k-block kb -> kb % kRBufs)
constexpr int kRowPitch = 129;  // floats per staged logits row (odd: conflict-free columns)

template <int NCH>
__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const __nv_bfloat16* x,
                     const __nv_bfloat16* Wr, int T, int H, int E, int nsplit,
                     float* parts, int32_t* status, int n_clear) {
    constexpr int N = NCH * 32;
    constexpr int kABytes = kRM * kRK * 2;
    constexpr int kStageBytes = kABytes + N * kRK * 2;
    constexpr uint32_t kTmemCols = kRBufs * N <= 128 ? 128u : (kRBufs * N <= 256 ? 256u : 512u);
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kRM, N);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[kRStages];
    __shared__ __align__(8) uint64_t empty_bar[kRStages];
    __shared__ __align__(8) uint64_t tfull_bar;
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRM;
    const int nkb_all = H / kRK;
    const int kb0 = (int)((long long)nkb_all * blockIdx.y / nsplit);
    const int kb1 = (int)((long long)nkb_all * (blockIdx.y + 1) / nsplit);
    const int num_kb = kb1 - kb0;

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], 1);
        }
        ptx::mbar_init(&tfull_bar, 1);
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
    pdl_wait();  // the prologue above overlaps the previous kernel's tail
    if (status && blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < n_clear; i += blockDim.x) status[i] = 0;

    if (warp == 0) {
        if (lane == 0) {
            // The TMA boxes read 128-byte column strips across rows H*2 bytes
            // apart; pulling the slice of the tile's rows and of the router
            // weights into L2 first turns that into sequential DRAM traffic.
            const int nrows = min(kRM, T - t0);
            const size_t slice = (size_t)num_kb * kRK * 2;
            for (int r = 0; r < nrows; ++r)
                ptx::prefetch_l2_bulk(x + (size_t)(t0 + r) * H + (size_t)kb0 * kRK, (uint32_t)slice);
            if (blockIdx.x == 0)
                for (int e = 0; e < E; ++e)
                    ptx::prefetch_l2_bulk(Wr + (size_t)e * H + (size_t)kb0 * kRK, (uint32_t)slice);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
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
            for (int j = 0; j < num_kb; ++j) {
                if (!ptx::mbar_wait_bounded(&full_bar[stage], phase, &abort_s, kRTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a_addr = ptx::smem_u32(smem + stage * kStageBytes);
                const uint64_t adesc = ptx::desc_sw128_kmajor(a_addr);
                const uint64_t bdesc = ptx::desc_sw128_kmajor(a_addr + kABytes);
                // k-block j of the slice accumulates into buffer j % kRBufs (fresh on first use)
                const uint32_t d = tmem_base + (uint32_t)((j % kRBufs) * N);
#pragma unroll
                for (int k = 0; k < kRK / 16; ++k)
                    ptx::mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdesc,
                                  (j >= kRBufs || k != 0) ? 1u : 0u);
                ptx::mma_commit(&empty_bar[stage]);
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) ptx::mma_commit(&tfull_bar);
            else atomicExch(status, MOE_ERR_TIMEOUT);
            ptx::mma_commit(&drain_bar);
            int dummy = 0;
            ptx::mbar_wait_bounded(&drain_bar, 0u, &dummy, kRTimeoutNs);
        }
    } else {
        // ---------------- accumulators -> staged rows (one token per thread) ----
        const int q = warp & 3;  // TMEM lane quadrant
        const int r = q * 32 + lane;
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
        float acc[N];
#pragma unroll
        for (int j = 0; j < N; ++j) acc[j] = 0.f;
        int ok = 1;
        if (lane == 0) ok = ptx::mbar_wait_bounded(&tfull_bar, 0u, &abort_s, kRTimeoutNs);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
            ptx::tc_fence_after();
            const int nbuf = num_kb < kRBufs ? num_kb : kRBufs;
            for (int b = 0; b < nbuf; ++b) {  // acc = ((b0 + b1) + b2) + b3
#pragma unroll
                for (int c = 0; c < NCH / 2; ++c) {  // 64 columns per TMEM load
                    uint32_t v[64];
                    ptx::tmem_ld64(taddr + (uint32_t)(b * N + c * 64), v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 64; ++j) acc[c * 64 + j] += __uint_as_float(v[j]);
                }
                if (NCH & 1) {
                    uint32_t v[32];
                    ptx::tmem_ld32(taddr + (uint32_t)(b * N + (NCH - 1) * 32), v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[(NCH - 1) * 32 + j] += __uint_as_float(v[j]);
                }
            }
            // every MMA has completed, so the stage ring is free for the rows
            float* myrow = reinterpret_cast<float*>(smem) + r * kRowPitch;
#pragma unroll
            for (int j = 0; j < N; ++j) myrow[j] = acc[j];
        } else if (lane == 0) {
            atomicExch(status, MOE_ERR_TIMEOUT);
        }
    }

    // all warps: coalesced copy of the staged rows into this slice's partials
    ptx::tc_fence_before();
    __syncthreads();
    if (!abort_s) {
        const float* rows = reinterpret_cast<const float*>(smem);
        float* dst = parts + (size_t)blockIdx.y * T * E;
        for (int rr = warp; rr < kRM; rr += kRThreads / 32) {
            const int t = t0 + rr;
            if (t >= T) break;
            for (int e = lane; e < E; e += 32) dst[(size_t)t * E + e] = rows[rr * kRowPitch + e];
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

template <int NCH>
cudaError_t launch_router_tc_n(const CUtensorMap& mx, const CUtensorMap& mw,
                               const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                               int nsplit, float* parts, int32_t* status, int n_clear,
                               cudaStream_t st) {
    const int ring = kRStages * (kRM * kRK * 2 + NCH * 32 * kRK * 2);
    const int smem = (ring > kRM * kRowPitch * 4 ? ring : kRM * kRowPitch * 4) + 1024;
    cudaError_t err = ensure_smem((const void*)router_tc_kernel<NCH>, smem);
    if (err != cudaSuccess) return err;
    dim3 grid((s.T + kRM - 1) / kRM, nsplit);
    err = launch_pdl(router_tc_kernel<NCH>, grid, dim3(kRThreads), smem, st, mx, mw, x, Wr, s.T,
                     s.H, s.E, nsplit, parts, status, n_clear);
    count_launches(1);
    return err;
}

}  // namespace

bool router_tc_supported(const Sizes& s) { return s.E <= 128; }

int router_tc_splits(const Sizes& s) {
    const int tiles = (s.T + kRM - 1) / kRM;
    int n = (num_sms() + tiles - 1) / tiles;
    if (n > kRouterMaxSplits) n = kRouterMaxSplits;
    if (n > s.H / kRK) n = s.H / kRK;
    return n < 1 ? 1 : n;
}

cudaError_t launch_router_tc(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                             int nsplit, float* parts, int32_t* status, int n_clear,
                             cudaStream_t st) {
    const int nch = (s.E + 31) / 32;
    if (nch > 4) return cudaErrorInvalidValue;
    CUtensorMap mx, mw;
    if (!make_tma_2d(&mx, x, (uint64_t)s.T, (uint64_t)s.H, kRM) ||
        !make_tma_2d(&mw, Wr, (uint64_t)s.E, (uint64_t)s.H, (uint32_t)(nch * 32)))
        return cudaErrorInvalidValue;
    switch (nch) {
        case 1: return launch_router_tc_n<1>(mx, mw, x, Wr, s, nsplit, parts, status, n_clear, st);
        case 2: return launch_router_tc_n<2>(mx, mw, x, Wr, s, nsplit, parts, status, n_clear, st);
        case 3: return launch_router_tc_n<3>(mx, mw, x, Wr, s, nsplit, parts, status, n_clear, st);
        default: return launch_router_tc_n<4>(mx, mw, x, Wr, s, nsplit, parts, status, n_clear, st);
    }
}

}  // namespace moe
