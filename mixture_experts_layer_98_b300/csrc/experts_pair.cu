// experts_pair.cu -- grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// The same two GEMMs as experts_tc.cu -- the SwiGLU expert MLP
// down(silu(gate(x)) ⊙ up(x)) with per-expert gate_proj / up_proj [I,H] and
// down_proj [H,I] (csdn page "MoE架构深度解析：128专家与8激活的智能路由",
// section "128个专家网络的组织结构与参数分布"), scaled by the pair's routing
// weight (Qwen3MoeSparseMoeBlock.forward on the cnblogs page
// "大模型-qwen3 MoE 详细解读") -- with a 2-CTA cluster as the unit of work.
// One pair MMA computes a 256-row x 256-column tile; each CTA stages 128 of
// the A rows and 128 of the B rows, so per 64-deep k-block a CTA writes 32 KB
// into shared memory and its tensor core reads 8 KB of operands per K=16 step
// (the peer supplies the other half of B).  A single CTA computing a 128x256
// tile writes 48 KB and reads 12 KB for the same tensor work; at full MMA
// rate that is more shared-memory traffic than an SM moves, and it held the
// single-CTA kernels near two thirds of the tensor pipe.
//
// Tiles are up to 256 rows of one expert (the dispatch step's tile table at
// 256 rows); a tile of at most 128 rows (usually an expert's last) runs the
// M=128 pair MMA, 64 rows per CTA.
//
//   gate/up, n-block nt = 128 intermediate columns from c0 = 128 nt:
//     CTA 0's B rows: W_gate c0..c0+63, then W_up c0..c0+63   (MMA n 0..127)
//     CTA 1's B rows: W_gate c0+64..c0+127, then W_up c0+64.. (MMA n 128..255)
//     so a TMEM lane holds matching gate and up columns of its row:
//     h[r, c0 + 64 j + i] = bf16(silu(D[r, 128 j + i]) · D[r, 128 j + 64 + i])
//   down, n-block nt = 256 output columns from 256 nt:
//     CTA c's B rows: W_down rows 256 nt + 128 c .. +127 of the expert;
//     Y[perm_tok[r]·K + perm_slot[r], 256 nt + n] = bf16(w_perm[r] · D[r, n])
//
// Roles (192 threads per CTA, one CTA per SM):
//   warp 0     both CTAs: TMA producer of the CTA's own A rows and B rows into
//              a 6-stage ring (pair-form copies: every stage's bytes, both
//              CTAs', complete on CTA 0's full barrier, which CTA 0's
//              producer arms with the pair's total)
//   warp 1     both CTAs: TMEM owner (512 columns = a double-buffered
//              256-column accumulator, allocated for the pair).  CTA 0: MMA
//              issuer -- waits its full barrier, issues the pair MMAs, and
//              commits each stage's empty barrier and the accumulator's full
//              barrier in both CTAs (multicast)
//   warps 2-5  both CTAs: epilogue over the CTA's own TMEM lanes (its rows);
//              each warp arrives on CTA 0's accumulator-empty barrier (8).
// Packed weights are read through tensor maps over the packed blocks (boxes
// copied as stored, no swizzle), so that they too complete on CTA 0's barrier.
// Every wait is bounded (2 s): on expiry the CTA records MOE_ERR_TIMEOUT, lets
// its copies and MMAs finish, and both CTAs meet at the final cluster barrier
// before the pair frees TMEM and exits.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kHalfRows = 128;         // A rows per CTA (M=256 tile)
constexpr int kBK = 64;                // 64 bf16 = 128 bytes: one swizzle row
constexpr int kBN = 256;               // N of the pair MMA
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kABytes = kHalfRows * kBK * 2;   // 16 KB
constexpr int kBBytes = (kBN / 2) * kBK * 2;   // 16 KB: this CTA's half of B
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr uint32_t kIdesc256 = ptx::idesc_bf16_f32(256, kBN);
constexpr uint32_t kIdesc128 = ptx::idesc_bf16_f32(128, kBN);
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint64_t kSettleNs = 100000ull;  // after an abort: copies in flight land
constexpr uint16_t kBothCtas = 0x3;

enum { kGateUp = 0, kDown = 1 };

struct PairParams {
    const RowTile* tiles;   // 256-row tiles
    const int32_t* n_tiles;
    int n_nt;               // n-blocks per row tile
    int num_kb;             // k-blocks of 64
    int b_rows_per_expert;  // I (gate/up) or H (down)
    __nv_bfloat16* out;     // h [P, I] or Y [P, H] (token-major)
    int out_ld;
    const float* w_perm;
    int32_t* status;
    // packed weights: the B maps cover the packed blocks as 128-byte rows
    int packed;
    int b_blocks_per_expert;
    const int32_t* perm_tok;
    const int32_t* perm_slot;
    int K;
    float* out32;           // down: fp32 Y [P, H] (under a capacity); null: bf16 Y in out
};

__device__ __forceinline__ void store8(__nv_bfloat16* dst, const float (&v)[8]) {
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = o;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmA64,
                             const __grid_constant__ CUtensorMap tmB0,
                             const __grid_constant__ CUtensorMap tmB1, const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cr = ptx::cluster_ctarank();  // 0: issues the pair MMAs
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull_bar[b], 1);
            ptx::mbar_init(&tempty_bar[b], 8);
        }
        ptx::mbar_init(&drain_bar, 1);
        abort_s = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmA64);
        ptx::prefetch_tmap(&tmB0);
        ptx::prefetch_tmap(&tmB1);
    }
    // Both CTAs resident and their barriers initialised before anything
    // arrives remotely or the pair allocates TMEM.
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tmem_alloc_pair(&tmem_base_s, kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    pdl_trigger();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    pdl_wait();  // the prologue above overlaps the previous kernel's tail
    const int total = (*p.n_tiles) * p.n_nt;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer (both CTAs) ----------------
            const uint32_t full0 = ptx::mapa_shared(&full_bar[0], 0);  // CTA 0's barriers
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int item = pair; item < total && ok; item += npairs) {
                const RowTile tl = p.tiles[item / p.n_nt];
                const int nt = item % p.n_nt;
                const bool m256 = tl.nrows > kHalfRows;
                const int arow = tl.row0 + (int)cr * (m256 ? kHalfRows : kHalfRows / 2);
                const uint32_t a_bytes = m256 ? kABytes : kABytes / 2;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::mbar_wait_bounded<true>(&empty_bar[stage], phase ^ 1u, &abort_s,
                                                      kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + stage * kStageBytes;
                    uint8_t* sB = sA + kABytes;
                    const uint32_t fb = full0 + 8u * (uint32_t)stage;
                    if (cr == 0)  // both CTAs' bytes of this stage
                        ptx::mbar_arrive_expect_tx(&full_bar[stage], 2 * (a_bytes + kBBytes));
                    ptx::tma_load_2d_pair(sA, m256 ? &tmA : &tmA64, fb, kb * kBK, arow);
                    if (MODE == kGateUp) {
                        // this CTA's 64 gate rows and 64 up rows of the n-block
                        int c0, c1;
                        if (p.packed) {
                            const long long blk =
                                ((long long)tl.expert * p.b_blocks_per_expert + nt) * p.num_kb + kb;
                            c0 = 0;
                            c1 = (int)(blk * kPackRows) + (int)cr * 64;
                        } else {
                            c0 = kb * kBK;
                            c1 = tl.expert * p.b_rows_per_expert + nt * 128 + (int)cr * 64;
                        }
                        ptx::tma_load_2d_pair(sB, &tmB0, fb, c0, c1);
                        ptx::tma_load_2d_pair(sB + kBBytes / 2, &tmB1, fb, c0, c1);
                    } else {
                        int c0, c1;
                        if (p.packed) {
                            const long long blk = ((long long)tl.expert * p.b_blocks_per_expert +
                                                   2 * nt + cr) * p.num_kb + kb;
                            c0 = 0;
                            c1 = (int)(blk * kPackRows);
                        } else {
                            c0 = kb * kBK;
                            c1 = tl.expert * p.b_rows_per_expert + nt * kBN + (int)cr * 128;
                        }
                        ptx::tma_load_2d_pair(sB, &tmB0, fb, c0, c1);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicExch(p.status, MOE_ERR_TIMEOUT);
                // the copies this CTA issued complete on CTA 0's barrier, which
                // this CTA cannot wait on: give them time to land before exiting
                const long long t0 = clock64();
                while (clock64() - t0 < (long long)(kSettleNs * 2.032)) {
                }
            } else {
                // the last stages' empty arrivals (multicast commits from CTA 0)
                // land before the CTA exits
                int dummy = 0;
                for (int n = 0; n < kStages; ++n) {
                    // stage (stage + n) % kStages was last filled in round phase ^ 1 (if
                    // it precedes `stage`) -- wait for that round's consumption
                    const int s = (stage + n) % kStages;
                    const uint32_t par = (s >= stage) ? (phase ^ 1u) : phase;
                    ptx::mbar_wait_bounded<true>(&empty_bar[s], par, &dummy, kTimeoutNs);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && cr == 0) {
            // ---------------- pair MMA issuer (CTA 0) ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int item = pair; item < total && ok; item += npairs) {
                const uint32_t idesc =
                    p.tiles[item / p.n_nt].nrows > kHalfRows ? kIdesc256 : kIdesc128;
                if (!ptx::mbar_wait_bounded<true>(&tempty_bar[acc], acc_phase ^ 1u, &abort_s,
                                                  kTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    // both CTAs' bytes of the stage have landed
                    if (!ptx::mbar_wait_bounded<true>(&full_bar[stage], phase, &abort_s,
                                                      kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint64_t adesc = ptx::desc_sw128_kmajor(a_addr);
                    const uint64_t bdesc = ptx::desc_sw128_kmajor(a_addr + kABytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)  // K = 16 per MMA: +32 bytes
                        ptx::mma_bf16_pair(d, adesc + 2u * k, bdesc + 2u * k, idesc,
                                           (kb | k) != 0 ? 1u : 0u);
                    ptx::mma_commit_pair(&empty_bar[stage], kBothCtas);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(&tfull_bar[acc], kBothCtas);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) atomicExch(p.status, MOE_ERR_TIMEOUT);
            // every pair MMA issued has completed before TMEM is freed
            ptx::mma_commit_pair(&drain_bar, 0x1);
            int dummy = 0;
            ptx::mbar_wait_bounded(&drain_bar, 0u, &dummy, kTimeoutNs);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        const uint32_t tempty0 = ptx::mapa_shared(&tempty_bar[0], 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = pair; item < total; item += npairs) {
            const RowTile tl = p.tiles[item / p.n_nt];
            const int nt = item % p.n_nt;
            int ok = 1;
            if (lane == 0)
                ok = ptx::mbar_wait_bounded<true>(&tfull_bar[acc], acc_phase, &abort_s,
                                                  kTimeoutNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) atomicExch(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            // M=256: lane l of this CTA = tile row 128 cr + l, all 256 n.
            // M=128: lane i < 64 = tile row 64 cr + i, n 0..127; lane 64 + i =
            // the same row, n 128..255 (TMEM columns 0..127 either way).
            const bool m256 = tl.nrows > kHalfRows;
            const int trow = m256 ? (int)cr * 128 + q * 32 + lane
                                  : (int)cr * 64 + (q & 1) * 32 + lane;
            const int nh = m256 ? 0 : (q >> 1);  // M=128: which half of n this lane holds
            const bool valid = trow < tl.nrows;
            const size_t row = (size_t)tl.row0 + trow;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
            if (MODE == kGateUp) {
                // j: which 64-column group of h; gate at TMEM 128 j', up at 128 j' + 64
                const int j0 = m256 ? 0 : nh, j1 = m256 ? 2 : nh + 1;
                for (int j = j0; j < j1; ++j) {
                    const uint32_t tg = tbase + (uint32_t)((m256 ? j : 0) * 128);
#pragma unroll 1
                    for (int c = 0; c < 64; c += 32) {
                        uint32_t g[32], u[32];
                        ptx::tmem_ld32(tg + c, g);
                        ptx::tmem_ld32(tg + 64 + c, u);
                        ptx::tmem_ld_wait();
                        if (valid) {
                            __nv_bfloat16* dst =
                                p.out + row * p.out_ld + (size_t)nt * 128 + j * 64 + c;
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                float hv[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    hv[i] = silu_f(__uint_as_float(g[8 * v + i])) *
                                            __uint_as_float(u[8 * v + i]);
                                store8(dst + 8 * v, hv);
                            }
                        }
                    }
                }
            } else {
                const float wr = valid ? p.w_perm[row] : 0.f;
                const size_t yrow =
                    valid ? (size_t)p.perm_tok[row] * p.K + (size_t)p.perm_slot[row] : 0;
                const int ncols = m256 ? kBN : kBN / 2;
                __nv_bfloat16* dst0 = p.out + yrow * p.out_ld + (size_t)nt * kBN + nh * (kBN / 2);
#pragma unroll 1
                for (int c = 0; c < ncols; c += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c, v);
                    ptx::tmem_ld_wait();
                    if (valid && p.out32) {
                        float4* dst = reinterpret_cast<float4*>(
                            p.out32 + yrow * p.out_ld + (size_t)nt * kBN + nh * (kBN / 2) + c);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(wr * __uint_as_float(v[4 * j + 0]),
                                                 wr * __uint_as_float(v[4 * j + 1]),
                                                 wr * __uint_as_float(v[4 * j + 2]),
                                                 wr * __uint_as_float(v[4 * j + 3]));
                    } else if (valid) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) o[i] = wr * __uint_as_float(v[8 * j + i]);
                            store8(dst0 + c + 8 * j, o);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_remote(tempty0 + 8u * (uint32_t)acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    // Both CTAs are done with each other's barriers, shared memory and TMEM.
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---- host side ----------------------------------------------------------------

template <int MODE>
int max_pairs() {
    static int cached[64] = {};  // per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 74);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)grouped_gemm_pair_kernel<MODE>, &cfg) !=
            cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        n = num_sms() / 2;
    }
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

// B0 / B1: the row-major [b_rows, a_cols] weight matrices, or with p.packed
// their packed blocks (b_rows x a_cols elements as 128-byte rows).
template <int MODE>
cudaError_t launch_pair(const void* A, uint64_t a_rows, uint64_t a_cols, const void* B0,
                        const void* B1, uint64_t b_rows, uint32_t b_box, const PairParams& p,
                        long long max_items, cudaStream_t st) {
    CUtensorMap ma, ma64, mb0, mb1;
    if (!make_tma_2d(&ma, A, a_rows, a_cols, kHalfRows) ||
        !make_tma_2d(&ma64, A, a_rows, a_cols, kHalfRows / 2))
        return cudaErrorInvalidValue;
    if (p.packed) {
        const uint64_t rows = b_rows * a_cols / kPackCols;
        if (!make_tma_packed(&mb0, B0, rows, b_box) || !make_tma_packed(&mb1, B1, rows, b_box))
            return cudaErrorInvalidValue;
    } else if (!make_tma_2d(&mb0, B0, b_rows, a_cols, b_box) ||
               !make_tma_2d(&mb1, B1, b_rows, a_cols, b_box)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = ensure_smem((const void*)grouped_gemm_pair_kernel<MODE>, kSmemBytes);
    if (err != cudaSuccess) return err;
    long long pairs = max_pairs<MODE>();
    if (pairs > max_items) pairs = max_items;
    if (pairs < 1) pairs = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE>, ma, ma64, mb0, mb1, p);
    count_launches(1);
    return err;
}

}  // namespace

bool experts_pair_supported(const Sizes& s) { return s.I % 128 == 0 && s.H % 256 == 0; }

cudaError_t launch_experts_pair(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                                cudaStream_t st, cudaEvent_t ev_mid) {
    if (!experts_pair_supported(s)) return cudaErrorInvalidValue;
    const long long P = s.P();
    const long long max_tiles = s.max_tiles(kPairRows);
    const bool packed = W.packed != nullptr;
    PairParams p{};
    p.tiles = ws.tiles;
    p.n_tiles = ws.n_tiles;
    p.status = ws.status;
    p.w_perm = ws.w_perm;

    // gate/up: A = x_perm rows; B = 64 gate rows over 64 up rows per CTA
    p.n_nt = s.I / 128;
    p.num_kb = s.H / kBK;
    p.b_rows_per_expert = s.I;
    p.out = ws.hbuf;
    p.out_ld = s.I;
    p.packed = packed ? 1 : 0;
    p.b_blocks_per_expert = s.I / kPackRows;
    cudaError_t err = launch_pair<kGateUp>(
        ws.x_perm, P, s.H, packed ? (const void*)W.packed_gate(s) : W.gate,
        packed ? (const void*)W.packed_up(s) : W.up, (uint64_t)s.E * s.I, 64, p,
        max_tiles * p.n_nt, st);
    if (err != cudaSuccess) return err;
    if (ev_mid) cudaEventRecord(ev_mid, st);

    // down: A = h rows; B = 128 W_down rows per CTA
    p.n_nt = s.H / kBN;
    p.num_kb = s.I / kBK;
    p.b_rows_per_expert = s.H;
    p.out = ws.ybuf;
    p.out_ld = s.H;
    p.b_blocks_per_expert = s.H / kPackRows;
    p.perm_tok = ws.perm_tok;
    p.perm_slot = ws.perm_slot;
    p.K = s.K;
    p.out32 = ws.ybuf_f32;
    const void* bd = packed ? (const void*)W.packed_down(s) : W.down;
    return launch_pair<kDown>(ws.hbuf, P, s.I, bd, bd, (uint64_t)s.E * s.H, 128, p,
                              max_tiles * p.n_nt, st);
}

}  // namespace moe
