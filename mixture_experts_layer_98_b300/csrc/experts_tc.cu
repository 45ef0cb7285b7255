// experts_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores.
//
// The expert is the SwiGLU MLP down(silu(gate(x)) ⊙ up(x)) with per-expert
// gate_proj / up_proj [I,H] and down_proj [H,I] (csdn page
// "MoE架构深度解析：128专家与8激活的智能路由", section
// "128个专家网络的组织结构与参数分布"), scaled by the pair's routing weight
// (Qwen3MoeSparseMoeBlock.forward on the cnblogs page "大模型-qwen3 MoE 详细解读").
// The rows of all experts are contiguous per expert after dispatch, so every
// expert's MLP is one GEMM over its row range; the kernels walk a table of
// 128-row tiles (one expert each) written on the device by the dispatch step.
//
//   gate/up : D[128, BN] = X[rows, H] · [Wg[e, n-block]; Wu[e, n-block]]ᵀ
//             (the B tile stacks BN/2 gate rows over BN/2 up rows, so one MMA
//             computes both); epilogue h = bf16(silu(D_gate) · D_up)
//   down    : D[128, BN] = h[rows, I] · Wd[e, n-block]ᵀ
//             epilogue Y = bf16(w_row · D) (fp32 under an expert capacity),
//             stored token-major (row t*K + k of the pair in dispatch row r:
//             t = perm_tok[r], k = perm_slot[r])
//
// Persistent, warp-specialised CTA (one per SM, 192 threads):
//   warp 0     TMA producer: A tile 128x64 and two B half-tiles (BN/2)x64 per
//              k-block into a 4-stage ring of 128-byte-swizzled buffers
//   warp 1     owns TMEM (2 x BN fp32 columns: a double-buffered accumulator)
//              and issues tcgen05.mma M=128 N=BN K=16 (4 per k-block); a tile
//              of at most 64 rows (an expert's last) loads a 64-row A box and
//              issues M=64 MMAs, half the tensor work of a padded 128-row tile
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//              32·(w%4)..+31 = tile rows), fused activation / scaling, bf16
//              stores of the rows that belong to the tile's expert
// Every wait is bounded (2 s); on expiry the CTA records MOE_ERR_TIMEOUT in
// the workspace status word, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = kTcRows;  // 128 rows per tile (M of the MMA)
constexpr int kBK = 64;       // 64 bf16 = 128 bytes: one swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint64_t kTimeoutNs = 2000000000ull;

enum { kGateUp = 0, kDown = 1 };

struct TcParams {
    const RowTile* tiles;
    const int32_t* n_tiles;
    int n_nt;               // N tiles per row tile
    int num_kb;             // k-blocks of 64
    int b_rows_per_expert;  // I (gate/up) or H (down)
    __nv_bfloat16* out;     // h [P, I] or Y [P, H]
    int out_ld;
    const float* w_perm;    // routing weight per row (down)
    int32_t* status;
    // Packed weights (null: row-major through the B tensor maps): block bases of
    // the two B halves and 128-row blocks per expert of the B matrix.
    const char* bpk0;
    const char* bpk1;
    int b_blocks_per_expert;
    // down: Y is stored token-major, row perm_tok[r] * K + perm_slot[r]
    const int32_t* perm_tok;
    const int32_t* perm_slot;
    int K;
    float* out32;           // down: fp32 Y [P, H] (under a capacity); null: bf16 Y in out
};

template <int MODE, int BN>
struct TcCfg {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBHalfBytes = (BN / 2) * kBK * 2;
    static constexpr int kStageBytes = kABytes + 2 * kBHalfBytes;
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
    static constexpr uint32_t kTmemCols = 2 * BN;
    static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, BN);
    static constexpr uint32_t kIdesc64 = ptx::idesc_bf16_f32(kBM / 2, BN);
};

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmA64,
                           const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const TcParams p) {
    using C = TcCfg<MODE, BN>;
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
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
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmA64);
        ptx::prefetch_tmap(&tmB0);
        ptx::prefetch_tmap(&tmB1);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&tmem_base_s, C::kTmemCols);
        ptx::tmem_relinquish();
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
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const RowTile tl = p.tiles[item / p.n_nt];
                const int nt = item % p.n_nt;
                int b0, b1;    // B rows in the row-major matrices
                int b0h, b1h;  // the halves' 128-row blocks within the expert (packed)
                if (MODE == kGateUp) {
                    b0 = b1 = tl.expert * p.b_rows_per_expert + nt * (BN / 2);
                    b0h = b1h = nt;
                } else {
                    b0 = tl.expert * p.b_rows_per_expert + nt * BN;
                    b1 = b0 + BN / 2;
                    b0h = 2 * nt;
                    b1h = 2 * nt + 1;
                }
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_s,
                                                kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + stage * C::kStageBytes;
                    uint8_t* sB = sA + C::kABytes;
                    if (tl.nrows <= kBM / 2) {  // a 64-row tile: M=64 MMA, 64-row A box
                        ptx::mbar_arrive_expect_tx(&full_bar[stage],
                                                   C::kStageBytes - C::kABytes / 2);
                        ptx::tma_load_2d(sA, &tmA64, &full_bar[stage], kb * kBK, tl.row0);
                    } else {
                        ptx::mbar_arrive_expect_tx(&full_bar[stage], C::kStageBytes);
                        ptx::tma_load_2d(sA, &tmA, &full_bar[stage], kb * kBK, tl.row0);
                    }
                    if (BN == 2 * kPackRows && p.bpk0) {
                        // packed: each B half is one contiguous 16 KB block
                        const size_t blk0 =
                            ((size_t)tl.expert * p.b_blocks_per_expert + (size_t)b0h) * p.num_kb + kb;
                        const size_t blk1 =
                            ((size_t)tl.expert * p.b_blocks_per_expert + (size_t)b1h) * p.num_kb + kb;
                        ptx::bulk_load(sB, p.bpk0 + blk0 * kPackBlockBytes, C::kBHalfBytes,
                                       &full_bar[stage]);
                        ptx::bulk_load(sB + C::kBHalfBytes, p.bpk1 + blk1 * kPackBlockBytes,
                                       C::kBHalfBytes, &full_bar[stage]);
                    } else {
                        ptx::tma_load_2d(sB, &tmB0, &full_bar[stage], kb * kBK, b0);
                        ptx::tma_load_2d(sB + C::kBHalfBytes, &tmB1, &full_bar[stage], kb * kBK,
                                         b1);
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicExch(p.status, MOE_ERR_TIMEOUT);
                // Let the copies already issued land before the CTA exits.
                int dummy = 0;
                const long long first = issued > kStages ? issued - kStages : 0;
                for (long long n = first; n < issued; ++n)
                    ptx::mbar_wait_bounded(&full_bar[n % kStages], (uint32_t)((n / kStages) & 1),
                                           &dummy, kTimeoutNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const uint32_t idesc =
                    p.tiles[item / p.n_nt].nrows <= kBM / 2 ? C::kIdesc64 : C::kIdesc;
                if (!ptx::mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, &abort_s,
                                            kTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::mbar_wait_bounded(&full_bar[stage], phase, &abort_s, kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + stage * C::kStageBytes);
                    const uint64_t adesc = ptx::desc_sw128_kmajor(a_addr);
                    const uint64_t bdesc = ptx::desc_sw128_kmajor(a_addr + C::kABytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)  // K = 16 per MMA: +32 bytes
                        ptx::mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, idesc,
                                      (kb | k) != 0 ? 1u : 0u);
                    ptx::mma_commit(&empty_bar[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(&tfull_bar[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) atomicExch(p.status, MOE_ERR_TIMEOUT);
            // All MMAs issued by this thread complete before TMEM is freed.
            ptx::mma_commit(&drain_bar);
            int dummy = 0;
            ptx::mbar_wait_bounded(&drain_bar, 0u, &dummy, kTimeoutNs);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            const RowTile tl = p.tiles[item / p.n_nt];
            const int nt = item % p.n_nt;
            int ok = 1;
            if (lane == 0)
                ok = ptx::mbar_wait_bounded(&tfull_bar[acc], acc_phase, &abort_s, kTimeoutNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) atomicExch(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            // M=128: tile row q*32 + lane sits in TMEM lane q*32 + lane.  M=64 (a
            // tile of <= 64 rows): row q*16 + l sits in lane q*32 + l, l < 16.
            const bool m64 = tl.nrows <= kBM / 2;
            const int r = m64 ? q * 16 + lane : q * 32 + lane;
            const bool valid = (!m64 || lane < 16) && r < tl.nrows;
            const size_t row = (size_t)tl.row0 + r;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (MODE == kGateUp) {
                constexpr int kHalf = BN / 2;
#pragma unroll 1
                for (int c = 0; c < kHalf; c += 32) {
                    uint32_t g[32], u[32];
                    ptx::tmem_ld32(tbase + c, g);
                    ptx::tmem_ld32(tbase + kHalf + c, u);
                    ptx::tmem_ld_wait();
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.out_ld +
                                                              (size_t)nt * kHalf + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float hv[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                hv[i] = silu_f(__uint_as_float(g[8 * j + i])) *
                                        __uint_as_float(u[8 * j + i]);
                            uint4 o;
                            o.x = pack_bf16x2(hv[0], hv[1]);
                            o.y = pack_bf16x2(hv[2], hv[3]);
                            o.z = pack_bf16x2(hv[4], hv[5]);
                            o.w = pack_bf16x2(hv[6], hv[7]);
                            dst[j] = o;
                        }
                    }
                }
            } else {
                const float wr = valid ? p.w_perm[row] : 0.f;
                const size_t yrow =
                    valid ? (size_t)p.perm_tok[row] * p.K + (size_t)p.perm_slot[row] : 0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c, v);
                    ptx::tmem_ld_wait();
                    if (valid && p.out32) {
                        float4* dst = reinterpret_cast<float4*>(p.out32 + yrow * p.out_ld +
                                                                (size_t)nt * BN + c);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(wr * __uint_as_float(v[4 * j + 0]),
                                                 wr * __uint_as_float(v[4 * j + 1]),
                                                 wr * __uint_as_float(v[4 * j + 2]),
                                                 wr * __uint_as_float(v[4 * j + 3]));
                    } else if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(p.out + yrow * p.out_ld +
                                                              (size_t)nt * BN + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 o;
                            o.x = pack_bf16x2(wr * __uint_as_float(v[8 * j + 0]),
                                              wr * __uint_as_float(v[8 * j + 1]));
                            o.y = pack_bf16x2(wr * __uint_as_float(v[8 * j + 2]),
                                              wr * __uint_as_float(v[8 * j + 3]));
                            o.z = pack_bf16x2(wr * __uint_as_float(v[8 * j + 4]),
                                              wr * __uint_as_float(v[8 * j + 5]));
                            o.w = pack_bf16x2(wr * __uint_as_float(v[8 * j + 6]),
                                              wr * __uint_as_float(v[8 * j + 7]));
                            dst[j] = o;
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---- host side ----------------------------------------------------------------

template <int MODE, int BN>
cudaError_t launch_tc(const void* A, uint64_t a_rows, uint64_t a_cols, const void* B0,
                      const void* B1, uint64_t b_rows, const TcParams& p, long long max_items,
                      cudaStream_t st) {
    using C = TcCfg<MODE, BN>;
    CUtensorMap ma, ma64, mb0, mb1;
    if (!make_tma_2d(&ma, A, a_rows, a_cols, kBM) || !make_tma_2d(&ma64, A, a_rows, a_cols, kBM / 2))
        return cudaErrorInvalidValue;
    if (p.bpk0) {  // packed weights: the B maps are not used
        mb0 = ma;
        mb1 = ma;
    } else if (!make_tma_2d(&mb0, B0, b_rows, a_cols, BN / 2) ||
               !make_tma_2d(&mb1, B1, b_rows, a_cols, BN / 2)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = ensure_smem((const void*)grouped_gemm_tc_kernel<MODE, BN>, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    long long grid = num_sms();
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    err = launch_pdl(grouped_gemm_tc_kernel<MODE, BN>, dim3((unsigned)grid), dim3(kThreads),
                     C::kSmemBytes, st, ma, ma64, mb0, mb1, p);
    count_launches(1);
    return err;
}

}  // namespace

cudaError_t launch_experts_tcgen05(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                                   cudaStream_t st, cudaEvent_t ev_mid) {
    const long long P = s.P();
    const long long max_tiles = s.max_tiles(kBM);
    const bool packed = W.packed != nullptr;
    if (packed && !packed_supported(s.H, s.E, s.I)) return cudaErrorInvalidValue;
    TcParams p{};
    p.tiles = ws.tiles;
    p.n_tiles = ws.n_tiles;
    p.status = ws.status;
    p.w_perm = ws.w_perm;

    // gate/up: A = x_perm rows of the tile; B = [BN/2 gate rows ; BN/2 up rows] of expert e
    p.num_kb = s.H / kBK;
    p.b_rows_per_expert = s.I;
    p.out = ws.hbuf;
    p.out_ld = s.I;
    p.bpk0 = packed ? W.packed_gate(s) : nullptr;
    p.bpk1 = packed ? W.packed_up(s) : nullptr;
    p.b_blocks_per_expert = s.I / kPackRows;
    cudaError_t err;
    if (s.I % 128 == 0) {
        p.n_nt = s.I / 128;
        err = launch_tc<kGateUp, 256>(ws.x_perm, P, s.H, W.gate, W.up, (uint64_t)s.E * s.I, p,
                                      max_tiles * p.n_nt, st);
    } else {
        p.n_nt = s.I / 64;
        err = launch_tc<kGateUp, 128>(ws.x_perm, P, s.H, W.gate, W.up, (uint64_t)s.E * s.I, p,
                                      max_tiles * p.n_nt, st);
    }
    if (err != cudaSuccess) return err;
    if (ev_mid) cudaEventRecord(ev_mid, st);

    // down: A = h rows of the tile; B = W_down rows [n0, n0 + BN) of expert e
    p.num_kb = s.I / kBK;
    p.b_rows_per_expert = s.H;
    p.out = ws.ybuf;
    p.out_ld = s.H;
    p.bpk0 = packed ? W.packed_down(s) : nullptr;
    p.bpk1 = p.bpk0;
    p.b_blocks_per_expert = s.H / kPackRows;
    p.perm_tok = ws.perm_tok;
    p.perm_slot = ws.perm_slot;
    p.K = s.K;
    p.out32 = ws.ybuf_f32;
    if (s.H % 256 == 0) {
        p.n_nt = s.H / 256;
        err = launch_tc<kDown, 256>(ws.hbuf, P, s.I, W.down, W.down, (uint64_t)s.E * s.H, p,
                                    max_tiles * p.n_nt, st);
    } else if (s.H % 128 == 0) {
        p.n_nt = s.H / 128;
        err = launch_tc<kDown, 128>(ws.hbuf, P, s.I, W.down, W.down, (uint64_t)s.E * s.H, p,
                                    max_tiles * p.n_nt, st);
    } else {
        p.n_nt = s.H / 64;
        err = launch_tc<kDown, 64>(ws.hbuf, P, s.I, W.down, W.down, (uint64_t)s.E * s.H, p,
                                   max_tiles * p.n_nt, st);
    }
    return err;
}

}  // namespace moe
