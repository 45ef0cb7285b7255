// experts_q4_mma.cu -- decode batches on 4-bit group-quantised experts:
// weights dequantised straight into the registers of warp-level tensor-core
// MMAs (mma.sync m16n8k16, bf16 inputs, fp32 accumulators).
//
// Same function as experts_q4.cu (the SwiGLU expert MLP of the csdn page
// "MoE架构深度解析：128专家与8激活的智能路由", section
// "128个专家网络的组织结构与参数分布", on the 4-bit weights of its section
// "参数量化与存储优化", layout and reading in quant.cu; the routing-weight
// scaling of Qwen3MoeSparseMoeBlock.forward on the cnblogs page
// "大模型-qwen3 MoE 详细解读").
//
// Why a second kernel.  At decode sizes an expert receives 1-8 token rows, so
// the expert MLP is a matrix-vector product that streams 4.25 bits per
// weight from HBM: about 40 weights per SM cycle at the measured copy
// bandwidth.  The tcgen05 kernel of experts_q4.cu needs every dequantised
// weight in shared memory as bf16 (written by threads, read by the MMA), about
// 5 bytes of shared-memory traffic per weight, which caps it near 23 weights
// per cycle (128 B/cycle); with the weights on the MMA's M side instead, an
// MMA takes about M cycles whatever its N, 16 weights per cycle.  Here the
// dequantised weights never leave the registers: they are the A fragments of
// m16n8k16 MMAs whose B fragments are the tile's tokens, 8 per MMA.
//
// Fragment mapping.  A thread (g = lane / 4, c = lane % 4) of the warp that
// owns weight rows R..R+15 reads, per 64-column k-block, the adjacent code
// words 2c and 2c + 1 of rows R + g and R + g + 8 (one 8-byte load per row;
// quant.cu: word c' of a row holds columns 8c'..8c'+7, pair j = columns
// 8c'+2j, 8c'+2j+1).  k-step t (0..3) of the block takes pair 2(t%2) of word
// 2c + t/2 as the fragment's columns 2c, 2c+1 and pair 2(t%2)+1 as its columns
// 2c+8, 2c+9: fragment column f of step t is block column
// 16((f%8)/2) + 8(t/2) + 4(t%2) + 2(f/8) + f%2, a permutation of the block's
// 64 columns.  The token fragment applies the same permutation: thread (g, c)
// needs, over the four steps, the 16 consecutive bf16 of token g from column
// 16c, two 16-byte loads from the 128-byte swizzled row.  The sum over k is
// order-free, so the MMA computes the exact products of the bf16 forward on
// the dequantised weights, accumulated in fp32 in another order.
//
// Work items: gate/up (row tile, 128 I rows: the gate rows and the same up
// rows), down (row tile, 256 H rows), on row tiles of at most 16 tokens
// (kQ4MmaRows), with K slices fitted to two CTAs per SM (q4mma_plan: an item
// count that does not fill the grid's last round leaves SMs idle for a whole
// item, and a decode batch has a few hundred items); warp w of the 8 consumer warps owns two
// 16-row MMA tiles: gate/up rows 16w.. of W_gate and of W_up (so that
// silu(gate)·up needs no exchange), down rows 32w.. and 32w+16.. .  With K
// slices each warp writes its slice accumulators and bumps its own counter of
// the item; the slice whose warp arrives last adds, for that warp's outputs,
// the slices in slice order and runs their epilogue.
//
// Roles: warp 0 producer (token boxes by TMA, code and scale blocks by bulk
// copy into a ring of stages, one 128-column group a stage: a group's scales
// serve both its k-blocks, and the per-stage waits and releases are paid once
// per 128 columns), warps 1-8 consumers.  Every wait is bounded
// (2 s); on expiry the CTA records MOE_ERR_TIMEOUT, lets its copies land and
// exits (no CTA-wide barrier follows the main loops).
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kConsumers = 8;
constexpr int kThreadsM = 32 * (kConsumers + 1);
constexpr int kBK = 64;
constexpr int kTokBox = 8;         // token rows per TMA box: one MMA's N
constexpr int kMaxStages = 16;
constexpr uint64_t kTimeoutNs = 2000000000ull;

enum { kGateUp = 0, kDown = 1 };

constexpr int kKbPerStage = 2;     // k-blocks per stage: one 128-column scale group

// Stage (one 128-column group of the item's 256 weight rows): for each of its
// two k-blocks NT token boxes (8 rows x 128 bytes, 128-byte swizzled, each on
// a 1024-byte boundary; box n of k-block h at (h·NT + n)·1024), then per plane
// the group's two 4 KB code blocks (contiguous in the packed layout, one 8 KB
// copy) and its 512-byte scale block.  Two CTAs per SM.
template <int NT>
struct MmaCfg {
    static_assert(NT * kTokBox <= kQ4MmaRows, "a stage holds a whole row tile");
    static constexpr int kTokOff = 0;
    static constexpr int kCodeOff = kKbPerStage * NT * kTokBox * 128;
    static constexpr int kPlaneCodeBytes = kKbPerStage * kQ4CodeBlockBytes;
    static constexpr int kScaleOff = kCodeOff + 2 * kPlaneCodeBytes;
    static constexpr int kBytes = kScaleOff + 2 * kQ4ScaleBlockBytes;
    static constexpr int kCtasPerSm = 2;
    static constexpr int kBudget = 112 * 1024 - 1024;
    static constexpr int kStages = kBudget / kBytes < kMaxStages ? kBudget / kBytes : kMaxStages;
    static constexpr int kSmemBytes = kStages * kBytes + 1024;
    static_assert(kBytes % 1024 == 0, "stages stay 1024-byte aligned");
    static_assert(kStages >= 4, "ring depth");
};

struct MmaParams {
    const RowTile* tiles;
    const int32_t* n_tiles;
    int n_nt;               // items per row tile: I / 128 (gate/up), H / 256 (down)
    int num_kb;             // k-blocks of 64
    int ksplit;
    int grp_per;            // 128-column groups per K slice
    float* partial;         // [items][ksplit][2][part_rows][128] slice accumulators
    int part_rows;
    int32_t* counters;      // per item and consumer warp: arrivals of its slices
    __nv_bfloat16* out;     // h [P, I] or Y [P, H]
    int out_ld;
    const float* w_perm;
    const int32_t* perm_tok;
    const int32_t* perm_slot;
    int K;
    float* out32;           // down: fp32 Y [P, H] (under a capacity); null: bf16 Y in out
    int32_t* status;
    const char* codes0;     // first / second 128-row block of an item
    const char* codes1;
    const char* scales0;
    const char* scales1;
    int blocks_per_expert;  // 128-row blocks per expert of the matrix
    int groups;             // 128-column groups per weight row
};

struct Item {
    int pitem, tile, nt, ks, g0, g1;  // groups [g0, g1) of the slice
};

__device__ __forceinline__ Item item_of(const MmaParams& p, int item) {
    Item it;
    it.pitem = item / p.ksplit;
    it.ks = item % p.ksplit;
    it.tile = it.pitem / p.n_nt;
    it.nt = it.pitem % p.n_nt;
    it.g0 = it.ks * p.grp_per;
    it.g1 = min(p.groups, it.g0 + p.grp_per);
    return it;
}

// A code pair dequantised: bf16x2 of bf16(q·s + b), one rounding (as
// q4_dequant8).  m is a code word with one code per byte (its low or its
// high nibbles, masked and shifted to bits 0-3 of each byte); sel picks the
// pair's two bytes (0x4240: bytes 0 and 2, 0x4341: bytes 1 and 3) and puts
// the bf16 exponent byte of 128.0 above each, so the halves read 128 + q.
__device__ __forceinline__ uint32_t dq_perm(uint32_t m, uint32_t sel, __nv_bfloat162 s2,
                                            __nv_bfloat162 b2) {
    const __nv_bfloat162 k128 = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)0x4300u));
    const uint32_t t = __byte_perm(m, 0x43434343u, sel);
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&t);
    v = __hfma2(__hsub2(v, k128), s2, b2);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Output position of accumulator element (tile i, fragment row half fi) of
// consumer warp cw, thread row g: the item's plane (gate/up: 0 gate, 1 up;
// down: which 128-row block) and the feature within it (0..127).
template <int MODE>
__device__ __forceinline__ int plane_of(int cw, int i) {
    return MODE == kGateUp ? i : (32 * cw + 16 * i) >> 7;
}
template <int MODE>
__device__ __forceinline__ int row_in_block(int cw, int i) {
    return MODE == kGateUp ? 16 * cw : (32 * cw + 16 * i) & 127;
}

// The epilogue of one (token, feature) of an item from its fp32 sums: gate/up
// h = bf16(silu(g)·u) at feature nt·128 + f; down Y = bf16(w·y) at feature
// nt·256 + plane·128 + f of the pair's token-major row.
template <int MODE>
__device__ __forceinline__ void store_one(const MmaParams& p, const RowTile& tl, int nt,
                                          int tok, int plane, int f, float a, float b) {
    const size_t row = (size_t)tl.row0 + tok;
    if (MODE == kGateUp) {
        p.out[row * p.out_ld + (size_t)nt * 128 + f] = __float2bfloat16_rn(silu_f(a) * b);
    } else {
        const size_t yrow = (size_t)p.perm_tok[row] * p.K + (size_t)p.perm_slot[row];
        const size_t col = (size_t)nt * 256 + plane * 128 + f;
        if (p.out32)
            p.out32[yrow * p.out_ld + col] = p.w_perm[row] * a;
        else
            p.out[yrow * p.out_ld + col] = __float2bfloat16_rn(p.w_perm[row] * a);
    }
}

// One stage (a 128-column group) of a consumer warp: its two 16-row weight
// tiles against NN token boxes.  code_off / scale_off: this thread's code and
// scale words of each tile within the stage; tok0 / tok1: its two 16-byte
// chunks of token row g within a box.
template <int NT, int NN>
__device__ __forceinline__ void stage_mma(const uint8_t* st, const int (&code_off)[2],
                                          const int (&scale_off)[2], int tok0, int tok1,
                                          float (&acc)[2][NT][4]) {
    static_assert(NN <= NT, "boxes of a stage");
    using C = MmaCfg<NT>;
    // scale and bias of rows g, g + 8 of both tiles (the group's)
    __nv_bfloat162 s2[2][2], b2[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t sbw = *reinterpret_cast<const uint32_t*>(st + scale_off[i] + 32 * h);
            s2[i][h] = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)(sbw & 0xFFFFu)));
            b2[i][h] = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)(sbw >> 16)));
        }
#pragma unroll
    for (int h = 0; h < kKbPerStage; ++h) {
        // words 2c (x) and 2c + 1 (y) of rows g and g + 8 of both tiles
        uint2 wq[2][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint8_t* cp = st + code_off[i] + h * kQ4CodeBlockBytes;
            wq[i][0] = *reinterpret_cast<const uint2*>(cp);
            wq[i][1] = *reinterpret_cast<const uint2*>(cp + 8 * 32);
        }
        // token g, columns 16c..16c+7 (chunk 0) and 16c+8..16c+15 (chunk 1)
        uint4 tk[NN][2];
#pragma unroll
        for (int n = 0; n < NN; ++n) {
            const uint8_t* tp = st + C::kTokOff + (h * NT + n) * (kTokBox * 128);
            tk[n][0] = *reinterpret_cast<const uint4*>(tp + tok0);
            tk[n][1] = *reinterpret_cast<const uint4*>(tp + tok1);
        }
        // each code word split into its low and its high nibbles, one code per
        // byte: pair j of the word (codes at bits 4j and 16 + 4j) is then bytes
        // 0, 2 (j = 0, 1) or 1, 3 (j = 2, 3) of the low (even j) or high (odd j)
        // nibbles: a byte permute each (shifting and masking each pair into
        // place instead measured 7 % slower at 16 and 64 tokens)
        uint32_t lo[2][2][2], hi[2][2][2];  // [tile][row g / g + 8][word 2c / 2c + 1]
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                lo[i][r][0] = wq[i][r].x & 0x0F0F0F0Fu;
                hi[i][r][0] = (wq[i][r].x >> 4) & 0x0F0F0F0Fu;
                lo[i][r][1] = wq[i][r].y & 0x0F0F0F0Fu;
                hi[i][r][1] = (wq[i][r].y >> 4) & 0x0F0F0F0Fu;
            }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            // step t: pairs 2(t%2) (low nibbles) and 2(t%2)+1 (high) of word 2c + t/2
            const uint32_t sel = (t & 1) ? 0x4341u : 0x4240u;
            const int wi = t >> 1;
            uint32_t a[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                a[i][0] = dq_perm(lo[i][0][wi], sel, s2[i][0], b2[i][0]);  // row g, cols 2c, 2c+1
                a[i][1] = dq_perm(lo[i][1][wi], sel, s2[i][1], b2[i][1]);  // row g + 8
                a[i][2] = dq_perm(hi[i][0][wi], sel, s2[i][0], b2[i][0]);  // row g, cols 2c+8, 2c+9
                a[i][3] = dq_perm(hi[i][1][wi], sel, s2[i][1], b2[i][1]);  // row g + 8
            }
#pragma unroll
            for (int n = 0; n < NN; ++n) {
                const uint4& v = tk[n][t >> 1];
                const uint32_t b0 = (t & 1) ? v.z : v.x;
                const uint32_t b1 = (t & 1) ? v.w : v.y;
                mma_bf16_16816(acc[0][n], a[0], b0, b1);
                mma_bf16_16816(acc[1][n], a[1], b0, b1);
            }
        }
    }
}

template <int MODE, int NT>
__global__ void __launch_bounds__(kThreadsM, MmaCfg<NT>::kCtasPerSm)
    expert_q4_mma_kernel(const __grid_constant__ CUtensorMap tmA, const MmaParams p) {
    using C = MmaCfg<NT>;
    constexpr int kS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];   // boxes, codes, scales landed
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];  // all consumer warps read the stage
    __shared__ volatile int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], kConsumers);
        }
        abort_s = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
    }
    pdl_trigger();
    __syncthreads();
    pdl_wait();  // the prologue above overlaps the previous kernel's tail
    const int total = (*p.n_tiles) * p.n_nt * p.ksplit;

    if (warp == 0) {
        if (lane != 0) return;
        // ---------------- producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        const uint64_t pol_once = ptx::l2_policy_evict_first();
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            const Item it = item_of(p, item);
            const RowTile tl = p.tiles[it.tile];
            const int nbox = min(NT, (tl.nrows + kTokBox - 1) / kTokBox);  // host: rows <= 8·NT
            // gate/up: the nt-th 128-row blocks of W_gate and W_up; down: the
            // blocks 2nt, 2nt + 1 of W_down
            const int b0 = MODE == kGateUp ? it.nt : 2 * it.nt;
            const int b1 = MODE == kGateUp ? it.nt : 2 * it.nt + 1;
            const size_t e0 = (size_t)tl.expert * p.blocks_per_expert;
            for (int gi = it.g0; gi < it.g1; ++gi) {
                const int kb = kKbPerStage * gi;
                const uint32_t bytes = kKbPerStage * nbox * kTokBox * 128 +
                                       2 * C::kPlaneCodeBytes + 2 * kQ4ScaleBlockBytes;
                if (!ptx::mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_s, kTimeoutNs)) {
                    ok = false;
                    break;
                }
                uint8_t* st = smem + stage * C::kBytes;
                ptx::mbar_arrive_expect_tx(&full_bar[stage], bytes);
                for (int h = 0; h < kKbPerStage; ++h)
                    for (int b = 0; b < nbox; ++b)
                        ptx::tma_load_2d(st + C::kTokOff + (h * NT + b) * kTokBox * 128, &tmA,
                                         &full_bar[stage], (kb + h) * kBK, tl.row0 + b * kTokBox);
                const size_t c0 = ((e0 + b0) * p.num_kb + kb) * kQ4CodeBlockBytes;
                const size_t c1 = ((e0 + b1) * p.num_kb + kb) * kQ4CodeBlockBytes;
                const size_t s0 = ((e0 + b0) * p.groups + gi) * kQ4ScaleBlockBytes;
                const size_t s1 = ((e0 + b1) * p.groups + gi) * kQ4ScaleBlockBytes;
                // codes and scales are read once per forward: evicted first
                ptx::bulk_load_hint(st + C::kCodeOff, p.codes0 + c0, C::kPlaneCodeBytes,
                                    &full_bar[stage], pol_once);
                ptx::bulk_load_hint(st + C::kCodeOff + C::kPlaneCodeBytes, p.codes1 + c1,
                                    C::kPlaneCodeBytes, &full_bar[stage], pol_once);
                ptx::bulk_load_hint(st + C::kScaleOff, p.scales0 + s0, kQ4ScaleBlockBytes,
                                    &full_bar[stage], pol_once);
                ptx::bulk_load_hint(st + C::kScaleOff + kQ4ScaleBlockBytes, p.scales1 + s1,
                                    kQ4ScaleBlockBytes, &full_bar[stage], pol_once);
                ++issued;
                if (++stage == kS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            atomicExch(p.status, MOE_ERR_TIMEOUT);
            // Let the copies already issued land before the CTA exits.
            int dummy = 0;
            const long long first = issued > kS ? issued - kS : 0;
            for (long long n = first; n < issued; ++n)
                ptx::mbar_wait_bounded(&full_bar[n % kS], (uint32_t)((n / kS) & 1), &dummy,
                                       kTimeoutNs);
        }
        return;
    }

    // ---------------- consumers (warps 1..8) ----------------
    const int cw = warp - 1;
    const int g = lane >> 2, c = lane & 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const Item it = item_of(p, item);
        const RowTile tl = p.tiles[it.tile];
        const int nn = min(NT, (tl.nrows + kTokBox - 1) / kTokBox);
        float acc[2][NT][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.f;
        // this thread's bytes of a stage: code words 2c, 2c + 1 of row g of
        // both 16-row tiles, their rows' scale words, token g's 32 bytes from
        // column 16c (two swizzled 16-byte chunks)
        int code_off[2], scale_off[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int bi = plane_of<MODE>(cw, i), ri = row_in_block<MODE>(cw, i);
            code_off[i] = C::kCodeOff + bi * C::kPlaneCodeBytes + (ri + g) * 32 + 8 * c;
            scale_off[i] = C::kScaleOff + bi * kQ4ScaleBlockBytes + (ri + g) * 4;
        }
        const int tok0 = g * 128 + (((2 * c) ^ g) << 4);
        const int tok1 = g * 128 + (((2 * c + 1) ^ g) << 4);

        for (int gi = it.g0; gi < it.g1; ++gi) {
            int good = 1;
            if (lane == 0) good = ptx::mbar_wait_bounded(&full_bar[stage], phase, &abort_s, kTimeoutNs);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                ok = false;
                break;
            }
            const uint8_t* st = smem + stage * C::kBytes;
            if constexpr (NT == 2) {
                if (nn == 2)
                    stage_mma<NT, 2>(st, code_off, scale_off, tok0, tok1, acc);
                else
                    stage_mma<NT, 1>(st, code_off, scale_off, tok0, tok1, acc);
            } else {
                stage_mma<NT, 1>(st, code_off, scale_off, tok0, tok1, acc);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty_bar[stage]);
            if (++stage == kS) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;

        // ---------------- epilogue ----------------
        // acc[i][n][e]: tile i's row g + 8(e/2) (feature), token 8n + 2c + e%2
        if (p.ksplit == 1) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n >= nn) continue;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = 8 * n + 2 * c + (e & 1);
                    const int fr = g + 8 * (e >> 1);
                    if (tok >= tl.nrows) continue;
                    if (MODE == kGateUp) {
                        store_one<MODE>(p, tl, it.nt, tok, 0, 16 * cw + fr, acc[0][n][e],
                                        acc[1][n][e]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            store_one<MODE>(p, tl, it.nt, tok, plane_of<MODE>(cw, i),
                                            row_in_block<MODE>(cw, i) + fr, acc[i][n][e], 0.f);
                    }
                }
            }
        } else {
            // slice accumulators partial[pitem][ks][plane][part_rows][128]: this
            // warp's outputs of every slice; the last slice to arrive (per warp)
            // adds them in slice order and stores them
            const size_t plane_sz = (size_t)p.part_rows * 128;
            const size_t slice_sz = 2 * plane_sz;
            float* base = p.partial + (size_t)it.pitem * p.ksplit * slice_sz;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n >= nn) continue;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = 8 * n + 2 * c + (e & 1);
                    if (tok >= tl.nrows) continue;
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        __stcg(base + (size_t)it.ks * slice_sz + plane_of<MODE>(cw, i) * plane_sz +
                                   (size_t)tok * 128 + row_in_block<MODE>(cw, i) + g + 8 * (e >> 1),
                               acc[i][n][e]);
                }
            }
            __threadfence();
            __syncwarp();
            int32_t* cnt = p.counters + (size_t)it.pitem * kConsumers + cw;
            int last = 0;
            if (lane == 0) last = atomicAdd(cnt, 1) == p.ksplit - 1;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n >= nn) continue;
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.f;
                    for (int sl = 0; sl < p.ksplit; ++sl) {
                        const float* src = base + (size_t)sl * slice_sz;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tok = 8 * n + 2 * c + (e & 1);
                            if (tok >= tl.nrows) continue;
#pragma unroll
                            for (int i = 0; i < 2; ++i)
                                acc[i][n][e] += __ldcg(src + plane_of<MODE>(cw, i) * plane_sz +
                                                       (size_t)tok * 128 +
                                                       row_in_block<MODE>(cw, i) + g + 8 * (e >> 1));
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = 8 * n + 2 * c + (e & 1);
                        const int fr = g + 8 * (e >> 1);
                        if (tok >= tl.nrows) continue;
                        if (MODE == kGateUp) {
                            store_one<MODE>(p, tl, it.nt, tok, 0, 16 * cw + fr, acc[0][n][e],
                                            acc[1][n][e]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 2; ++i)
                                store_one<MODE>(p, tl, it.nt, tok, plane_of<MODE>(cw, i),
                                                row_in_block<MODE>(cw, i) + fr, acc[i][n][e], 0.f);
                        }
                    }
                }
                if (lane == 0) *cnt = 0;  // ready for the next forward
            }
        }
    }
    if (!ok && lane == 0) atomicExch(p.status, MOE_ERR_TIMEOUT);
}

// ---- host side ----------------------------------------------------------------

template <int MODE, int NT>
cudaError_t launch_mma(const void* A, uint64_t a_rows, uint64_t k_cols, const MmaParams& p,
                       long long max_items, cudaStream_t st) {
    CUtensorMap ma;
    if (!make_tma_2d(&ma, A, a_rows, k_cols, kTokBox)) return cudaErrorInvalidValue;
    constexpr int smem = MmaCfg<NT>::kSmemBytes;
    cudaError_t err = ensure_smem((const void*)expert_q4_mma_kernel<MODE, NT>, smem);
    if (err != cudaSuccess) return err;
    long long grid = (long long)num_sms() * MmaCfg<NT>::kCtasPerSm;
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    err = launch_pdl(expert_q4_mma_kernel<MODE, NT>, dim3((unsigned)grid), dim3(kThreadsM), smem,
                     st, ma, p);
    count_launches(1);
    return err;
}

// Token boxes per stage: a row tile holds at most min(T, kQ4MmaRows) rows (one
// row per token and expert), so one 8-row box covers T <= 8.
template <int MODE>
cudaError_t launch_mma_any(const void* A, uint64_t a_rows, uint64_t k_cols, const MmaParams& p,
                           long long max_items, int T, cudaStream_t st) {
    static_assert(kQ4MmaRows == 2 * kTokBox, "two token boxes cover a row tile");
    if (T <= kTokBox) return launch_mma<MODE, 1>(A, a_rows, k_cols, p, max_items, st);
    return launch_mma<MODE, 2>(A, a_rows, k_cols, p, max_items, st);
}

// The grid the K split is fitted to: two CTAs on each SM of a 148-SM B300 (a
// constant: the plan sizes the workspace before any device is known).
constexpr long long kMmaGrid = 2 * 148;

// Fraction of the persistent grid's rounds that n equal items keep busy.
double mma_fill(long long n) {
    const long long rounds = (n + kMmaGrid - 1) / kMmaGrid;
    return (double)n / (double)(rounds * kMmaGrid);
}

// K slices for `items` items of ngroups 128-column groups: below two rounds of
// the grid (where an unfilled last round costs the most, and the slice
// accumulators stay small), the count (at most 6, at least 4 groups a slice,
// no empty slice) whose items fill the grid's rounds best; ties go to fewer
// slices.
int mma_split(long long items, int ngroups) {
    if (items <= 0 || items >= 2 * kMmaGrid) return 1;
    int best = 1;
    double best_fill = mma_fill(items);
    for (int ks = 2; ks <= 6 && ngroups / ks >= 4; ++ks) {
        const int g_per = (ngroups + ks - 1) / ks;
        if ((ngroups + g_per - 1) / g_per != ks) continue;
        const double f = mma_fill(items * ks);
        if (f > best_fill + 0.02) {
            best = ks;
            best_fill = f;
        }
    }
    return best;
}

}  // namespace

Q4MmaPlan q4mma_plan(const Sizes& s) {
    Q4MmaPlan pl;
    if (!experts_wt_supported(s) || s.T <= 0) return pl;
    const long long P = s.P();
    // Row tiles: sum over experts of ceil(count / 16) <= P / 16 + experts touched.
    long long tiles = (s.E < P ? s.E : P) + P / kQ4MmaRows;
    if (tiles > s.max_tiles(kQ4MmaRows)) tiles = s.max_tiles(kQ4MmaRows);
    pl.items_gu = tiles * (s.I / 128);
    pl.items_dn = tiles * (s.H / 256);
    pl.ks_gu = mma_split(pl.items_gu, s.H / 128);
    pl.ks_dn = mma_split(pl.items_dn, s.I / 128);
    // A tile holds at most min(T, 16) rows.
    pl.part_rows = s.T < kQ4MmaRows ? (s.T + kTokBox - 1) / kTokBox * kTokBox : kQ4MmaRows;
    const size_t per_slice = (size_t)2 * pl.part_rows * 128;
    pl.partial_floats_gu = pl.ks_gu > 1 ? (size_t)pl.items_gu * pl.ks_gu * per_slice : 0;
    pl.partial_floats = pl.partial_floats_gu +
                        (pl.ks_dn > 1 ? (size_t)pl.items_dn * pl.ks_dn * per_slice : 0);
    pl.n_counters_gu = (int)(pl.ks_gu > 1 ? pl.items_gu * kConsumers : 0);
    pl.n_counters = pl.n_counters_gu + (int)(pl.ks_dn > 1 ? pl.items_dn * kConsumers : 0);
    return pl;
}

cudaError_t launch_experts_q4_mma(const char* q4, const Sizes& s, const Workspace& ws,
                                  cudaStream_t st, cudaEvent_t ev_mid) {
    if (!q4_supported(s.H, s.E, s.I) || !experts_wt_supported(s)) return cudaErrorInvalidValue;
    const long long P = s.P();
    const Q4MmaPlan pl = q4mma_plan(s);
    const Q4Sections q = q4_sections(q4, s.H, s.E, s.I);
    MmaParams p{};
    p.tiles = ws.tiles;
    p.n_tiles = ws.n_tiles;
    p.status = ws.status;
    p.w_perm = ws.w_perm;
    p.part_rows = pl.part_rows;

    // gate/up: tokens = x_perm rows; weights = the nt-th 128 rows of W_gate and W_up
    p.n_nt = s.I / 128;
    p.num_kb = s.H / kBK;
    p.groups = s.H / 128;
    p.ksplit = pl.ks_gu;
    p.grp_per = (p.groups + p.ksplit - 1) / p.ksplit;
    p.partial = ws.wt_partial;
    p.counters = ws.status + 4;
    p.out = ws.hbuf;
    p.out_ld = s.I;
    p.codes0 = q.codes[0];
    p.codes1 = q.codes[1];
    p.scales0 = q.scales[0];
    p.scales1 = q.scales[1];
    p.blocks_per_expert = s.I / kPackRows;
    cudaError_t err =
        launch_mma_any<kGateUp>(ws.x_perm, P, s.H, p, pl.items_gu * p.ksplit, s.T, st);
    if (err != cudaSuccess) return err;
    if (ev_mid) cudaEventRecord(ev_mid, st);

    // down: tokens = h rows; weights = W_down rows [256 nt, 256 nt + 256)
    p.n_nt = s.H / 256;
    p.num_kb = s.I / kBK;
    p.groups = s.I / 128;
    p.ksplit = pl.ks_dn;
    p.grp_per = (p.groups + p.ksplit - 1) / p.ksplit;
    p.partial = ws.wt_partial + pl.partial_floats_gu;
    p.counters = ws.status + 4 + pl.n_counters_gu;
    p.out = ws.ybuf;
    p.out_ld = s.H;
    p.codes0 = p.codes1 = q.codes[2];
    p.scales0 = p.scales1 = q.scales[2];
    p.blocks_per_expert = s.H / kPackRows;
    p.perm_tok = ws.perm_tok;
    p.perm_slot = ws.perm_slot;
    p.K = s.K;
    p.out32 = ws.ybuf_f32;
    return launch_mma_any<kDown>(ws.hbuf, P, s.I, p, pl.items_dn * p.ksplit, s.T, st);
}

}  // namespace moe
