// experts_q4.cu -- expert MLPs with 4-bit group-quantised weights,
// dequantised in shared memory, on the tensor cores.
//
// The experts' weights in the 4-bit format of the csdn page
// "MoE架构深度解析：128专家与8激活的智能路由" (section "参数量化与存储优化":
// groups of 128 parameters, a scale and a bias per group; layout and reading in
// quant.cu) computed as the bf16 experts on the dequantised weights
// w' = bf16(q·s + b): the SwiGLU expert MLP (same page, section
// "128个专家网络的组织结构与参数分布") and the routing-weight scaling
// (Qwen3MoeSparseMoeBlock.forward on the cnblogs page "大模型-qwen3 MoE 详细解读").
//
// Orientation.  A tcgen05.mma of kind::f16 takes about M cycles whatever its
// N (up to 256): one row of the output per cycle.  With the weights on the M
// side and a decode batch's few tokens on the N side (experts_wt.cu), a K=16
// step of 128 weight rows costs 128 cycles -- enough for bf16 weights, whose
// bytes arrive no faster, but a 4-bit stream delivers four times the weights
// per byte.  Here a row tile's tokens (<= 64) are the M = 64 side and 256
// weight rows the N side: 256 weight rows per 64 cycles.  Padding token rows
// cost nothing extra (the MMA time is fixed by M = 64), and rows past the
// tile's are masked in the epilogue.
//
//   gate/up item (tile, nt): D[64, 256] = X[rows] · [Wg'[e, 128 nt..+127]; Wu'[same]]ᵀ
//                            h[row, 128 nt + c] = bf16(silu(D[row, c]) · D[row, 128 + c])
//   down item (tile, nt):    D[64, 256] = h[rows] · Wd'[e, 256 nt..+255]ᵀ
//                            Y[perm_tok[row]·K + perm_slot[row], 256 nt + c] = bf16(w · D[row, c])
// with K split into slices for few items as in experts_wt.cu (the same plan:
// items, slices, slice accumulators, arrival counters); the last slice of an
// item adds the slices in slice order and runs the epilogue.
//
// Stages.  A raw stage holds the token rows of a k-block (TMA boxes of 16
// rows: the A operand, of which the M = 64 MMA reads 64 rows from the stage's
// start -- rows past the boxes loaded are other bytes of the stage and land in
// masked output rows) and, by bulk copy, the two 4 KB code blocks and two
// 512-byte scale blocks of the item's 256 weight rows; the raw stages form a
// deep ring so that enough bytes stay in flight.  Eight dequantisation warps
// turn a stage's codes into the 32 KB bf16 B operand (256 rows, 128-byte
// swizzled, K-major) in a second, double-buffered ring.  The MMA's commits free
// both stages.
//
// Roles (448 threads, one CTA per SM):
//   warp 0      producer (raw stages)
//   warp 1      TMEM owner (two 256-column accumulators) and MMA issuer
//   warps 2-5   epilogue: warp q's lanes 0-15 hold tile rows 16q..16q+15 (the
//               M = 64 accumulator puts row i in TMEM lane 32·(i/16) + i%16)
//   warps 6-13  dequantisation: thread d writes weight row d % 128 of B tile d / 128
// Every wait is bounded (2 s); on expiry the CTA records MOE_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kM = 64;      // token rows per tile (M of the MMA)
constexpr int kBN = 256;    // weight rows per item (N of the MMA): two 128-row tiles
constexpr int kBK = 64;     // k-block: 64 columns
constexpr int kBox = 16;    // token rows per TMA box
constexpr int kThreads = 448;
constexpr int kDeqWarps = 8;
constexpr int kTileBytes = 128 * kBK * 2;                 // one dequantised 128-row tile
constexpr int kBoxBytes = kBox * kBK * 2;                 // 2 KB
constexpr int kDeqStages = 2;
constexpr int kDeqBytes = kDeqStages * 2 * kTileBytes;    // the bf16 ring, first in smem
constexpr int kMaxRawStages = 14;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kM, kBN);
constexpr uint64_t kTimeoutNs = 2000000000ull;

static_assert(kWtRows == kM, "row tiles of the weights-as-M plan are the M side here");

// Raw stage: NBOX token boxes (the A operand: the MMA reads kM rows = 8 KB
// from the stage's start), then the codes and scales of the two weight tiles.
template <int NBOX>
struct RawCfg {
    static constexpr int kAOff = 0;
    static constexpr int kCodeOff = NBOX * kBoxBytes;
    static constexpr int kScaleOff = kCodeOff + 2 * kQ4CodeBlockBytes;
    static constexpr int kBytes = kScaleOff + 2 * kQ4ScaleBlockBytes;
    static constexpr int kStages = (224 * 1024 - kDeqBytes) / kBytes < kMaxRawStages
                                       ? (224 * 1024 - kDeqBytes) / kBytes
                                       : kMaxRawStages;
    static constexpr int kSmemBytes = kDeqBytes + kStages * kBytes + 1024;
    static_assert(kBytes % 1024 == 0, "raw stages stay 1024-byte aligned");
    static_assert(kBytes >= kM * kBK * 2, "the MMA's 64 A rows lie inside the stage");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

enum { kGateUp = 0, kDown = 1 };

struct Q4Params {
    const RowTile* tiles;
    const int32_t* n_tiles;
    int n_nt;               // 256-row weight blocks per row tile
    int num_kb;             // k-blocks of 64
    int ksplit;
    int kb_per;
    float* partial;         // [items][ksplit][part_rows][256] slice accumulators
    int part_rows;
    int32_t* counters;      // [items][4]
    __nv_bfloat16* out;     // h [P, I] or Y [P, H]
    int out_ld;
    const float* w_perm;
    int32_t* status;
    // codes / scales of the two 128-row weight tiles of an item and the
    // 128-row blocks per expert of their matrix
    const char* codes0;
    const char* codes1;
    const char* scales0;
    const char* scales1;
    int a_blocks_per_expert;
    int groups;             // 128-column groups per weight row (num_kb / 2)
    const int32_t* perm_tok;
    const int32_t* perm_slot;
    int K;
    float* out32;           // down: fp32 Y [P, H] (under a capacity); null: bf16 Y in out
};

// Item -> row tile, 256-row weight block, K slice and its k-block range.
struct Item {
    int pitem, tile, nt, ks, kb0, kb1;
};

__device__ __forceinline__ Item item_of(const Q4Params& p, int item) {
    Item it;
    it.pitem = item / p.ksplit;
    it.ks = item % p.ksplit;
    it.tile = it.pitem / p.n_nt;
    it.nt = it.pitem % p.n_nt;
    it.kb0 = it.ks * p.kb_per;
    it.kb1 = min(p.num_kb, it.kb0 + p.kb_per);
    return it;
}

__device__ __forceinline__ void store8(__nv_bfloat16* dst, const float (&v)[8]) {
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = o;
}

// Epilogue of 32 columns [c0, c0 + 32) of one row from fp32 accumulators:
// gate/up (a = gate columns c0.., b = up columns 128 + c0..) writes h; down
// (a = columns c0..) writes Y.
template <int MODE>
__device__ __forceinline__ void store_cols(const Q4Params& p, size_t row, int nt, int c0,
                                           const float (&a)[32], const float (&b)[32]) {
    if (MODE == kGateUp) {
        __nv_bfloat16* dst = p.out + row * p.out_ld + (size_t)nt * 128 + c0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = silu_f(a[8 * j + i]) * b[8 * j + i];
            store8(dst + 8 * j, v);
        }
    } else {
        const float wr = p.w_perm[row];
        const size_t yrow = (size_t)p.perm_tok[row] * p.K + (size_t)p.perm_slot[row];
        if (p.out32) {
            float4* dst = reinterpret_cast<float4*>(p.out32 + yrow * p.out_ld +
                                                    (size_t)nt * kBN + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(wr * a[4 * j], wr * a[4 * j + 1], wr * a[4 * j + 2],
                                     wr * a[4 * j + 3]);
            return;
        }
        __nv_bfloat16* dst = p.out + yrow * p.out_ld + (size_t)nt * kBN + c0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = wr * a[8 * j + i];
            store8(dst + 8 * j, v);
        }
    }
}

template <int MODE, int NBOX>
__global__ void __launch_bounds__(kThreads, 1)
    expert_q4_kernel(const __grid_constant__ CUtensorMap tmA, const Q4Params p) {
    using R = RawCfg<NBOX>;
    constexpr int kRS = R::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* const deq_base = smem;              // kDeqStages x 256 bf16 weight rows
    uint8_t* const raw_base = smem + kDeqBytes;  // kRS raw stages
    __shared__ __align__(8) uint64_t raw_full[kMaxRawStages];   // boxes, codes, scales landed
    __shared__ __align__(8) uint64_t raw_empty[kMaxRawStages];  // the stage's MMAs are done
    __shared__ __align__(8) uint64_t deq_full[kDeqStages];      // bf16 weights written
    __shared__ __align__(8) uint64_t deq_empty[kDeqStages];     // their MMAs are done
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRS; ++s) {
            ptx::mbar_init(&raw_full[s], 1);
            ptx::mbar_init(&raw_empty[s], 1);
        }
        for (int s = 0; s < kDeqStages; ++s) {
            ptx::mbar_init(&deq_full[s], kDeqWarps);
            ptx::mbar_init(&deq_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull_bar[b], 1);
            ptx::mbar_init(&tempty_bar[b], 4);
        }
        ptx::mbar_init(&drain_bar, 1);
        abort_s = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&tmem_base_s, kTmemCols);
        ptx::tmem_relinquish();
    }
    pdl_trigger();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    pdl_wait();  // the prologue above overlaps the previous kernel's tail
    const int total = (*p.n_tiles) * p.n_nt * p.ksplit;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: raw stages ----------------
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const Item it = item_of(p, item);
                const RowTile tl = p.tiles[it.tile];
                const int nbox = (tl.nrows + kBox - 1) / kBox;  // <= NBOX (host-checked)
                // the item's 256 weight rows: gate/up = 128 gate rows over the
                // same 128 up rows; down = two 128-row blocks of W_down
                const int b0 = MODE == kGateUp ? it.nt : 2 * it.nt;
                const int b1 = MODE == kGateUp ? it.nt : 2 * it.nt + 1;
                const size_t e0 = (size_t)tl.expert * p.a_blocks_per_expert;
                const uint32_t bytes =
                    nbox * kBoxBytes + 2 * kQ4CodeBlockBytes + 2 * kQ4ScaleBlockBytes;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&raw_empty[stage], phase ^ 1u, &abort_s,
                                                kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sr = raw_base + stage * R::kBytes;
                    ptx::mbar_arrive_expect_tx(&raw_full[stage], bytes);
                    for (int b = 0; b < nbox; ++b)
                        ptx::tma_load_2d(sr + R::kAOff + b * kBoxBytes, &tmA, &raw_full[stage],
                                         kb * kBK, tl.row0 + b * kBox);
                    const size_t c0 = ((e0 + b0) * p.num_kb + kb) * kQ4CodeBlockBytes;
                    const size_t c1 = ((e0 + b1) * p.num_kb + kb) * kQ4CodeBlockBytes;
                    const size_t s0 = ((e0 + b0) * p.groups + kb / 2) * kQ4ScaleBlockBytes;
                    const size_t s1 = ((e0 + b1) * p.groups + kb / 2) * kQ4ScaleBlockBytes;
                    ptx::bulk_load(sr + R::kCodeOff, p.codes0 + c0, kQ4CodeBlockBytes,
                                   &raw_full[stage]);
                    ptx::bulk_load(sr + R::kCodeOff + kQ4CodeBlockBytes, p.codes1 + c1,
                                   kQ4CodeBlockBytes, &raw_full[stage]);
                    ptx::bulk_load(sr + R::kScaleOff, p.scales0 + s0, kQ4ScaleBlockBytes,
                                   &raw_full[stage]);
                    ptx::bulk_load(sr + R::kScaleOff + kQ4ScaleBlockBytes, p.scales1 + s1,
                                   kQ4ScaleBlockBytes, &raw_full[stage]);
                    ++issued;
                    if (++stage == kRS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicExch(p.status, MOE_ERR_TIMEOUT);
                // Let the copies already issued land before the CTA exits.
                int dummy = 0;
                const long long first = issued > kRS ? issued - kRS : 0;
                for (long long n = first; n < issued; ++n)
                    ptx::mbar_wait_bounded(&raw_full[n % kRS], (uint32_t)((n / kRS) & 1), &dummy,
                                           kTimeoutNs);
            }
        }
    } else if (warp >= 6) {
        // ---------------- dequantisation (warps 6..13) ----------------
        // Thread d writes weight row r = d % 128 of B tile t = d / 128: its 8
        // code words and scale word from the raw stage, 8 swizzled 16-byte
        // chunks (row r at r*128 bytes, chunk c at ((c ^ r % 8) * 16)).
        const int d = threadIdx.x - 6 * 32;
        const int t = d >> 7, r = d & 127;
        int rs = 0, ds = 0;
        uint32_t rph = 0, dph = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            const Item it = item_of(p, item);
            for (int kb = it.kb0; kb < it.kb1; ++kb) {
                int good = 1;
                if (lane == 0)
                    good = ptx::mbar_wait_bounded(&raw_full[rs], rph, &abort_s, kTimeoutNs) &&
                           ptx::mbar_wait_bounded(&deq_empty[ds], dph ^ 1u, &abort_s, kTimeoutNs);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    ok = false;
                    break;
                }
                const uint8_t* sr = raw_base + rs * R::kBytes;
                const uint4* cw = reinterpret_cast<const uint4*>(
                    sr + R::kCodeOff + t * kQ4CodeBlockBytes + r * 32);
                const uint4 w0 = cw[0], w1 = cw[1];
                const uint32_t sbw = *reinterpret_cast<const uint32_t*>(
                    sr + R::kScaleOff + t * kQ4ScaleBlockBytes + r * 4);
                const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint8_t* row = deq_base + ds * (2 * kTileBytes) + t * kTileBytes + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                        q4_dequant8(words[c], sbw);
                ptx::fence_proxy_async_shared();  // the MMA reads the tile (async proxy)
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&deq_full[ds]);
                if (++rs == kRS) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (++ds == kDeqStages) {
                    ds = 0;
                    dph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) atomicExch(p.status, MOE_ERR_TIMEOUT);
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int rs = 0, ds = 0;
            uint32_t rph = 0, dph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const Item it = item_of(p, item);
                if (!ptx::mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, &abort_s,
                                            kTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t dacc = tmem_base + (uint32_t)(acc * kBN);
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&raw_full[rs], rph, &abort_s, kTimeoutNs) ||
                        !ptx::mbar_wait_bounded(&deq_full[ds], dph, &abort_s, kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t adesc = ptx::desc_sw128_kmajor(
                        ptx::smem_u32(raw_base + rs * R::kBytes + R::kAOff));
                    const uint64_t bdesc =
                        ptx::desc_sw128_kmajor(ptx::smem_u32(deq_base + ds * (2 * kTileBytes)));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)  // K = 16 per MMA: +32 bytes
                        ptx::mma_bf16(dacc, adesc + 2u * k, bdesc + 2u * k, kIdesc,
                                      (kb != it.kb0 || k != 0) ? 1u : 0u);
                    ptx::mma_commit(&raw_empty[rs]);
                    ptx::mma_commit(&deq_empty[ds]);
                    if (++rs == kRS) {
                        rs = 0;
                        rph ^= 1u;
                    }
                    if (++ds == kDeqStages) {
                        ds = 0;
                        dph ^= 1u;
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
    } else if (warp >= 2) {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;         // TMEM lane quadrant of this warp
        const int r = q * 16 + lane;    // tile row of lanes 0..15 (M = 64 layout)
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            const Item it = item_of(p, item);
            const RowTile tl = p.tiles[it.tile];
            int ok = 1;
            if (lane == 0)
                ok = ptx::mbar_wait_bounded(&tfull_bar[acc], acc_phase, &abort_s, kTimeoutNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) atomicExch(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const bool valid = lane < 16 && r < tl.nrows;
            const size_t row = (size_t)tl.row0 + r;
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
            if (p.ksplit == 1) {
#pragma unroll 1
                for (int c0 = 0; c0 < (MODE == kGateUp ? 128 : kBN); c0 += 32) {
                    uint32_t va[32], vb[32];
                    ptx::tmem_ld32(tb + c0, va);
                    if (MODE == kGateUp) ptx::tmem_ld32(tb + 128 + c0, vb);
                    ptx::tmem_ld_wait();
                    if (valid) {
                        float a[32], b[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            a[j] = __uint_as_float(va[j]);
                            b[j] = MODE == kGateUp ? __uint_as_float(vb[j]) : 0.f;
                        }
                        store_cols<MODE>(p, row, it.nt, c0, a, b);
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
            } else {
                // This slice's accumulators -> partial[pitem][ks][row][256], then
                // free TMEM; the last slice of the item (per warp quadrant) adds
                // all slices in slice order and runs the epilogue.
                const size_t slice = (size_t)p.part_rows * kBN;
                float* mine = p.partial + ((size_t)it.pitem * p.ksplit + it.ks) * slice +
                              (size_t)r * kBN;
#pragma unroll 1
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tb + c0, v);
                    ptx::tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            __stcg(reinterpret_cast<float4*>(mine + c0 + j),
                                   make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                               __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])));
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
                __threadfence();
                __syncwarp();
                int32_t* cnt = p.counters + it.pitem * 4 + q;
                int last = 0;
                if (lane == 0) last = atomicAdd(cnt, 1) == p.ksplit - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    const float* all = p.partial + (size_t)it.pitem * p.ksplit * slice +
                                       (size_t)r * kBN;
                    if (valid) {
#pragma unroll 1
                        for (int c0 = 0; c0 < (MODE == kGateUp ? 128 : kBN); c0 += 32) {
                            float a[32], b[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                a[j] = 0.f;
                                b[j] = 0.f;
                            }
                            for (int sl = 0; sl < p.ksplit; ++sl) {
                                const float* src = all + (size_t)sl * slice;
#pragma unroll
                                for (int j = 0; j < 32; j += 4) {
                                    const float4 x = __ldcg(reinterpret_cast<const float4*>(src + c0 + j));
                                    a[j] += x.x;
                                    a[j + 1] += x.y;
                                    a[j + 2] += x.z;
                                    a[j + 3] += x.w;
                                    if (MODE == kGateUp) {
                                        const float4 y = __ldcg(
                                            reinterpret_cast<const float4*>(src + 128 + c0 + j));
                                        b[j] += y.x;
                                        b[j + 1] += y.y;
                                        b[j + 2] += y.z;
                                        b[j + 3] += y.w;
                                    }
                                }
                            }
                            store_cols<MODE>(p, row, it.nt, c0, a, b);
                        }
                    }
                    if (lane == 0) *cnt = 0;  // ready for the next forward
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

// ---- host side ----------------------------------------------------------------

template <int MODE, int NBOX>
cudaError_t launch_q4(const void* A, uint64_t a_rows, uint64_t k_cols, const Q4Params& p,
                      long long max_items, cudaStream_t st) {
    CUtensorMap ma;
    if (!make_tma_2d(&ma, A, a_rows, k_cols, kBox)) return cudaErrorInvalidValue;
    constexpr int smem = RawCfg<NBOX>::kSmemBytes;
    cudaError_t err = ensure_smem((const void*)expert_q4_kernel<MODE, NBOX>, smem);
    if (err != cudaSuccess) return err;
    long long grid = num_sms();
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    err = launch_pdl(expert_q4_kernel<MODE, NBOX>, dim3((unsigned)grid), dim3(kThreads), smem, st,
                     ma, p);
    count_launches(1);
    return err;
}

// One token box per raw stage while a row tile holds at most 16 rows: an
// expert receives at most one row per token, so T <= 16 guarantees it.
template <int MODE>
cudaError_t launch_q4_any(const void* A, uint64_t a_rows, uint64_t k_cols, const Q4Params& p,
                          long long max_items, int T, cudaStream_t st) {
    if (T <= kBox) return launch_q4<MODE, 1>(A, a_rows, k_cols, p, max_items, st);
    return launch_q4<MODE, kM / kBox>(A, a_rows, k_cols, p, max_items, st);
}

}  // namespace

cudaError_t launch_experts_q4(const char* q4, const Sizes& s, const Workspace& ws,
                              cudaStream_t st, cudaEvent_t ev_mid) {
    if (!q4_supported(s.H, s.E, s.I) || !experts_wt_supported(s)) return cudaErrorInvalidValue;
    const long long P = s.P();
    // the items, K slices, slice accumulators and counters of the weights-as-M
    // plan: the same item counts (row tiles x I/128, row tiles x H/256) and slice sizes
    const WtPlan pl = wt_plan(s);
    const Q4Sections q = q4_sections(q4, s.H, s.E, s.I);
    Q4Params p{};
    p.tiles = ws.tiles;
    p.n_tiles = ws.n_tiles;
    p.status = ws.status;
    p.w_perm = ws.w_perm;
    p.part_rows = pl.part_rows;

    // gate/up: A = x_perm rows; B = 128 W_gate rows over the same 128 W_up rows
    p.n_nt = s.I / 128;
    p.num_kb = s.H / kBK;
    p.groups = s.H / 128;
    p.ksplit = pl.ks_gu;
    p.kb_per = (p.num_kb + p.ksplit - 1) / p.ksplit;
    p.partial = ws.wt_partial;
    p.counters = ws.status + 4;
    p.out = ws.hbuf;
    p.out_ld = s.I;
    p.codes0 = q.codes[0];
    p.codes1 = q.codes[1];
    p.scales0 = q.scales[0];
    p.scales1 = q.scales[1];
    p.a_blocks_per_expert = s.I / kPackRows;
    cudaError_t err =
        launch_q4_any<kGateUp>(ws.x_perm, P, s.H, p, pl.items_gu * p.ksplit, s.T, st);
    if (err != cudaSuccess) return err;
    if (ev_mid) cudaEventRecord(ev_mid, st);

    // down: A = h rows; B = W_down rows [256 nt, 256 nt + 256)
    p.n_nt = s.H / kBN;
    p.num_kb = s.I / kBK;
    p.groups = s.I / 128;
    p.ksplit = pl.ks_dn;
    p.kb_per = (p.num_kb + p.ksplit - 1) / p.ksplit;
    p.partial = ws.wt_partial + pl.partial_floats_gu;
    p.counters = ws.status + 4 + pl.n_counters_gu;
    p.out = ws.ybuf;
    p.out_ld = s.H;
    p.codes0 = p.codes1 = q.codes[2];
    p.scales0 = p.scales1 = q.scales[2];
    p.a_blocks_per_expert = s.H / kPackRows;
    p.perm_tok = ws.perm_tok;
    p.perm_slot = ws.perm_slot;
    p.K = s.K;
    p.out32 = ws.ybuf_f32;
    return launch_q4_any<kDown>(ws.hbuf, P, s.I, p, pl.items_dn * p.ksplit, s.T, st);
}

}  // namespace moe
