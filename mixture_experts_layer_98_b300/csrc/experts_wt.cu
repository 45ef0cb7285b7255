// experts_wt.cu -- expert MLPs of small batches on the tensor cores, with the
// expert weights on the MMA's M side.
//
// The expert is the SwiGLU MLP down(silu(gate(x)) ⊙ up(x)) with per-expert
// gate_proj / up_proj [I,H] and down_proj [H,I] (csdn page
// "MoE架构深度解析：128专家与8激活的智能路由", section
// "128个专家网络的组织结构与参数分布"), scaled by the pair's routing weight
// (Qwen3MoeSparseMoeBlock.forward on the cnblogs page "大模型-qwen3 MoE 详细解读").
//
// In decode-sized batches an expert sees a handful of rows, so the work is
// bound by streaming the touched experts' weights from HBM once.  Putting the
// rows on the 128-wide M side of the MMA would pad each expert to 128 rows and
// make a third of every stage's bytes padding; here the product is computed
// transposed instead: 128 weight rows form the M side (they are K-major in
// HBM, as an A operand wants) and the tile's <= 64 token rows the N side
// (N = 16, 32, 48 or 64), so nearly every byte a stage moves is weights.
//
//   gate/up : Dg[i, j] = Wg[e, i0 + i] · x_perm[row0 + j]
//             Du[i, j] = Wu[e, i0 + i] · x_perm[row0 + j]
//             h[row0 + j, i0 + i] = bf16(silu(Dg) · Du)
//   down    : D0[i, j] = Wd[e, n0 + i] · h[row0 + j],  D1 likewise for n0 + 128 + i
//             Y[t*K + k, n0 + i] = bf16(w[row0 + j] · D) for the pair (t, k) of
//             dispatch row row0 + j (token-major Y)
//
// One work item is (row tile, block of weight rows): 128 gate rows with the
// same 128 up rows, or 256 down rows.  When a batch has fewer items than
// about one per SM (a single decode token touches 8 experts: 96 gate/up
// items), each item is split along K into ksplit slices so that every SM
// streams weights: a slice stores its fp32 accumulators, and the last slice
// to finish (per-item arrival counter) adds all slices in slice order and runs
// the epilogue, so the result does not depend on which slice finishes last.
// The counters are zeroed by the router kernel at the start of each forward
// and reset by their last arriver.  Persistent, warp-specialised CTA (one per
// SM, 192 threads):
//   warp 0     TMA producer: two 128x64 weight tiles and ceil(rows/16) 16x64
//              token boxes per k-block into a 5-stage ring (128-byte swizzle)
//   warp 1     owns TMEM (two buffers x two accumulators x 64 columns) and
//              issues tcgen05.mma M=128 N=16·boxes K=16 (8 per k-block)
//   warps 2-5  epilogue: warp w reads TMEM lanes 32·(w%4)..+31 (weight rows)
//              16 token columns at a time and stores the tile's valid rows
// Every wait is bounded (2 s); on expiry the CTA records MOE_ERR_TIMEOUT in the
// workspace status word, drains its in-flight copies and MMAs, frees TMEM and
// exits.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kWM = 128;      // weight rows per MMA (M)
constexpr int kBK = 64;       // 64 bf16 = 128 bytes: one swizzle row
constexpr int kBox = 16;      // token rows per TMA box
constexpr int kStages = 5;
constexpr int kThreads = 192;
constexpr int kABytes = kWM * kBK * 2;                         // 16 KB
constexpr int kBoxBytes = kBox * kBK * 2;                      // 2 KB
constexpr int kStageBytes = 2 * kABytes + (kWtRows / kBox) * kBoxBytes;  // 40 KB
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr uint32_t kAccCols = kWtRows;       // columns of one accumulator
constexpr uint32_t kTmemCols = 4 * kAccCols;  // 2 buffers x 2 accumulators
constexpr uint64_t kTimeoutNs = 2000000000ull;

static_assert(kWtRows % kBox == 0 && kWtRows <= 64, "token tile must be <= 64 rows");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

enum { kGateUp = 0, kDown = 1 };

struct WtParams {
    const RowTile* tiles;
    const int32_t* n_tiles;
    int n_blk;              // weight-row blocks per row tile
    int num_kb;             // k-blocks of 64
    int ksplit;             // K slices per item (1: no split)
    int kb_per;             // k-blocks per slice
    float* partial;         // [items][ksplit][2][part_rows][128] slice accumulators
    int part_rows;
    int32_t* counters;      // [items][4]: slices finished, per epilogue warp
    int w_rows_per_expert;  // I (gate/up) or H (down)
    __nv_bfloat16* out;     // h [P, I] or Y [P, H]
    int out_ld;
    const float* w_perm;    // routing weight per row (down)
    int32_t* status;
    // Packed weights (null: row-major through the A tensor maps): block bases of
    // A0 and A1 and 128-row blocks per expert of the weight matrix.
    const char* apk0;
    const char* apk1;
    int a_blocks_per_expert;
    // down: Y is stored token-major, row perm_tok[r] * K + perm_slot[r]
    const int32_t* perm_tok;
    const int32_t* perm_slot;
    int K;
    float* out32;           // down: fp32 Y [P, H] (under a capacity); null: bf16 Y in out
};

// Epilogue of one output row and weight row i of the block: gate/up writes
// h = silu(D0)·D1; down writes Y = w·D0 and Y = w·D1 for the two 128-row halves.
template <int MODE>
__device__ __forceinline__ void store_out(const WtParams& p, size_t row, int blk, int i, float d0,
                                          float d1) {
    if (MODE == kGateUp) {
        p.out[row * p.out_ld + (size_t)blk * kWM + i] = __float2bfloat16_rn(silu_f(d0) * d1);
    } else {
        const float wr = p.w_perm[row];
        const size_t yrow = (size_t)p.perm_tok[row] * p.K + (size_t)p.perm_slot[row];
        if (p.out32) {
            float* o = p.out32 + yrow * p.out_ld + (size_t)blk * (2 * kWM);
            o[i] = wr * d0;
            o[kWM + i] = wr * d1;
        } else {
            __nv_bfloat16* o = p.out + yrow * p.out_ld + (size_t)blk * (2 * kWM);
            o[i] = __float2bfloat16_rn(wr * d0);
            o[kWM + i] = __float2bfloat16_rn(wr * d1);
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    expert_wt_tc_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB, const WtParams p) {
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
        ptx::prefetch_tmap(&tmA0);
        ptx::prefetch_tmap(&tmA1);
        ptx::prefetch_tmap(&tmB);
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
    const int total = (*p.n_tiles) * p.n_blk * p.ksplit;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            const uint64_t pol_once = ptx::l2_policy_evict_first();
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const int pitem = item / p.ksplit, ks = item % p.ksplit;
                const RowTile tl = p.tiles[pitem / p.n_blk];
                const int blk = pitem % p.n_blk;
                const int kb0 = ks * p.kb_per, kb1 = min(p.num_kb, kb0 + p.kb_per);
                const int nbox = (tl.nrows + kBox - 1) / kBox;
                int a0, a1;    // weight rows in the row-major matrices
                int a0b, a1b;  // the same as 128-row blocks within the expert (packed)
                if (MODE == kGateUp) {
                    a0 = a1 = tl.expert * p.w_rows_per_expert + blk * kWM;
                    a0b = a1b = blk;
                } else {
                    a0 = tl.expert * p.w_rows_per_expert + blk * (2 * kWM);
                    a1 = a0 + kWM;
                    a0b = 2 * blk;
                    a1b = 2 * blk + 1;
                }
                const uint32_t bytes = 2 * kABytes + nbox * kBoxBytes;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_s,
                                                kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + stage * kStageBytes;
                    uint8_t* sB = sA + 2 * kABytes;
                    ptx::mbar_arrive_expect_tx(&full_bar[stage], bytes);
                    if (p.apk0) {  // packed: each weight tile is one contiguous 16 KB block
                        // (read once per forward: evicted first, ahead of the
                        // activations and h the forward reads back)
                        const size_t e0 = (size_t)tl.expert * p.a_blocks_per_expert;
                        ptx::bulk_load_hint(
                            sA, p.apk0 + ((e0 + a0b) * p.num_kb + kb) * kPackBlockBytes, kABytes,
                            &full_bar[stage], pol_once);
                        ptx::bulk_load_hint(
                            sA + kABytes, p.apk1 + ((e0 + a1b) * p.num_kb + kb) * kPackBlockBytes,
                            kABytes, &full_bar[stage], pol_once);
                    } else {
                        ptx::tma_load_2d(sA, &tmA0, &full_bar[stage], kb * kBK, a0);
                        ptx::tma_load_2d(sA + kABytes, &tmA1, &full_bar[stage], kb * kBK, a1);
                    }
                    for (int b = 0; b < nbox; ++b)
                        ptx::tma_load_2d(sB + b * kBoxBytes, &tmB, &full_bar[stage], kb * kBK,
                                         tl.row0 + b * kBox);
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
                const int pitem = item / p.ksplit, ks = item % p.ksplit;
                const int kb0 = ks * p.kb_per, kb1 = min(p.num_kb, kb0 + p.kb_per);
                const int nrows = p.tiles[pitem / p.n_blk].nrows;
                const int n = ((nrows + kBox - 1) / kBox) * kBox;
                const uint32_t idesc = ptx::idesc_bf16_f32(kWM, n);
                if (!ptx::mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, &abort_s,
                                            kTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)acc * (2 * kAccCols);
                const uint32_t d1 = d0 + kAccCols;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&full_bar[stage], phase, &abort_s, kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint64_t adesc0 = ptx::desc_sw128_kmajor(a_addr);
                    const uint64_t adesc1 = ptx::desc_sw128_kmajor(a_addr + kABytes);
                    const uint64_t bdesc = ptx::desc_sw128_kmajor(a_addr + 2 * kABytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {  // K = 16 per MMA: +32 bytes
                        const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
                        ptx::mma_bf16(d0, adesc0 + 2u * k, bdesc + 2u * k, idesc, accum);
                        ptx::mma_bf16(d1, adesc1 + 2u * k, bdesc + 2u * k, idesc, accum);
                    }
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
        const int i = q * 32 + lane;  // weight row within the 128-row block
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            const int pitem = item / p.ksplit, ks = item % p.ksplit;
            const RowTile tl = p.tiles[pitem / p.n_blk];
            const int blk = pitem % p.n_blk;
            int ok = 1;
            if (lane == 0)
                ok = ptx::mbar_wait_bounded(&tfull_bar[acc], acc_phase, &abort_s, kTimeoutNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) atomicExch(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16) +
                                (uint32_t)acc * (2 * kAccCols);
            const uint32_t t1 = t0 + kAccCols;
            const int n = ((tl.nrows + kBox - 1) / kBox) * kBox;
            if (p.ksplit == 1) {
#pragma unroll 1
                for (int c = 0; c < n; c += kBox) {
                    uint32_t v0[kBox], v1[kBox];
                    ptx::tmem_ld16(t0 + c, v0);
                    ptx::tmem_ld16(t1 + c, v1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < kBox; ++j)
                        if (c + j < tl.nrows)
                            store_out<MODE>(p, (size_t)tl.row0 + c + j, blk, i,
                                            __uint_as_float(v0[j]), __uint_as_float(v1[j]));
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
            } else {
                // This slice's accumulators -> partial[pitem][ks] (rows j, column i:
                // each warp store is 128 contiguous bytes), then free TMEM.
                const size_t slice = (size_t)2 * p.part_rows * kWM;
                float* mine = p.partial + ((size_t)pitem * p.ksplit + ks) * slice;
#pragma unroll 1
                for (int c = 0; c < n; c += kBox) {
                    uint32_t v0[kBox], v1[kBox];
                    ptx::tmem_ld16(t0 + c, v0);
                    ptx::tmem_ld16(t1 + c, v1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < kBox; ++j)
                        if (c + j < tl.nrows) {
                            __stcg(mine + (size_t)(c + j) * kWM + i, __uint_as_float(v0[j]));
                            __stcg(mine + ((size_t)p.part_rows + c + j) * kWM + i,
                                   __uint_as_float(v1[j]));
                        }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
                // Publish, count; the last slice of this item (per warp
                // quadrant) adds all slices in slice order.
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(&p.counters[pitem * 4 + q], 1) == p.ksplit - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    const float* all = p.partial + (size_t)pitem * p.ksplit * slice;
#pragma unroll 1
                    for (int j = 0; j < tl.nrows; ++j) {
                        float a0 = 0.f, a1 = 0.f;
                        for (int sl = 0; sl < p.ksplit; ++sl) {
                            const float* src = all + (size_t)sl * slice;
                            a0 += __ldcg(src + (size_t)j * kWM + i);
                            a1 += __ldcg(src + ((size_t)p.part_rows + j) * kWM + i);
                        }
                        store_out<MODE>(p, (size_t)tl.row0 + j, blk, i, a0, a1);
                    }
                    if (lane == 0) p.counters[pitem * 4 + q] = 0;  // ready for the next forward
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

template <int MODE>
cudaError_t launch_wt(const void* A0, const void* A1, uint64_t a_rows, uint64_t k_cols,
                      const void* B, uint64_t b_rows, const WtParams& p, long long max_items,
                      cudaStream_t st) {
    CUtensorMap ma0, ma1, mb;
    if (!make_tma_2d(&mb, B, b_rows, k_cols, kBox)) return cudaErrorInvalidValue;
    if (p.apk0) {  // packed weights: the A maps are not used
        ma0 = mb;
        ma1 = mb;
    } else if (!make_tma_2d(&ma0, A0, a_rows, k_cols, kWM) ||
               !make_tma_2d(&ma1, A1, a_rows, k_cols, kWM)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = ensure_smem((const void*)expert_wt_tc_kernel<MODE>, kSmemBytes);
    if (err != cudaSuccess) return err;
    long long grid = num_sms();
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    err = launch_pdl(expert_wt_tc_kernel<MODE>, dim3((unsigned)grid), dim3(kThreads), kSmemBytes,
                     st, ma0, ma1, mb, p);
    count_launches(1);
    return err;
}

}  // namespace

bool experts_wt_supported(const Sizes& s) { return s.I % kWM == 0 && s.H % (2 * kWM) == 0; }

namespace {

// Items below which the K split starts, and the grid the split is fitted to:
// one CTA per SM of a 148-SM B300.  The plan must depend on the sizes only
// (the workspace is sized from it before any device is known), so this is a
// constant rather than the device's count.
constexpr long long kSplitBelow = 148;

// Fraction of the last round of a persistent grid of kSplitBelow CTAs that
// n equal work items keep busy, over all rounds (1 = no idle tail).
double round_fill(long long n) {
    const long long rounds = (n + kSplitBelow - 1) / kSplitBelow;
    return (double)n / (double)(rounds * kSplitBelow);
}

// K slices for `items` items of num_kb k-blocks: the slice count (at most 8,
// at least 8 k-blocks per slice -- shorter slices measured slower, the
// per-item epilogue and hand-off then dominate -- and no empty slice) whose
// items fill the rounds of the persistent grid best; ties go to fewer slices.
int split_for(long long items, int num_kb) {
    if (items <= 0 || items >= kSplitBelow) return 1;
    int best = 1;
    double best_fill = round_fill(items);
    for (int ks = 2; ks <= 8 && num_kb / ks >= 8; ++ks) {
        const int kb_per = (num_kb + ks - 1) / ks;
        if ((num_kb + kb_per - 1) / kb_per != ks) continue;  // would leave a slice empty
        const double f = round_fill(items * ks);
        if (f > best_fill + 0.02) {
            best = ks;
            best_fill = f;
        }
    }
    return best;
}

}  // namespace

WtPlan wt_plan(const Sizes& s) {
    WtPlan pl;
    if (!experts_wt_supported(s) || s.T <= 0) return pl;
    const long long P = s.P();
    // Row tiles: sum over experts of ceil(count / kWtRows) <= P / kWtRows + experts touched.
    long long tiles = (s.E < P ? s.E : P) + P / kWtRows;
    if (tiles > s.max_tiles(kWtRows)) tiles = s.max_tiles(kWtRows);
    pl.items_gu = tiles * (s.I / kWM);
    pl.items_dn = tiles * (s.H / (2 * kWM));
    pl.ks_gu = split_for(pl.items_gu, s.H / kBK);
    pl.ks_dn = split_for(pl.items_dn, s.I / kBK);
    if (s.T <= kDecodeAutoTokens) {
        // The fused decode kernel runs both GEMMs in one grid and a down unit
        // waits for its tile's gate/up units, so there round fill is not the
        // whole story: measured (graph replay, the fused kernel), two slices
        // of gate/up while its items are under four rounds (four tokens:
        // 193.5 -> 187.3 us) and of down while its items are under one round
        // (one token: 80.8 -> 76.4 us) are faster; more slices, or down slices
        // with a round of items or more, measured slower.
        if (pl.items_gu < 4 * kSplitBelow && pl.ks_gu < 2 && s.H / kBK >= 16) pl.ks_gu = 2;
        if (pl.items_dn < kSplitBelow && pl.ks_dn < 2 && s.I / kBK >= 16) pl.ks_dn = 2;
    }
    // A tile holds at most one row per token, so at most min(kWtRows, T) rows.
    pl.part_rows = s.T < kWtRows ? ((s.T + kBox - 1) / kBox) * kBox : kWtRows;
    // Separate gate/up and down regions: the fused decode kernel runs units of
    // both kinds at once.
    const size_t per_slice = (size_t)2 * pl.part_rows * kWM;
    pl.partial_floats_gu = pl.ks_gu > 1 ? (size_t)pl.items_gu * pl.ks_gu * per_slice : 0;
    pl.partial_floats = pl.partial_floats_gu +
                        (pl.ks_dn > 1 ? (size_t)pl.items_dn * pl.ks_dn * per_slice : 0);
    pl.n_counters_gu = (int)(pl.ks_gu > 1 ? pl.items_gu : 0) * 4;
    pl.n_counters_dn = (int)(pl.ks_dn > 1 ? pl.items_dn : 0) * 4;
    if (s.T <= kDecodeFusedTokens) {
        pl.n_ready = (int)tiles;
        pl.n_cdone = s.T * (s.H / (2 * kWM) * 4);
    }
    pl.n_counters = pl.n_counters_gu + pl.n_counters_dn + pl.n_ready + pl.n_cdone;
    return pl;
}

cudaError_t launch_experts_wt(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                              cudaStream_t st, cudaEvent_t ev_mid) {
    if (!experts_wt_supported(s)) return cudaErrorInvalidValue;
    const bool packed = W.packed != nullptr;
    const long long P = s.P();
    const WtPlan pl = wt_plan(s);
    WtParams p{};
    p.tiles = ws.tiles;
    p.n_tiles = ws.n_tiles;
    p.status = ws.status;
    p.w_perm = ws.w_perm;
    p.partial = ws.wt_partial;
    p.part_rows = pl.part_rows;

    // gate/up: A0 = 128 W_gate rows, A1 = the same 128 W_up rows; B = x_perm rows
    p.n_blk = s.I / kWM;
    p.num_kb = s.H / kBK;
    p.ksplit = pl.ks_gu;
    p.kb_per = (p.num_kb + p.ksplit - 1) / p.ksplit;
    p.counters = ws.status + 4;
    p.w_rows_per_expert = s.I;
    p.out = ws.hbuf;
    p.out_ld = s.I;
    p.apk0 = packed ? W.packed_gate(s) : nullptr;
    p.apk1 = packed ? W.packed_up(s) : nullptr;
    p.a_blocks_per_expert = s.I / kPackRows;
    cudaError_t err = launch_wt<kGateUp>(W.gate, W.up, (uint64_t)s.E * s.I, s.H, ws.x_perm, P, p,
                                         pl.items_gu * p.ksplit, st);
    if (err != cudaSuccess) return err;
    if (ev_mid) cudaEventRecord(ev_mid, st);

    // down: A0/A1 = W_down rows [n0, n0 + 128) and [n0 + 128, n0 + 256); B = h rows
    p.n_blk = s.H / (2 * kWM);
    p.num_kb = s.I / kBK;
    p.ksplit = pl.ks_dn;
    p.kb_per = (p.num_kb + p.ksplit - 1) / p.ksplit;
    p.counters = ws.status + 4 + pl.n_counters_gu;
    p.partial = ws.wt_partial + pl.partial_floats_gu;
    p.w_rows_per_expert = s.H;
    p.out = ws.ybuf;
    p.out_ld = s.H;
    p.apk0 = packed ? W.packed_down(s) : nullptr;
    p.apk1 = p.apk0;
    p.a_blocks_per_expert = s.H / kPackRows;
    p.perm_tok = ws.perm_tok;
    p.perm_slot = ws.perm_slot;
    p.K = s.K;
    p.out32 = ws.ybuf_f32;
    return launch_wt<kDown>(W.down, W.down, (uint64_t)s.E * s.H, s.I, ws.hbuf, P, p,
                            pl.items_dn * p.ksplit, st);
}

}  // namespace moe
