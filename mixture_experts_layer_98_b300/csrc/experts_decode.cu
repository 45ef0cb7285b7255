// experts_decode.cu -- the expert MLPs and the combine of a decode-sized batch
// (T <= kDecodeFusedTokens) in one persistent kernel.
//
// The arithmetic is that of experts_wt.cu -- the SwiGLU expert MLP
// down(silu(gate(x)) ⊙ up(x)) with per-expert gate_proj / up_proj [I,H] and
// down_proj [H,I] (csdn page "MoE架构深度解析：128专家与8激活的智能路由",
// section "128个专家网络的组织结构与参数分布"), computed with 128 weight rows
// on the MMA's M side and a row tile's tokens on its N side, K split into
// slices when there are few items -- followed by that of combine.cu: the
// routing-weight-scaled outputs Y of a token's K pairs summed in fp32 in k
// order and rounded once (Qwen3MoeSparseMoeBlock.forward, cnblogs page
// "大模型-qwen3 MoE 详细解读").  Results are bit for bit those of the separate
// kernels.
//
// One launch runs every gate/up unit, then every down unit, then the combine,
// so a decode step pays one kernel ramp and tail instead of three:
//   * a down unit of row tile j reads all of tile j's h columns: every final
//     gate/up epilogue warp fences its h stores (for the async proxy, then at
//     gpu scope) and counts h_ready[j]; the down unit's producer waits
//     (bounded, acquire) until the count is complete, prefetching the unit's
//     first stages of packed weights into L2 meanwhile;
//   * every final down epilogue warp (column block cb = blk·4 + q: 64 output
//     columns) fences its Y stores and counts, for every row of its tile, the
//     row's token in tok_done[t·n_cb + cb]; the lane that completes a token's
//     count (its K kept pairs) has that token's K rows of those 64 columns
//     summed by its warp -- the combine is spread over the down epilogues.
// Each CTA runs its units in increasing order and every gate/up unit precedes
// every down unit, so a CTA that waits has finished its own gate/up units and
// waits only on units of CTAs that never wait; the launch is cooperative, so
// every CTA is resident.  The counters are in the workspace's status region,
// zeroed by the router kernel at the start of every forward.
//
// Up to kDecodeDirectTokens (= one 16-row box) tokens, the gate/up units take
// their token box from x itself, rows 0..T-1, rather than from gathered rows:
// the MMA computes every token of the batch against the tile's weights (the
// same N = 16 columns a gathered tile would occupy) and the epilogue keeps the
// columns of the tile's tokens, writing column perm_tok[row] to h row `row`.
// No gather runs at all.
//
// Up to kDecodeRouteTokens tokens (one per warp) the kernel also routes and
// dispatches the batch itself (launched straight after the router logits):
// every CTA sums the partial logits, routes each token (routing.cuh: softmax,
// top-k, renormalisation), counts, scans and scatters the pairs into its own
// shared memory -- the same arithmetic, in the same order, as the one-CTA
// routing kernel of dispatch.cu, so every CTA holds the same tile table --
// and the grid's last CTAs (the ones with the fewest units) write the
// forward's routing outputs (logits, top-k, counts, offsets, tile table,
// permutation) and aux, each a share.  The expert weights then start
// streaming one kernel boundary earlier.
//
// Roles per CTA (192 threads, one CTA per SM) as in experts_wt.cu: warp 0 TMA
// producer (5-stage ring: two 128x64 weight tiles and ceil(rows/16) 16-row
// token boxes per k-block), warp 1 TMEM owner and MMA issuer, warps 2-5
// epilogue.  Every wait is bounded (2 s); on expiry the CTA records
// MOE_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include "moe_common.cuh"
#include "routing.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kWM = 128;  // weight rows per MMA (M)
constexpr int kBK = 64;   // 64 bf16 = 128 bytes: one swizzle row
constexpr int kBox = 16;  // token rows per TMA box
constexpr int kStages = 5;
constexpr int kThreads = 192;
constexpr int kABytes = kWM * kBK * 2;                                 // 16 KB
constexpr int kBoxBytes = kBox * kBK * 2;                              // 2 KB
constexpr int kStageBytes = 2 * kABytes + (kWtRows / kBox) * kBoxBytes;  // 40 KB
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr uint32_t kAccCols = kWtRows;
constexpr uint32_t kTmemCols = 4 * kAccCols;  // 2 buffers x 2 accumulators
constexpr uint64_t kTimeoutNs = 2000000000ull;

enum { kGateUp = 0, kDown = 1 };

struct DecParams {
    const RowTile* tiles;
    const int32_t* n_tiles;
    int T, K, H, I;
    // per kind (0 gate/up, 1 down)
    int n_blk[2];          // weight-row blocks per row tile: I/128, H/256
    int num_kb[2];         // k-blocks of 64: H/64, I/64
    int ksplit[2];         // K slices per item
    int kb_per[2];         // k-blocks per slice
    float* partial[2];     // [items][ksplit][2][part_rows][128] slice accumulators
    int32_t* counters[2];  // [items][4] slice arrivals
    int w_rows[2];         // weight rows per expert: I, H
    int part_rows;
    int32_t* h_ready;      // [tiles] final gate/up epilogue warps done
    int32_t* tok_done;     // [T][H/256 * 4] pairs of token t stored, per column block
    __nv_bfloat16* h;      // [P, I]
    __nv_bfloat16* y;      // [P, H] token-major
    float* y32;            // the same as fp32 under a capacity (null: bf16 y)
    __nv_bfloat16* out;    // [T, H]
    const float* w_perm;
    const int32_t* perm_tok;
    const int32_t* perm_slot;
    const int32_t* inv;    // [P] (null: no pair dropped)
    int32_t* status;
    // packed weight blocks (null: row-major through the tensor maps)
    const char* pk_gate;
    const char* pk_up;
    const char* pk_down;
    int a_blocks[2];       // 128-row weight blocks per expert: I/128, H/128
    int x_direct;          // gate/up token boxes: x rows 0..T-1 (T <= kBox), not x_perm
    // routing in the kernel (routed != 0): inputs, and the outputs CTA 0 writes
    int routed;
    int E, cap, norm, nparts;
    const float* parts;    // [nparts][T][E] partial logits, summed in slice order
    const float* bias;     // selection-only expert bias [E] or null
    float* logits_out;     // [T][E] or null
    int32_t* idx_out;      // [T][K]
    float* w_out;          // [T][K]
    float* aux_out;        // [1] or null
    int32_t* counts_out;   // [E]
    int32_t* offsets_out;  // [E + 1]
    RowTile* tiles_out;
    int32_t* n_tiles_out;
    int32_t* perm_tok_out;
    int32_t* perm_slot_out;
    int32_t* inv_out;
    float* w_perm_out;
};

// The dispatch of a batch routed inside the kernel, in each CTA's shared
// memory (at most kDecodeRouteTokens tokens, so a token bitmap is one word).
constexpr int kRoutePairs = kDecodeRouteTokens * kMaxTopK;
struct RouteSmem {
    RowTile tiles[kRoutePairs];
    int32_t perm_tok[kRoutePairs];
    int32_t perm_slot[kRoutePairs];
    int32_t inv[kRoutePairs];
    float w_perm[kRoutePairs];
    int32_t idx[kRoutePairs];
    float w[kRoutePairs];
    int32_t cnt[kMaxExperts];
    int32_t base[kMaxExperts];
    uint32_t sel[kMaxExperts];
    int n_tiles;
};

template <int EPL>
__device__ __forceinline__ void route_one(const DecParams& p, int t, RouteSmem& rs,
                                          float* prob) {
    const int lane = threadIdx.x & 31;
    float l[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        if (e < p.E) {
            // every slice loaded before the first add (one memory round trip),
            // then summed in slice order
            float pv[kRouterMaxSplits];
#pragma unroll
            for (int sl = 0; sl < kRouterMaxSplits; ++sl)
                pv[sl] = sl < p.nparts ? p.parts[((size_t)sl * p.T + t) * p.E + e] : 0.f;
            float v = pv[0];
#pragma unroll
            for (int sl = 1; sl < kRouterMaxSplits; ++sl)
                if (sl < p.nparts) v += pv[sl];
            l[q] = v;
            if (p.logits_out && blockIdx.x == gridDim.x - 1)
                p.logits_out[(size_t)t * p.E + e] = v;
        } else {
            l[q] = -INFINITY;
        }
    }
    route_token<EPL>(l, p.E, p.K, p.norm, p.bias, rs.idx + t * p.K, rs.w + t * p.K,
                     prob + (size_t)t * p.E);
}

// Routing and dispatch of the whole batch by one CTA (all its threads), into
// rs; scratch: [T][E] + [E] floats of free shared memory.  The grid's last
// CTAs also write the forward's routing outputs (the logits, the tile table
// and offsets, the top-k and permutation, aux: one share each, so that no
// CTA waits on all the stores).  Ends with a CTA barrier.
__device__ void route_batch(const DecParams& p, RouteSmem& rs, float* scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.T, E = p.E, K = p.K, P = T * K;
    const int last = (int)gridDim.x - 1;
    const bool w_tab = (int)blockIdx.x == max(0, last - 1);
    const bool w_perm = (int)blockIdx.x == max(0, last - 2);
    const bool w_aux = (int)blockIdx.x == max(0, last - 3);
    float* prob = scratch;               // [T][E]
    float* term = scratch + (size_t)T * E;  // [E]
    for (int e = tid; e < E; e += blockDim.x) {
        rs.cnt[e] = 0;
        rs.sel[e] = 0u;
    }
    const int epl = (E + 31) / 32;
    for (int t = warp; t < T; t += blockDim.x / 32) {  // warp-uniform
        if (epl <= 1) route_one<1>(p, t, rs, prob);
        else if (epl <= 2) route_one<2>(p, t, rs, prob);
        else if (epl <= 4) route_one<4>(p, t, rs, prob);
        else route_one<8>(p, t, rs, prob);
    }
    __syncthreads();
    for (int i = tid; i < P; i += blockDim.x) {
        const int e = rs.idx[i];
        atomicAdd(&rs.cnt[e], 1);
        atomicOr(&rs.sel[e], 1u << (i / K));
    }
    __syncthreads();
    // rows and tiles in expert order: one warp, lane l owning the run of
    // experts [l·epl, (l+1)·epl), one shuffle scan over the lanes' totals
    if (warp == 0) {
        const int e0 = lane * epl, e1 = min(E, e0 + epl);
        int sk = 0, st = 0;
        for (int e = e0; e < e1; ++e) {
            const int c = rs.cnt[e];
            const int kept = (p.cap > 0 && c > p.cap) ? p.cap : c;  // first cap pairs, token order
            sk += kept;
            st += (kept + kWtRows - 1) / kWtRows;
        }
        int ik = sk, it = st;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ik, off);
            const int b = __shfl_up_sync(0xffffffffu, it, off);
            if (lane >= off) {
                ik += a;
                it += b;
            }
        }
        int base = ik - sk, tb = it - st;
        for (int e = e0; e < e1; ++e) {
            const int c = rs.cnt[e];
            const int kept = (p.cap > 0 && c > p.cap) ? p.cap : c;
            const int nt = (kept + kWtRows - 1) / kWtRows;
            rs.base[e] = base;
            for (int j = 0; j < nt; ++j) {
                RowTile tl;
                tl.expert = e;
                tl.row0 = base + j * kWtRows;
                tl.nrows = min(kWtRows, kept - j * kWtRows);
                tl.pad = 0;
                rs.tiles[tb + j] = tl;
            }
            if (w_tab) {
                p.counts_out[e] = c;
                p.offsets_out[e] = base;
            }
            base += kept;
            tb += nt;
        }
        if (lane == 31) {
            rs.n_tiles = it;
            if (w_tab) {
                p.offsets_out[E] = ik;
                *p.n_tiles_out = it;
            }
        }
    }
    __syncthreads();
    // scatter: a pair's row is its expert's base + the tokens before it that chose the expert
    for (int i = tid; i < P; i += blockDim.x) {
        const int t = i / K, k = i - t * K, e = rs.idx[i];
        const int rank = __popc(rs.sel[e] & ((1u << t) - 1u));
        if (p.cap > 0 && rank >= p.cap) {
            rs.inv[i] = -1;
            continue;
        }
        const int row = rs.base[e] + rank;
        rs.perm_tok[row] = t;
        rs.perm_slot[row] = k;
        rs.w_perm[row] = rs.w[i];
        rs.inv[i] = row;
    }
    if (w_aux && p.aux_out) {
        // aux = E · sum_e f_e · P_e, f_e = counts/(T·K), P_e the mean probability
        // (token order), the expert terms summed in a fixed order
        for (int e = tid; e < E; e += blockDim.x) {
            float psum = 0.f;
            for (int t = 0; t < T; ++t) psum += prob[(size_t)t * E + e];
            const float f = (float)rs.cnt[e] / ((float)T * (float)K);
            term[e] = f * (psum / (float)T);
        }
        __syncthreads();
        if (warp == 0) {
            float v = 0.f;
            for (int j = lane; j < E; j += 32) v += term[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) *p.aux_out = (float)E * v;
        }
    }
    if (w_perm || w_tab) __syncthreads();  // the scatter's rows, for the stores below
    if (w_perm) {
        for (int i = tid; i < P; i += blockDim.x) {
            p.idx_out[i] = rs.idx[i];
            p.w_out[i] = rs.w[i];
            const int row = rs.inv[i];
            p.inv_out[i] = row;
            if (row >= 0) {
                p.perm_tok_out[row] = rs.perm_tok[row];
                p.perm_slot_out[row] = rs.perm_slot[row];
                p.w_perm_out[row] = rs.w_perm[row];
            }
        }
    }
    if (w_tab)
        for (int j = tid; j < rs.n_tiles; j += blockDim.x) p.tiles_out[j] = rs.tiles[j];
    __syncthreads();
}

struct Unit {
    int kind, pitem, ks, tile, blk;
};

__device__ __forceinline__ Unit unit_of(const DecParams& p, int u, int n_gu) {
    Unit x;
    x.kind = u >= n_gu ? kDown : kGateUp;
    const int v = x.kind == kDown ? u - n_gu : u;
    x.pitem = v / p.ksplit[x.kind];
    x.ks = v % p.ksplit[x.kind];
    x.tile = x.pitem / p.n_blk[x.kind];
    x.blk = x.pitem % p.n_blk[x.kind];
    return x;
}

// Epilogue of one output row and weight row i of the block (experts_wt.cu).
__device__ __forceinline__ void store_out(const DecParams& p, const float* w_perm,
                                          const int32_t* perm_tok, const int32_t* perm_slot,
                                          int kind, size_t row, int blk, int i, float d0,
                                          float d1) {
    if (kind == kGateUp) {
        p.h[row * p.I + (size_t)blk * kWM + i] = __float2bfloat16_rn(silu_f(d0) * d1);
    } else {
        const float wr = w_perm[row];
        const size_t yrow = (size_t)perm_tok[row] * p.K + (size_t)perm_slot[row];
        if (p.y32) {
            float* o = p.y32 + yrow * p.H + (size_t)blk * (2 * kWM);
            o[i] = wr * d0;
            o[kWM + i] = wr * d1;
        } else {
            __nv_bfloat16* o = p.y + yrow * p.H + (size_t)blk * (2 * kWM);
            o[i] = __float2bfloat16_rn(wr * d0);
            o[kWM + i] = __float2bfloat16_rn(wr * d1);
        }
    }
}

__device__ __forceinline__ float ld_bf16_cg(const __nv_bfloat16* p) {
    const unsigned short v = __ldcg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float((uint32_t)v << 16);
}

__global__ void __launch_bounds__(kThreads, 1)
    expert_decode_kernel(const __grid_constant__ CUtensorMap tmWg,
                         const __grid_constant__ CUtensorMap tmWu,
                         const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmWd,
                         const __grid_constant__ CUtensorMap tmH, const DecParams p) {
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
    __shared__ RouteSmem rs;

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
        ptx::prefetch_tmap(&tmWg);
        ptx::prefetch_tmap(&tmWu);
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmWd);
        ptx::prefetch_tmap(&tmH);
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
    // the dispatch: routed here (the ring is still free: scratch), or read
    // from the dispatch kernel's outputs
    if (p.routed) route_batch(p, rs, reinterpret_cast<float*>(smem));
    const RowTile* tiles = p.routed ? rs.tiles : p.tiles;
    const int32_t* perm_tok = p.routed ? rs.perm_tok : p.perm_tok;
    const int32_t* perm_slot = p.routed ? rs.perm_slot : p.perm_slot;
    const float* w_perm = p.routed ? rs.w_perm : p.w_perm;
    const int32_t* inv = p.routed ? (p.cap > 0 ? rs.inv : nullptr) : p.inv;
    const int n_tiles = p.routed ? rs.n_tiles : *p.n_tiles;
    const int n_gu = n_tiles * p.n_blk[0] * p.ksplit[0];
    const int total = n_gu + n_tiles * p.n_blk[1] * p.ksplit[1];

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // the weights are read once per forward: their lines go first when
            // L2 needs room, so they do not push out the activations, h, the
            // slice accumulators and Y that the forward reads back
            const uint64_t pol_once = ptx::l2_policy_evict_first();
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                const Unit x = unit_of(p, u, n_gu);
                const RowTile tl = tiles[x.tile];
                const int kb0 = x.ks * p.kb_per[x.kind];
                const int kb1 = min(p.num_kb[x.kind], kb0 + p.kb_per[x.kind]);
                const int nbox = (tl.nrows + kBox - 1) / kBox;
                int a0, a1, a0b, a1b;
                const char* pk0;
                const char* pk1;
                if (x.kind == kGateUp) {
                    a0 = a1 = tl.expert * p.w_rows[0] + x.blk * kWM;
                    a0b = a1b = x.blk;
                    pk0 = p.pk_gate;
                    pk1 = p.pk_up;
                } else {
                    a0 = tl.expert * p.w_rows[1] + x.blk * (2 * kWM);
                    a1 = a0 + kWM;
                    a0b = 2 * x.blk;
                    a1b = 2 * x.blk + 1;
                    pk0 = pk1 = p.pk_down;
                }
                const size_t e0 = (size_t)tl.expert * p.a_blocks[x.kind];
                const size_t nkb = (size_t)p.num_kb[x.kind];
                if (x.kind == kDown) {
                    // h rows of this tile: every gate/up epilogue warp of the tile done
                    const int need = p.n_blk[0] * 4;
                    if (ptx::ld_acquire_gpu(&p.h_ready[x.tile]) < need) {
                        if (pk0) {  // the unit's first stages of weights into L2 meanwhile
                            const int npf = min(kb1 - kb0, kStages);
                            ptx::prefetch_l2_range(
                                pk0 + ((e0 + a0b) * nkb + kb0) * kPackBlockBytes,
                                (size_t)npf * kPackBlockBytes);
                            ptx::prefetch_l2_range(
                                pk1 + ((e0 + a1b) * nkb + kb0) * kPackBlockBytes,
                                (size_t)npf * kPackBlockBytes);
                        }
                        const long long t0 = clock64();
                        const long long lim = (long long)(kTimeoutNs * 2.032);
                        for (uint32_t i = 1;; ++i) {
                            __nanosleep(64);
                            if (ptx::ld_acquire_gpu(&p.h_ready[x.tile]) >= need) break;
                            if ((i & 15u) == 0u && (abort_s || clock64() - t0 > lim)) {
                                abort_s = 1;
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                    }
                    // (the writers of h fenced their stores for the async proxy
                    // before counting them)
                }
                const CUtensorMap* mw0 = x.kind == kGateUp ? &tmWg : &tmWd;
                const CUtensorMap* mw1 = x.kind == kGateUp ? &tmWu : &tmWd;
                const CUtensorMap* mb = x.kind == kGateUp ? &tmX : &tmH;
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
                    if (pk0) {  // packed: each weight tile is one contiguous 16 KB block
                        ptx::bulk_load_hint(sA, pk0 + ((e0 + a0b) * nkb + kb) * kPackBlockBytes,
                                            kABytes, &full_bar[stage], pol_once);
                        ptx::bulk_load_hint(sA + kABytes,
                                            pk1 + ((e0 + a1b) * nkb + kb) * kPackBlockBytes,
                                            kABytes, &full_bar[stage], pol_once);
                    } else {
                        ptx::tma_load_2d(sA, mw0, &full_bar[stage], kb * kBK, a0);
                        ptx::tma_load_2d(sA + kABytes, mw1, &full_bar[stage], kb * kBK, a1);
                    }
                    // x read directly: one box, the whole batch (nrows <= T <= kBox)
                    const int brow = (p.x_direct && x.kind == kGateUp) ? 0 : tl.row0;
                    for (int b = 0; b < nbox; ++b)
                        ptx::tma_load_2d(sB + b * kBoxBytes, mb, &full_bar[stage], kb * kBK,
                                         brow + b * kBox);
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
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                const Unit x = unit_of(p, u, n_gu);
                const int kb0 = x.ks * p.kb_per[x.kind];
                const int kb1 = min(p.num_kb[x.kind], kb0 + p.kb_per[x.kind]);
                const int nrows = tiles[x.tile].nrows;
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
        const int q = warp & 3;       // TMEM lane quadrant of this warp
        const int i = q * 32 + lane;  // weight row within the 128-row block
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit x = unit_of(p, u, n_gu);
            const RowTile tl = tiles[x.tile];
            // Accumulator column -> tile row: the identity, except for gate/up
            // units on x itself, where column cc is token cc and lane cc holds
            // its row in the tile (-1: the token is not in the tile).  Read
            // before the accumulator wait, so the loads overlap the MMAs.
            const bool direct = p.x_direct && x.kind == kGateUp;
            int jm = -1;
            if (direct) {
                const int tok = lane < tl.nrows ? perm_tok[tl.row0 + lane] : -1;
                for (int j = 0; j < tl.nrows; ++j)
                    if (__shfl_sync(0xffffffffu, tok, j) == lane) jm = j;
            }
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
            bool final_part = true;  // this warp wrote the unit's outputs
            if (p.ksplit[x.kind] == 1) {
#pragma unroll 1
                for (int c = 0; c < n; c += kBox) {
                    uint32_t v0[kBox], v1[kBox];
                    ptx::tmem_ld16(t0 + c, v0);
                    ptx::tmem_ld16(t1 + c, v1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < kBox; ++cc) {
                        const int j = direct ? __shfl_sync(0xffffffffu, jm, cc)
                                             : (c + cc < tl.nrows ? c + cc : -1);
                        if (j >= 0)
                            store_out(p, w_perm, perm_tok, perm_slot, x.kind, (size_t)tl.row0 + j, x.blk, i,
                                      __uint_as_float(v0[cc]), __uint_as_float(v1[cc]));
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
            } else {
                // This slice's accumulators -> partial[kind][pitem][ks], then free
                // TMEM; the last slice of the item (per warp quadrant) adds all
                // slices in slice order.
                const int ksn = p.ksplit[x.kind];
                const size_t slice = (size_t)2 * p.part_rows * kWM;
                float* mine = p.partial[x.kind] + ((size_t)x.pitem * ksn + x.ks) * slice;
#pragma unroll 1
                for (int c = 0; c < n; c += kBox) {
                    uint32_t v0[kBox], v1[kBox];
                    ptx::tmem_ld16(t0 + c, v0);
                    ptx::tmem_ld16(t1 + c, v1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < kBox; ++cc) {
                        const int j = direct ? __shfl_sync(0xffffffffu, jm, cc)
                                             : (c + cc < tl.nrows ? c + cc : -1);
                        if (j >= 0) {
                            __stcg(mine + (size_t)j * kWM + i, __uint_as_float(v0[cc]));
                            __stcg(mine + ((size_t)p.part_rows + j) * kWM + i,
                                   __uint_as_float(v1[cc]));
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
                __threadfence();
                __syncwarp();
                int32_t* cnt = p.counters[x.kind] + x.pitem * 4 + q;
                int last = 0;
                if (lane == 0) last = atomicAdd(cnt, 1) == ksn - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                final_part = last != 0;
                if (last) {
                    __threadfence();
                    const float* all = p.partial[x.kind] + (size_t)x.pitem * ksn * slice;
#pragma unroll 1
                    for (int j = 0; j < tl.nrows; ++j) {
                        float s0 = 0.f, s1 = 0.f;
                        for (int sl = 0; sl < ksn; ++sl) {
                            const float* src = all + (size_t)sl * slice;
                            s0 += __ldcg(src + (size_t)j * kWM + i);
                            s1 += __ldcg(src + ((size_t)p.part_rows + j) * kWM + i);
                        }
                        store_out(p, w_perm, perm_tok, perm_slot, x.kind, (size_t)tl.row0 + j, x.blk, i, s0, s1);
                    }
                    if (lane == 0) *cnt = 0;
                }
            }
            if (final_part) {
                // this warp's h / Y stores before its count; h is read back by
                // other CTAs' TMA loads (the async proxy)
                if (x.kind == kGateUp) ptx::fence_proxy_async_global();
                __threadfence();
                __syncwarp();
                if (x.kind == kGateUp) {
                    if (lane == 0) atomicAdd(&p.h_ready[x.tile], 1);
                } else {
                    const int ncb = p.n_blk[1] * 4, cb = x.blk * 4 + q;
                    const size_t c0 = (size_t)x.blk * (2 * kWM) + (size_t)q * 32 + lane;
                    const size_t c1 = c0 + kWM;
                    for (int r0 = 0; r0 < tl.nrows; r0 += 32) {
                        // lane: row r0 + lane of the tile -> its token's count
                        int tok = -1;
                        if (r0 + lane < tl.nrows) {
                            const int t = perm_tok[tl.row0 + r0 + lane];
                            int kept = p.K;
                            if (inv) {
                                kept = 0;
                                for (int k = 0; k < p.K; ++k)
                                    kept += inv[(size_t)t * p.K + k] >= 0 ? 1 : 0;
                            }
                            if (atomicAdd(&p.tok_done[(size_t)t * ncb + cb], 1) == kept - 1)
                                tok = t;
                        }
                        unsigned m = __ballot_sync(0xffffffffu, tok >= 0);
                        if (m) __threadfence();  // the other warps' Y stores of these tokens
                        while (m) {
                            const int src = __ffs(m) - 1;
                            m &= m - 1;
                            const int t = __shfl_sync(0xffffffffu, tok, src);
                            // out[t] = sum over kept k of Y[t*K + k] (k order, fp32, one
                            // rounding): all K loads in flight, then the adds in order
                            float v0[kMaxTopK], v1[kMaxTopK];
                            bool kp[kMaxTopK];
#pragma unroll
                            for (int k = 0; k < kMaxTopK; ++k) {
                                const size_t pr = (size_t)t * p.K + k;
                                kp[k] = k < p.K && (!inv || inv[pr] >= 0);
                                if (p.y32) {
                                    v0[k] = kp[k] ? __ldcg(p.y32 + pr * p.H + c0) : 0.f;
                                    v1[k] = kp[k] ? __ldcg(p.y32 + pr * p.H + c1) : 0.f;
                                } else {
                                    v0[k] = kp[k] ? ld_bf16_cg(p.y + pr * p.H + c0) : 0.f;
                                    v1[k] = kp[k] ? ld_bf16_cg(p.y + pr * p.H + c1) : 0.f;
                                }
                            }
                            float s0 = 0.f, s1 = 0.f;
#pragma unroll
                            for (int k = 0; k < kMaxTopK; ++k)
                                if (kp[k]) {
                                    s0 += v0[k];
                                    s1 += v1[k];
                                }
                            p.out[(size_t)t * p.H + c0] = __float2bfloat16_rn(s0);
                            p.out[(size_t)t * p.H + c1] = __float2bfloat16_rn(s1);
                        }
                    }
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

}  // namespace

bool experts_decode_supported(const Sizes& s) {
    return s.T >= 1 && s.T <= kDecodeFusedTokens && experts_wt_supported(s);
}

cudaError_t launch_experts_decode(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                                  const __nv_bfloat16* x, const int32_t* inv,
                                  __nv_bfloat16* out, cudaStream_t st, const DecodeRouting* route) {
    if (!experts_decode_supported(s)) return cudaErrorInvalidValue;
    static_assert(kThreads / 32 >= kDecodeRouteTokens, "one routing warp per token");
    if (route && (s.T > kDecodeRouteTokens || s.K > kMaxTopK || s.E > kMaxExperts ||
                  route->nparts < 1 || route->nparts > kRouterMaxSplits))
        return cudaErrorInvalidValue;
    const bool packed = W.packed != nullptr;
    const long long P = s.P();
    const WtPlan pl = wt_plan(s);
    DecParams p{};
    p.tiles = ws.tiles;
    p.n_tiles = ws.n_tiles;
    p.T = s.T;
    p.K = s.K;
    p.H = s.H;
    p.I = s.I;
    p.n_blk[0] = s.I / kWM;
    p.n_blk[1] = s.H / (2 * kWM);
    p.num_kb[0] = s.H / kBK;
    p.num_kb[1] = s.I / kBK;
    p.ksplit[0] = pl.ks_gu;
    p.ksplit[1] = pl.ks_dn;
    for (int k = 0; k < 2; ++k) p.kb_per[k] = (p.num_kb[k] + p.ksplit[k] - 1) / p.ksplit[k];
    p.partial[0] = ws.wt_partial;
    p.partial[1] = ws.wt_partial + pl.partial_floats_gu;
    p.counters[0] = ws.status + 4;
    p.counters[1] = ws.status + 4 + pl.n_counters_gu;
    p.w_rows[0] = s.I;
    p.w_rows[1] = s.H;
    p.part_rows = pl.part_rows;
    p.h_ready = ws.status + 4 + pl.n_counters_gu + pl.n_counters_dn;
    p.tok_done = p.h_ready + pl.n_ready;
    p.h = ws.hbuf;
    p.y = ws.ybuf;
    p.y32 = ws.ybuf_f32;
    p.out = out;
    p.w_perm = ws.w_perm;
    p.perm_tok = ws.perm_tok;
    p.perm_slot = ws.perm_slot;
    p.inv = inv;
    p.status = ws.status;
    p.pk_gate = packed ? W.packed_gate(s) : nullptr;
    p.pk_up = packed ? W.packed_up(s) : nullptr;
    p.pk_down = packed ? W.packed_down(s) : nullptr;
    p.a_blocks[0] = s.I / kPackRows;
    p.a_blocks[1] = s.H / kPackRows;
    static_assert(kDecodeDirectTokens <= kBox, "the whole batch in one token box");
    static_assert(kDecodeRouteTokens <= 32, "a token bitmap is one word");
    p.x_direct = s.T <= kDecodeDirectTokens ? 1 : 0;
    if (route) {
        p.routed = 1;
        p.E = s.E;
        p.cap = route->cap;
        p.norm = route->norm;
        p.nparts = route->nparts;
        p.parts = route->parts;
        p.bias = route->bias;
        p.logits_out = route->logits;
        p.idx_out = route->idx;
        p.w_out = route->w;
        p.aux_out = route->aux;
        p.counts_out = ws.counts;
        p.offsets_out = ws.offsets;
        p.tiles_out = ws.tiles;
        p.n_tiles_out = ws.n_tiles;
        p.perm_tok_out = ws.perm_tok;
        p.perm_slot_out = ws.perm_slot;
        p.inv_out = ws.inv;
        p.w_perm_out = ws.w_perm;
    }

    CUtensorMap mx, mh, mg, mu, md;
    const bool mx_ok = p.x_direct ? make_tma_2d(&mx, x, s.T, s.H, kBox)
                                  : make_tma_2d(&mx, ws.x_perm, P, s.H, kBox);
    if (!mx_ok || !make_tma_2d(&mh, ws.hbuf, P, s.I, kBox)) return cudaErrorInvalidValue;
    if (packed) {  // the weight maps are not used
        mg = mu = md = mx;
    } else if (!make_tma_2d(&mg, W.gate, (uint64_t)s.E * s.I, s.H, kWM) ||
               !make_tma_2d(&mu, W.up, (uint64_t)s.E * s.I, s.H, kWM) ||
               !make_tma_2d(&md, W.down, (uint64_t)s.E * s.H, s.I, kWM)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = ensure_smem((const void*)expert_decode_kernel, kSmemBytes);
    if (err != cudaSuccess) return err;
    long long grid = num_sms();
    const long long items = pl.items_gu * pl.ks_gu + pl.items_dn * pl.ks_dn;
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, expert_decode_kernel, mg, mu, mx, md, mh, p);
    count_launches(1);
    return err;
}

}  // namespace moe
