// moe_common.cuh -- shared definitions of the CUDA library (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe_b300.h"

namespace moe {

// ---- limits of this implementation ----------------------------------------
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 16;
constexpr int kChunkTokens = 256;    // tokens per dispatch chunk (one CTA)
constexpr int kRouterTokens = 32;    // tokens per router CTA (SIMT router)
constexpr int kStreamRows = 8;       // rows per tile of the weight-streaming kernels
constexpr int kTcRows = 128;         // rows per tile of the tcgen05 grouped GEMMs
constexpr int kPairRows = 256;       // rows per tile of the CTA-pair grouped GEMMs
constexpr int kWtRows = 64;          // rows per tile of the weights-as-M tcgen05 kernels
constexpr int kRouterMaxSplits = 4;  // slices of H the tensor-core router may split into

// Packed expert weights (pack.cu): 128-row x 64-column blocks of 16 KB, each
// in the 128-byte swizzled K-major arrangement, ordered (expert, row block,
// column block); W_gate's blocks, then W_up's, then W_down's.
constexpr int kPackRows = 128;
constexpr int kPackCols = 64;
constexpr int kPackBlockBytes = kPackRows * kPackCols * 2;

// 4-bit group-quantised experts (quant.cu): 4 KB code blocks of 128 rows x
// 64 columns and 512-byte scale blocks of 128 rows x one 128-column group.
constexpr int kQ4CodeBlockBytes = kPackRows * kPackCols / 2;
constexpr int kQ4ScaleBlockBytes = kPackRows * 4;
struct Q4Sections {
    const char* codes[3];   // W_gate, W_up, W_down
    const char* scales[3];
};
bool q4_supported(int H, int E, int I);  // I % 128 == 0, H % 256 == 0
size_t q4_experts_bytes(int H, int E, int I);
Q4Sections q4_sections(const char* base, int H, int E, int I);
cudaError_t launch_quantize_q4(const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                               const __nv_bfloat16* Wd, int H, int E, int I, char* q4,
                               cudaStream_t st);
cudaError_t launch_dequantize_q4(const char* q4, int H, int E, int I, __nv_bfloat16* Wg,
                                 __nv_bfloat16* Wu, __nv_bfloat16* Wd, cudaStream_t st);

// Eight dequantised weights (one code word, columns 8c..8c+7) as four bf16
// pairs: w' = bf16(q·s + b) with one rounding.  (word >> 4j) & 0x000F000F puts
// the codes of columns 2j, 2j+1 in the two halves; OR-ing 0x4300 makes each
// half the bf16 value 128 + q, and subtracting 128 leaves q exactly.
__device__ __forceinline__ uint4 q4_dequant8(uint32_t w, uint32_t sbw) {
    const __nv_bfloat162 s2 = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)(sbw & 0xFFFFu)));
    const __nv_bfloat162 b2 = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)(sbw >> 16)));
    const __nv_bfloat162 k128 = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)0x4300u));
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t t = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&t);
        v = __hfma2(__hsub2(v, k128), s2, b2);
        o[j] = *reinterpret_cast<const uint32_t*>(&v);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

struct Sizes;

// The expert weights of a forward: row-major matrices, or the packed blocks.
struct ExpertWeights {
    const __nv_bfloat16* gate;  // [E, I, H] row-major (null when packed)
    const __nv_bfloat16* up;    // [E, I, H]
    const __nv_bfloat16* down;  // [E, H, I]
    const char* packed;         // packed blocks (null when row-major)
    const char* q4 = nullptr;   // 4-bit quantised experts (quant.cu), or null
    const char* packed_gate(const Sizes& s) const;
    const char* packed_up(const Sizes& s) const;
    const char* packed_down(const Sizes& s) const;
};

// One tile of token-expert rows, all routed to one expert: rows
// [row0, row0 + nrows) of the dispatch order.
struct __align__(16) RowTile {
    int expert;
    int row0;
    int nrows;
    int pad;
};

// Scratch regions carved from one workspace allocation (device pointers).
struct Workspace {
    int32_t* chunk_counts;  // [nchunks, E]
    int32_t* chunk_base;    // [nchunks, E]
    int32_t* counts;        // [E]
    int32_t* offsets;       // [E + 1]
    RowTile* tiles;         // [max_tiles]
    int32_t* n_tiles;       // [1]
    int32_t* status;        // [4 + wt counters] device-side error words, then the
                            // split-K arrival counters; all zeroed by the router
    int n_clear;            // ints zeroed from status at the start of a forward
    float* wt_partial;      // slice accumulators of the split weights-as-M kernels
    float* p_partial;       // [n_router_blocks, E]
    int32_t* perm_tok;      // [P]
    int32_t* perm_slot;     // [P]
    int32_t* inv;           // [P]
    float* w_perm;          // [P]
    float* logit_parts;     // [kRouterMaxSplits, T, E] partial logits
    int32_t* topk_idx;      // [T, K] when the caller passes NULL
    float* topk_w;          // [T, K] when the caller passes NULL
    __nv_bfloat16* x_perm;  // [P, H] (tcgen05 path)
    __nv_bfloat16* hbuf;    // [P, I]
    __nv_bfloat16* ybuf;    // [P, H] token-major: the pair (t, k) at row t*K + k
    float* ybuf_f32;        // the same region as fp32 [P, H] when the forward keeps the
                            // weighted expert outputs in fp32 (under an expert
                            // capacity), else null; the expert kernels then store Y
                            // here and the combine reads it from here
    size_t bytes;
};

struct Sizes {
    int T, H, E, K, I;
    long long P() const { return (long long)T * K; }
    int nchunks() const { return (T + kChunkTokens - 1) / kChunkTokens; }
    int nrouter() const { return (T + kRouterTokens - 1) / kRouterTokens; }
    long long max_tiles(int rows_per_tile) const {
        return (P() + rows_per_tile - 1) / rows_per_tile + E;
    }
};

inline const char* ExpertWeights::packed_gate(const Sizes&) const { return packed; }
inline const char* ExpertWeights::packed_up(const Sizes& s) const {
    return packed + (size_t)s.E * s.I * s.H * 2;
}
inline const char* ExpertWeights::packed_down(const Sizes& s) const {
    return packed + (size_t)2 * s.E * s.I * s.H * 2;
}

// Packing (pack.cu): shapes with I % 128 == 0 and H % 256 == 0.
bool packed_supported(int H, int E, int I);
size_t packed_matrix_bytes(int H, int E, int I);
cudaError_t launch_pack_experts(const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                                const __nv_bfloat16* Wd, int H, int E, int I, char* packed,
                                cudaStream_t st);

// Lays out (and, when base != nullptr, fills) the workspace; returns bytes.
// y_f32: the Y region holds fp32 values (twice the bytes; Y is the last
// region, so every other region sits at the same offset either way).
size_t layout_workspace(const Sizes& s, char* base, Workspace* ws, bool y_f32);

// ---- kernels' host launchers (each returns cudaError_t of the launch) ------
// CUDA-core router: expert- and H-split logits kernel (partial logits in
// parts [kRouterMaxSplits][T][E]) + per-token routing kernel; writes
// s.nrouter() rows of probability sums; logits (may be null) gets the sum.
// bias (fp32 [E] or null): selection-only expert bias (routing.cuh).
cudaError_t launch_router(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                          int norm, const float* bias, float* logits, float* parts, int32_t* idx,
                          float* w, float* p_partial, int32_t* status, int n_clear,
                          cudaStream_t st);
// The logits kernel of launch_router alone (nsplit slices of H, from
// router_simt_splits), for the small-batch path that routes in the dispatch.
int router_simt_splits(const Sizes& s);
cudaError_t launch_router_logits(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                                 int nsplit, float* parts, int32_t* status, int n_clear,
                                 cudaStream_t st);
// tcgen05 router logits: nsplit slices of H, partial logits [nsplit][T][E]
// into parts (then launch_route_from_logits with those parts).
cudaError_t launch_router_tc(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const Sizes& s,
                             int nsplit, float* parts, int32_t* status, int n_clear,
                             cudaStream_t st);
int router_tc_splits(const Sizes& s);
bool router_tc_supported(const Sizes& s);  // E <= 128
// Softmax, top-k, renorm and per-32-token probability sums (s.nrouter() rows)
// from the sum of nparts partial-logit arrays; logits_out (may be null) gets the sum.
cudaError_t launch_route_from_logits(const float* parts, int nparts, float* logits_out,
                                     const Sizes& s, int norm, const float* bias, int32_t* idx,
                                     float* w, float* p_partial, cudaStream_t st);
// p_partial holds n_partials rows of per-expert probability sums (for aux).
// x != null: also gather x_perm[row] = x[perm_tok[row]].
// cap > 0: each expert keeps its first cap pairs (token order); the others
// get inv = -1 and no row.  counts stay the routed pairs; offsets[E] = rows.
cudaError_t launch_dispatch(const int32_t* idx, const float* w, const __nv_bfloat16* x,
                            const Sizes& s, const Workspace& ws, int rows_per_tile,
                            const float* p_partial, int n_partials, float* aux, int cap,
                            cudaStream_t st);
// Batches of at most kRouteDispatchTokens tokens: routing (softmax, top-k,
// renorm from nparts partial logits) and the whole dispatch (counts, offsets,
// tile table, aux, permutation; gather when x != null) in one CTA, then the
// gather kernel.
constexpr int kRouteDispatchTokens = 32;
cudaError_t launch_route_dispatch_small(const float* parts, int nparts, float* logits_out,
                                        int norm, const float* bias, int32_t* idx, float* w,
                                        const __nv_bfloat16* x, const Sizes& s,
                                        const Workspace& ws, int rows_per_tile, float* aux,
                                        int cap, cudaStream_t st);
// ev_mid (may be null) is recorded between the gate/up and the down launch.
// The streaming kernels stage their input rows from x through ws.perm_tok;
// the tcgen05 kernels read the gathered rows from ws.x_perm.
// The streaming kernels need row-major weights; the tcgen05 kernels take
// either form.
cudaError_t launch_experts_streaming(const __nv_bfloat16* x, const ExpertWeights& W,
                                     const Sizes& s, const Workspace& ws, cudaStream_t st,
                                     cudaEvent_t ev_mid);
cudaError_t launch_experts_tcgen05(const ExpertWeights& W, const Sizes& s,
                                   const Workspace& ws, cudaStream_t st, cudaEvent_t ev_mid);
// The same GEMMs on CTA pairs (tcgen05 cta_group::2, 256-row tiles from a tile
// table built at kPairRows); needs I % 128 == 0 and H % 256 == 0.
bool experts_pair_supported(const Sizes& s);
cudaError_t launch_experts_pair(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                                cudaStream_t st, cudaEvent_t ev_mid);
// Small batches: the expert weights are the MMA's M side (128 weight rows per
// MMA) and a tile's <= kWtRows token rows its N side; reads ws.x_perm.
// Needs I % 128 == 0 and H % 256 == 0 (experts_wt_supported).
bool experts_wt_supported(const Sizes& s);
// K-split plan of the weights-as-M kernels (a function of the sizes only, so
// that the workspace size does not depend on the device).
struct WtPlan {
    int ks_gu = 1, ks_dn = 1;               // K slices of the gate/up and down items
    long long items_gu = 0, items_dn = 0;   // upper bounds on the items
    int part_rows = 0;                      // token rows kept per slice accumulator
    size_t partial_floats_gu = 0;           // gate/up slice accumulators (first)
    size_t partial_floats = 0;              // slice-accumulator buffer: gate/up, then down
    int n_counters_gu = 0, n_counters_dn = 0;  // split-K arrival counters
    int n_ready = 0, n_cdone = 0;           // fused decode kernel: h_ready, tok_done
    int n_counters = 0;                     // all of the above, zeroed every forward
};
WtPlan wt_plan(const Sizes& s);
cudaError_t launch_experts_wt(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                              cudaStream_t st, cudaEvent_t ev_mid);
// The experts on 4-bit quantised weights (experts_q4.cu): the q4 buffer of
// launch_quantize_q4; shapes q4_supported and experts_wt_supported.
cudaError_t launch_experts_q4(const char* q4, const Sizes& s, const Workspace& ws,
                              cudaStream_t st, cudaEvent_t ev_mid);
// The same on warp-level MMAs with the weights dequantised into registers
// (experts_q4_mma.cu): decode batches, T <= kQ4MmaTokens under MOE_PATH_AUTO,
// from a tile table of kQ4MmaRows-row tiles; its own items and K slices
// (fitted to two CTAs per SM), whose slice accumulators and counters share the
// weights-as-M plan's workspace regions (sized for the larger of the two).
constexpr int kQ4MmaTokens = 64;
constexpr int kQ4MmaRows = 16;
struct Q4MmaPlan {
    int ks_gu = 1, ks_dn = 1;
    long long items_gu = 0, items_dn = 0;   // upper bounds on the items
    int part_rows = 0;
    size_t partial_floats_gu = 0;           // gate/up slice accumulators (first)
    size_t partial_floats = 0;              // gate/up, then down
    int n_counters_gu = 0;                  // arrival counters: 8 per split item
    int n_counters = 0;
};
Q4MmaPlan q4mma_plan(const Sizes& s);
cudaError_t launch_experts_q4_mma(const char* q4, const Sizes& s, const Workspace& ws,
                                  cudaStream_t st, cudaEvent_t ev_mid);
// Decode batches (1 <= T <= kDecodeFusedTokens, shapes experts_wt_supported):
// the weights-as-M gate/up and down units and the combine in one cooperative
// persistent kernel (experts_decode.cu); writes out directly.  Up to
// kDecodeDirectTokens tokens its gate/up units read x itself (all tokens in
// one MMA column block) and no gathered rows are needed; above, x_perm.
constexpr int kDecodeFusedTokens = 64;
constexpr int kDecodeAutoTokens = 16;  // MOE_PATH_AUTO uses the fused kernel up to here
constexpr int kDecodeDirectTokens = 16;
// ... and up to kDecodeRouteTokens tokens it also routes and dispatches the
// batch itself (one routing warp per token), right after the router logits.
constexpr int kDecodeRouteTokens = 6;
bool experts_decode_supported(const Sizes& s);
// Routing done by the fused decode kernel itself (T <= kDecodeDirectTokens):
// its inputs (the router's partial logits) and the forward's routing outputs.
struct DecodeRouting {
    const float* parts;
    int nparts;
    float* logits;       // may be null
    int norm;
    const float* bias;   // may be null
    int32_t* idx;
    float* w;
    float* aux;          // may be null
    int cap;
};
cudaError_t launch_experts_decode(const ExpertWeights& W, const Sizes& s, const Workspace& ws,
                                  const __nv_bfloat16* x, const int32_t* inv,
                                  __nv_bfloat16* out, cudaStream_t st,
                                  const DecodeRouting* route = nullptr);
// out[t] = sum over k of Y row t*K + k (Y token-major, as the expert kernels
// store it), skipping the pairs with inv[t*K + k] < 0 when inv != null
// (dropped by a capacity); with y_by_inv, Y is in dispatch order and row
// inv[t*K + k] is read instead.  Y32 != null: Y is fp32 there (Y unused).
cudaError_t launch_combine(const __nv_bfloat16* Y, const float* Y32, const int32_t* inv,
                           bool y_by_inv, int T, int K, int H, __nv_bfloat16* out,
                           cudaStream_t st);

int num_sms();  // of the current device (cached)

// Raises func's dynamic shared-memory limit to at least `bytes` on the current
// device (once per device and kernel; later calls are a cached no-op).
cudaError_t ensure_smem(const void* func, int bytes);

// Row-major bf16 matrix [rows, cols] -> 2-D TMA map with a box of box_rows x 64
// columns (128 bytes), 128-byte swizzle, zero fill outside the matrix.
bool make_tma_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);
// Packed weight blocks (already swizzled in memory) as a [rows, 64] bf16 matrix
// of 128-byte rows; box of box_rows x 64 copied as-is (no swizzle).
bool make_tma_packed(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);


// MOE_OK for cudaSuccess, else records the error for moe_last_cuda_error and
// returns MOE_ERR_CUDA (moe_api.cu).
int cuda_status(cudaError_t e);

// The forward's argument checks and its kernel sequence (moe_api.cu).
int check_forward_args(const void* x, int T, int H, const void* Wr, const void* Wg,
                       const void* Wu, const void* Wd, int E, int K, int I, const void* out,
                       const void* logits, const void* idx, const void* w, const void* aux);
// cap: expert capacity in pairs (0: none).  ev_routed (may be null) is
// recorded on st once logits, idx, w and aux are final (after the dispatch).
int run_forward(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const ExpertWeights& W,
                const Sizes& s, int norm, const float* bias, int cap, __nv_bfloat16* out,
                float* logits, int32_t* idx, float* w, float* aux, const Workspace& ws,
                cudaStream_t st, cudaEvent_t ev_routed = nullptr);

// Every launcher adds the number of kernels it launched.
void count_launches(int n);

// ---- programmatic dependent launch ------------------------------------------
// Every kernel of a forward is launched with programmatic stream serialization:
// it may start while the previous kernel on the stream is still finishing, so
// it must call pdl_wait() before it reads anything an earlier kernel (or the
// caller's earlier work) wrote, and it calls pdl_trigger() early so that the
// next kernel's launch overlaps its own tail.  Dependent CTAs are launched only
// after every CTA of the running grid has triggered or exited.  Because a
// grid's lifetime now overlaps its predecessors', no kernel may use
// non-coherent (ld.global.nc / __ldg) loads: their contract is that the data
// stays unchanged for the whole lifetime of the reading grid.  That is also why
// no kernel pointer is declared __restrict__: with `const T* __restrict__` the
// compiler is free to turn ordinary loads into non-coherent ones.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- small device helpers --------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

}  // namespace moe
