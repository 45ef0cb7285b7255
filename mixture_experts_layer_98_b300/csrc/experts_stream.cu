// experts_stream.cu -- weight-streaming expert MLP kernels (CUDA cores).
//
// The expert is the SwiGLU MLP down(silu(gate(x)) ⊙ up(x)) with per-expert
// gate_proj / up_proj [I,H] and down_proj [H,I] (csdn page
// "MoE架构深度解析：128专家与8激活的智能路由", section
// "128个专家网络的组织结构与参数分布"); its output is scaled by the pair's
// routing weight as in Qwen3MoeSparseMoeBlock.forward (cnblogs page
// "大模型-qwen3 MoE 详细解读": expert_layer(current_state) * routing_weights).
//
// For decode-sized batches each expert sees a handful of rows, so the work is
// bound by reading the touched experts' weights once from HBM.  Each CTA takes
// one row tile (<= kStreamRows rows of one expert, staged in shared memory) and
// a block of weight rows; every weight row is streamed once per row tile with
// 16-byte loads and dotted with all the tile's rows in fp32.
//
//   gate/up : h[r, i]  = bf16( silu(x_r·Wg[e,i]) · (x_r·Wu[e,i]) )
//   down    : Y[t*K + k, n] = bf16( w_r · (h_r·Wd[e,n]) ) for the pair (t, k)
//             of dispatch row r (token-major Y)
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kRowsPerWarp = 2;                     // weight rows per warp per item
constexpr int kWarps = 8;
constexpr int kRowsPerItem = kRowsPerWarp * kWarps;  // 16 weight rows per item

// Streaming 16-byte load of weights: coherent, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
    acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
    acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
    acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
    acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
    acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
    acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
    acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
    acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
    return acc;
}

// Stages rows [row0, row0+nrows) of a [P, D] bf16 matrix into shared memory;
// with perm != null, dispatch row r is row perm[r] of src (a gather from x).
__device__ __forceinline__ void stage_rows(const __nv_bfloat16* src,
                                           const int32_t* perm, int row0, int nrows,
                                           int D, uint4* dst) {
    const int vpr = D / 8;
    const uint4* s = reinterpret_cast<const uint4*>(src);
    for (int i = threadIdx.x; i < nrows * vpr; i += blockDim.x) {
        const int m = i / vpr, c = i % vpr;
        const size_t r = perm ? (size_t)perm[row0 + m] : (size_t)(row0 + m);
        dst[i] = s[r * vpr + c];
    }
}

__global__ void __launch_bounds__(256) gateup_stream_kernel(
    const __nv_bfloat16* x, const int32_t* perm_tok,
    const RowTile* tiles,
    const int32_t* n_tiles_p, const __nv_bfloat16* Wg,
    const __nv_bfloat16* Wu, __nv_bfloat16* h, int H, int I) {
    extern __shared__ uint4 xs[];  // [kStreamRows][H/8]
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int vpr = H / 8;
    const int nblk = I / kRowsPerItem;
    const long long total = (long long)(*n_tiles_p) * nblk;
    for (long long item = blockIdx.x; item < total; item += gridDim.x) {
        const RowTile tl = tiles[item / nblk];
        const int i0 = (int)(item % nblk) * kRowsPerItem + wid * kRowsPerWarp;
        __syncthreads();
        stage_rows(x, perm_tok, tl.row0, tl.nrows, H, xs);
        __syncthreads();
        float g[kRowsPerWarp][kStreamRows], u[kRowsPerWarp][kStreamRows];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int m = 0; m < kStreamRows; ++m) g[r][m] = u[r][m] = 0.f;
        const uint4* wg = reinterpret_cast<const uint4*>(Wg) + ((size_t)tl.expert * I + i0) * vpr;
        const uint4* wu = reinterpret_cast<const uint4*>(Wu) + ((size_t)tl.expert * I + i0) * vpr;
#pragma unroll 2
        for (int c = lane; c < vpr; c += 32) {
            uint4 a[kRowsPerWarp], b[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                a[r] = ldg_stream(wg + (size_t)r * vpr + c);
                b[r] = ldg_stream(wu + (size_t)r * vpr + c);
            }
#pragma unroll
            for (int m = 0; m < kStreamRows; ++m) {
                if (m < tl.nrows) {
                    const uint4 xv = xs[m * vpr + c];
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r) {
                        g[r][m] = dot8(a[r], xv, g[r][m]);
                        u[r][m] = dot8(b[r], xv, u[r][m]);
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kStreamRows; ++m) {
            if (m < tl.nrows) {
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    float gv = g[r][m], uv = u[r][m];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        gv += __shfl_xor_sync(0xffffffffu, gv, off);
                        uv += __shfl_xor_sync(0xffffffffu, uv, off);
                    }
                    if (lane == r)
                        h[(size_t)(tl.row0 + m) * I + i0 + r] = __float2bfloat16_rn(silu_f(gv) * uv);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256) down_stream_kernel(
    const __nv_bfloat16* hbuf, const RowTile* tiles,
    const int32_t* n_tiles_p, const __nv_bfloat16* Wd,
    const float* w_perm, const int32_t* perm_tok, const int32_t* perm_slot, int K,
    __nv_bfloat16* Y, float* Y32, int H, int I) {
    extern __shared__ uint4 hs[];  // [kStreamRows][I/8]
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int vpr = I / 8;
    const int nblk = H / kRowsPerItem;
    const long long total = (long long)(*n_tiles_p) * nblk;
    for (long long item = blockIdx.x; item < total; item += gridDim.x) {
        const RowTile tl = tiles[item / nblk];
        const int n0 = (int)(item % nblk) * kRowsPerItem + wid * kRowsPerWarp;
        __syncthreads();
        stage_rows(hbuf, nullptr, tl.row0, tl.nrows, I, hs);
        __syncthreads();
        float acc[kRowsPerWarp][kStreamRows];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int m = 0; m < kStreamRows; ++m) acc[r][m] = 0.f;
        const uint4* wd = reinterpret_cast<const uint4*>(Wd) + ((size_t)tl.expert * H + n0) * vpr;
#pragma unroll 2
        for (int c = lane; c < vpr; c += 32) {
            uint4 a[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) a[r] = ldg_stream(wd + (size_t)r * vpr + c);
#pragma unroll
            for (int m = 0; m < kStreamRows; ++m) {
                if (m < tl.nrows) {
                    const uint4 hv = hs[m * vpr + c];
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r) acc[r][m] = dot8(a[r], hv, acc[r][m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kStreamRows; ++m) {
            if (m < tl.nrows) {
                const float wr = w_perm[tl.row0 + m];
                const size_t yrow =
                    (size_t)perm_tok[tl.row0 + m] * K + (size_t)perm_slot[tl.row0 + m];
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    float v = acc[r][m];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == r) {
                        if (Y32)  // under a capacity: fp32 Y
                            Y32[yrow * H + n0 + r] = wr * v;
                        else
                            Y[yrow * H + n0 + r] = __float2bfloat16_rn(wr * v);
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_experts_streaming(const __nv_bfloat16* x, const ExpertWeights& W,
                                     const Sizes& s, const Workspace& ws, cudaStream_t st,
                                     cudaEvent_t ev_mid) {
    if (W.packed) return cudaErrorInvalidValue;  // reads row-major weight rows
    const __nv_bfloat16* Wg = W.gate;
    const __nv_bfloat16* Wu = W.up;
    const __nv_bfloat16* Wd = W.down;
    const int sms = num_sms();
    const size_t smem_gu = (size_t)kStreamRows * s.H * 2;
    const size_t smem_dn = (size_t)kStreamRows * s.I * 2;
    cudaError_t err = ensure_smem((const void*)gateup_stream_kernel, (int)smem_gu);
    if (err != cudaSuccess) return err;
    err = ensure_smem((const void*)down_stream_kernel, (int)smem_dn);
    if (err != cudaSuccess) return err;
    // Upper bound on the items; the kernels read the real tile count on the device.
    const long long max_tiles = s.max_tiles(kStreamRows);
    long long items_gu = max_tiles * (s.I / kRowsPerItem);
    long long items_dn = max_tiles * (s.H / kRowsPerItem);
    const long long cap = (long long)sms * 4;
    const int g_gu = (int)(items_gu < cap ? items_gu : cap);
    const int g_dn = (int)(items_dn < cap ? items_dn : cap);
    err = launch_pdl(gateup_stream_kernel, dim3(g_gu), dim3(256), smem_gu, st, x,
                     (const int32_t*)ws.perm_tok, (const RowTile*)ws.tiles,
                     (const int32_t*)ws.n_tiles, Wg, Wu, ws.hbuf, s.H, s.I);
    count_launches(1);
    if (err != cudaSuccess) return err;
    if (ev_mid) cudaEventRecord(ev_mid, st);
    err = launch_pdl(down_stream_kernel, dim3(g_dn), dim3(256), smem_dn, st,
                     (const __nv_bfloat16*)ws.hbuf, (const RowTile*)ws.tiles,
                     (const int32_t*)ws.n_tiles, Wd, (const float*)ws.w_perm,
                     (const int32_t*)ws.perm_tok, (const int32_t*)ws.perm_slot, s.K, ws.ybuf,
                     ws.ybuf_f32, s.H, s.I);
    count_launches(1);
    return err;
}

}  // namespace moe
