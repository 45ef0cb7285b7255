// dispatch.cu -- expert histogram, prefix sums and the stable permutation of
// the token-expert pairs, plus the load-balance statistic.
//
// Replaces the per-expert loop of Qwen3MoeSparseMoeBlock.forward (cnblogs
// page "大模型-qwen3 MoE 详细解读": one_hot expert mask, torch.where per
// expert, gather of hidden_states[top_x]) by one grouping of all pairs.  The
// commentary on that page names the production form: permute the tokens so
// that those of one expert are contiguous, run all experts, permute back.
//
// Row order: by expert, then by token (unique: a token picks an expert at most
// once).  Integer work only; every result is bit-exact and independent of
// scheduling (shared-memory atomics only count or set bits).
//
//   count   : per 256-token chunk, per expert pair counts
//   scan    : per expert running sums over the chunks, exclusive prefix over
//             experts (offsets, warp-shuffle scan), the row-tile table for the
//             expert kernels,
//             and aux = E · Σ_e (counts_e/(T·K)) · (Σ_t p[t,e] / T) of the csdn
//             page "MoE架构深度解析" (section "负载均衡机制", n · Σ f_i · P_i)
//   scatter : rank of each pair inside its chunk from per-expert token
//             bitmaps -> perm_tok, perm_slot, inv, w_perm
//   gather  : x_perm[row] = x[perm_tok[row]] for the tensor-core expert GEMMs
//             (16-byte vectors); the streaming kernels read x through perm_tok
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kWords = kChunkTokens / 32;

__global__ void __launch_bounds__(kChunkTokens) dispatch_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int K, int32_t* __restrict__ chunk_counts) {
    __shared__ int cnt[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * kChunkTokens + threadIdx.x;
    if (t < T)
        for (int k = 0; k < K; ++k) atomicAdd(&cnt[idx[(size_t)t * K + k]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

// Inclusive prefix sum of v over the CTA's kMaxExperts threads (8 warps).
__device__ __forceinline__ int block_inclusive_scan(int v, int* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    int add = 0;
    for (int j = 0; j < warp; ++j) add += warp_tot[j];
    __syncthreads();
    return v + add;
}

// One CTA of kMaxExperts threads; thread e owns expert e.
//   chunk_base[c,e] = pairs of expert e in chunks before c (within-expert prefix)
//   counts[e], offsets[0..E], the row-tile table and n_tiles, and aux.
__global__ void __launch_bounds__(kMaxExperts) dispatch_scan_kernel(
    const int32_t* __restrict__ chunk_counts, int32_t* __restrict__ chunk_base, int nchunks, int T,
    int E, int K, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    RowTile* __restrict__ tiles, int32_t* __restrict__ n_tiles, int rows_per_tile,
    const float* __restrict__ p_partial, int nrouter, float* __restrict__ aux) {
    __shared__ int warp_tot[kMaxExperts / 32];
    __shared__ float term_s[kMaxExperts];
    const int e = threadIdx.x;
    const bool own = e < E;
    int run = 0;
    if (own) {
        int c = 0;
        for (; c + 4 <= nchunks; c += 4) {
            const int v0 = chunk_counts[(size_t)(c + 0) * E + e];
            const int v1 = chunk_counts[(size_t)(c + 1) * E + e];
            const int v2 = chunk_counts[(size_t)(c + 2) * E + e];
            const int v3 = chunk_counts[(size_t)(c + 3) * E + e];
            chunk_base[(size_t)(c + 0) * E + e] = run;
            chunk_base[(size_t)(c + 1) * E + e] = run + v0;
            chunk_base[(size_t)(c + 2) * E + e] = run + v0 + v1;
            chunk_base[(size_t)(c + 3) * E + e] = run + v0 + v1 + v2;
            run += v0 + v1 + v2 + v3;
        }
        for (; c < nchunks; ++c) {
            const int v = chunk_counts[(size_t)c * E + e];
            chunk_base[(size_t)c * E + e] = run;
            run += v;
        }
        counts[e] = run;
    }
    const int nt = own ? (run + rows_per_tile - 1) / rows_per_tile : 0;
    const int off_incl = block_inclusive_scan(own ? run : 0, warp_tot);
    const int toff_incl = block_inclusive_scan(nt, warp_tot);
    const int base = off_incl - (own ? run : 0);
    const int tbase = toff_incl - nt;
    if (own) {
        offsets[e] = base;
        if (e == E - 1) {
            offsets[E] = off_incl;
            *n_tiles = toff_incl;
        }
        for (int j = 0; j < nt; ++j) {
            RowTile tl;
            tl.expert = e;
            tl.row0 = base + j * rows_per_tile;
            tl.nrows = min(rows_per_tile, run - j * rows_per_tile);
            tl.pad = 0;
            tiles[tbase + j] = tl;
        }
        if (aux) {
            float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
            int b = 0;
            for (; b + 4 <= nrouter; b += 4) {  // four interleaved partial sums, combined in order
                p0 += p_partial[(size_t)(b + 0) * E + e];
                p1 += p_partial[(size_t)(b + 1) * E + e];
                p2 += p_partial[(size_t)(b + 2) * E + e];
                p3 += p_partial[(size_t)(b + 3) * E + e];
            }
            for (; b < nrouter; ++b) p0 += p_partial[(size_t)b * E + e];
            const float psum = (p0 + p1) + (p2 + p3);
            const float f = (float)run / ((float)T * (float)K);
            term_s[e] = f * (psum / (float)T);
        }
    }
    if (aux) {
        __syncthreads();
        if (e < 32) {  // fixed-order reduction over the experts
            float v = 0.f;
            for (int j = e; j < E; j += 32) v += term_s[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (e == 0) *aux = (float)E * v;
        }
    }
}

// Row of each pair: offsets[e] + chunk_base[c,e] + (tokens of this chunk
// before t that chose e), the last from per-expert token bitmaps.
__global__ void __launch_bounds__(kChunkTokens) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int E, int K,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ perm_tok, int32_t* __restrict__ perm_slot, int32_t* __restrict__ inv,
    float* __restrict__ w_perm) {
    __shared__ uint32_t sel[kMaxExperts * kWords];
    __shared__ int base_s[kMaxExperts];
    for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) sel[i] = 0u;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        base_s[e] = offsets[e] + chunk_base[(size_t)blockIdx.x * E + e];
    __syncthreads();
    const int tl = threadIdx.x, word = tl >> 5, bit = tl & 31;
    const int t = blockIdx.x * kChunkTokens + tl;
    int ev[kMaxTopK];
    if (t < T) {
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < K) ev[k] = idx[(size_t)t * K + k];
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < K) atomicOr(&sel[ev[k] * kWords + word], 1u << bit);
    }
    __syncthreads();
    if (t >= T) return;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
        if (k >= K) break;
        const int e = ev[k];
        const uint32_t* sb = sel + e * kWords;
        int rank = __popc(sb[word] & ((1u << bit) - 1u));
        for (int j = 0; j < word; ++j) rank += __popc(sb[j]);
        const int row = base_s[e] + rank;
        perm_tok[row] = t;
        if (perm_slot) perm_slot[row] = k;
        inv[(size_t)t * K + k] = row;
        if (w_perm) w_perm[row] = w[(size_t)t * K + k];
    }
}

// x_perm[row, :] = x[perm_tok[row], :]; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ perm_tok,
                                                          long long P, int vec_per_row,
                                                          uint4* __restrict__ x_perm) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = warp; r < P; r += nwarps) {
        const uint4* src = x + (size_t)perm_tok[r] * vec_per_row;
        uint4* dst = x_perm + (size_t)r * vec_per_row;
        for (int c = lane; c < vec_per_row; c += 32) dst[c] = __ldg(src + c);
    }
}

}  // namespace

cudaError_t launch_dispatch(const int32_t* idx, const float* w, const __nv_bfloat16* x,
                            const Sizes& s, const Workspace& ws, int rows_per_tile,
                            const float* p_partial, int n_partials, float* aux, cudaStream_t st) {
    const int nch = s.nchunks();
    dispatch_count_kernel<<<nch, kChunkTokens, 0, st>>>(idx, s.T, s.E, s.K, ws.chunk_counts);
    dispatch_scan_kernel<<<1, kMaxExperts, 0, st>>>(
        ws.chunk_counts, ws.chunk_base, nch, s.T, s.E, s.K, ws.counts, ws.offsets, ws.tiles,
        ws.n_tiles, rows_per_tile, p_partial, n_partials, aux);
    dispatch_scatter_kernel<<<nch, kChunkTokens, 0, st>>>(idx, w, s.T, s.E, s.K, ws.offsets,
                                                          ws.chunk_base, ws.perm_tok, ws.perm_slot,
                                                          ws.inv, ws.w_perm);
    count_launches(3);
    if (x) {
        const long long P = s.P();
        long long blocks = (P + 7) / 8;
        const long long cap = (long long)num_sms() * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        gather_rows_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(x),
                                                        ws.perm_tok, P, s.H / 8,
                                                        reinterpret_cast<uint4*>(ws.x_perm));
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace moe
