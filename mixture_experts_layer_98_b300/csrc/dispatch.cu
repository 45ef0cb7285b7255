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
//             experts (offsets), the row-tile table for the expert kernels,
//             and aux = E · Σ_e (counts_e/(T·K)) · (Σ_t p[t,e] / T) of the csdn
//             page "MoE架构深度解析" (section "负载均衡机制", n · Σ f_i · P_i)
//   scatter : rank of each pair inside its chunk from per-expert token
//             bitmaps -> perm_tok, perm_slot, inv, w_perm
//   gather  : x_perm[row] = x[perm_tok[row]] (16-byte vectors)
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

// One CTA of kMaxExperts threads; thread e owns expert e.
__global__ void __launch_bounds__(kMaxExperts) dispatch_scan_kernel(
    int32_t* __restrict__ chunk_counts, int32_t* __restrict__ chunk_base, int nchunks, int T,
    int E, int K, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    RowTile* __restrict__ tiles, int32_t* __restrict__ n_tiles, int rows_per_tile,
    const float* __restrict__ p_partial, int nrouter, float* __restrict__ aux) {
    __shared__ int cnt_s[kMaxExperts];
    __shared__ int off_s[kMaxExperts + 1];
    __shared__ int toff_s[kMaxExperts + 1];
    __shared__ float term_s[kMaxExperts];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int c = 0; c < nchunks; ++c) {
            const int v = chunk_counts[(size_t)c * E + e];
            chunk_base[(size_t)c * E + e] = run;
            run += v;
        }
        cnt_s[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    if (e == 0) {
        int o = 0, to = 0;
        for (int j = 0; j < E; ++j) {
            off_s[j] = o;
            toff_s[j] = to;
            o += cnt_s[j];
            to += (cnt_s[j] + rows_per_tile - 1) / rows_per_tile;
        }
        off_s[E] = o;
        toff_s[E] = to;
        offsets[E] = o;
        *n_tiles = to;
    }
    __syncthreads();
    if (e < E) {
        const int base = off_s[e];
        offsets[e] = base;
        for (int c = 0; c < nchunks; ++c) chunk_base[(size_t)c * E + e] += base;
        const int nt = toff_s[e + 1] - toff_s[e];
        for (int j = 0; j < nt; ++j) {
            RowTile tl;
            tl.expert = e;
            tl.row0 = base + j * rows_per_tile;
            tl.nrows = min(rows_per_tile, run - j * rows_per_tile);
            tl.pad = 0;
            tiles[toff_s[e] + j] = tl;
        }
        if (aux) {
            float psum = 0.f;
            for (int b = 0; b < nrouter; ++b) psum += p_partial[(size_t)b * E + e];
            const float f = (float)run / ((float)T * (float)K);
            term_s[e] = f * (psum / (float)T);
        }
    }
    __syncthreads();
    if (aux && e == 0) {
        float s = 0.f;
        for (int j = 0; j < E; ++j) s += term_s[j];
        *aux = (float)E * s;
    }
}

__global__ void __launch_bounds__(kChunkTokens) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int E, int K,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_tok,
    int32_t* __restrict__ perm_slot, int32_t* __restrict__ inv, float* __restrict__ w_perm) {
    __shared__ uint32_t sel[kMaxExperts * kWords];
    for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) sel[i] = 0u;
    __syncthreads();
    const int tl = threadIdx.x, word = tl >> 5, bit = tl & 31;
    const int t = blockIdx.x * kChunkTokens + tl;
    if (t < T)
        for (int k = 0; k < K; ++k) atomicOr(&sel[idx[(size_t)t * K + k] * kWords + word], 1u << bit);
    __syncthreads();
    if (t >= T) return;
    for (int k = 0; k < K; ++k) {
        const int e = idx[(size_t)t * K + k];
        const uint32_t* s = sel + e * kWords;
        int rank = __popc(s[word] & ((1u << bit) - 1u));
        for (int j = 0; j < word; ++j) rank += __popc(s[j]);
        const int row = chunk_base[(size_t)blockIdx.x * E + e] + rank;
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
                            bool gather_x, const float* p_partial, float* aux,
                            cudaStream_t st) {
    const int nch = s.nchunks();
    dispatch_count_kernel<<<nch, kChunkTokens, 0, st>>>(idx, s.T, s.E, s.K, ws.chunk_counts);
    dispatch_scan_kernel<<<1, kMaxExperts, 0, st>>>(
        ws.chunk_counts, ws.chunk_base, nch, s.T, s.E, s.K, ws.counts, ws.offsets, ws.tiles,
        ws.n_tiles, rows_per_tile, p_partial, s.nrouter(), aux);
    dispatch_scatter_kernel<<<nch, kChunkTokens, 0, st>>>(idx, w, s.T, s.E, s.K, ws.chunk_base,
                                                          ws.perm_tok, ws.perm_slot, ws.inv,
                                                          ws.w_perm);
    count_launches(3);
    if (gather_x && x) {
        const long long P = s.P();
        const int vpr = s.H / 8;
        long long blocks = (P + 7) / 8;
        const long long cap = (long long)num_sms() * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        gather_rows_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(x),
                                                        ws.perm_tok, P, vpr,
                                                        reinterpret_cast<uint4*>(ws.x_perm));
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace moe
