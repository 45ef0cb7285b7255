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
//             (16-byte vectors; in row order, or token by token through inv once
//             x exceeds 48 MB); the streaming kernels read x through perm_tok
//
// A batch of at most one chunk (256 tokens) runs count, scan and scatter as
// one CTA (dispatch_small_kernel); at most 32 tokens, that CTA also routes
// them (softmax, top-k, renorm from the partial logits) and, up to 128 KB of
// rows, gathers them, so a decode step has one kernel between the router
// logits and the expert GEMMs.  It produces the same rows, tiles and aux bit
// for bit as the chunked kernels.
#include "moe_common.cuh"
#include "routing.cuh"

namespace moe {

namespace {

constexpr int kWords = kChunkTokens / 32;

// Sum of column pe over the rows j, j+4, j+8, ... of p_partial (the routing
// CTAs' per-expert probability sums), in a fixed order: eight running sums
// (row j + 4i goes to sum i mod 8, so eight loads are in flight), added
// pairwise at the end.
__device__ __forceinline__ float psum_rows(const float* p_partial, int nrouter, int E, int pe,
                                           int j) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.f;
    int b = j;
    for (; b + 28 < nrouter; b += 32) {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] += p_partial[(size_t)(b + 4 * i) * E + pe];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (b + 4 * i < nrouter) a[i] += p_partial[(size_t)(b + 4 * i) * E + pe];
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

__global__ void __launch_bounds__(kChunkTokens) dispatch_count_kernel(
    const int32_t* idx, int T, int E, int K, int32_t* chunk_counts) {
    pdl_trigger();
    __shared__ int cnt[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    pdl_wait();
    __syncthreads();
    const int t = blockIdx.x * kChunkTokens + threadIdx.x;
    if (t < T)
        for (int k = 0; k < K; ++k) atomicAdd(&cnt[idx[(size_t)t * K + k]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

// Inclusive prefix sum of v over all threads of the CTA, in thread order
// (warp_tot holds one int per warp).  Every thread must call it.
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

constexpr int kScanThreads = 4 * kMaxExperts;

// One CTA of 4 * kMaxExperts threads.  First, four threads per expert add up
// the routing CTAs' probability sums (rows j, j+4, ... each); then thread e
// (e < E) owns expert e and computes
//   chunk_base[c,e] = pairs of expert e in chunks before c (within-expert prefix)
//   counts[e], offsets[0..E], the row-tile table and n_tiles, and aux.
__global__ void __launch_bounds__(kScanThreads) dispatch_scan_kernel(
    const int32_t* chunk_counts, int32_t* chunk_base, int nchunks, int T,
    int E, int K, int32_t* counts, int32_t* offsets,
    RowTile* tiles, int32_t* n_tiles, int rows_per_tile,
    const float* p_partial, int nrouter, float* aux, int cap) {
    __shared__ int warp_tot[kScanThreads / 32];
    __shared__ float term_s[kMaxExperts];
    __shared__ float psum_s[4][kMaxExperts];
    pdl_trigger();
    pdl_wait();
    if (aux) {
        const int pe = threadIdx.x % kMaxExperts, pj = threadIdx.x / kMaxExperts;
        if (pe < E) psum_s[pj][pe] = psum_rows(p_partial, nrouter, E, pe, pj);
        __syncthreads();
    }
    // threads past kMaxExperts own no expert but still take part in the barriers
    const int e = threadIdx.x;
    const bool own = e < E;
    int run = 0;
    if (own) {
        int c = 0;
        // eight chunks' counts loaded before their bases are stored (the
        // stores may alias the loads as far as the compiler knows)
        for (; c + 8 <= nchunks; c += 8) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = chunk_counts[(size_t)(c + i) * E + e];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                chunk_base[(size_t)(c + i) * E + e] = run;
                run += v[i];
            }
        }
        for (; c < nchunks; ++c) {
            const int v = chunk_counts[(size_t)c * E + e];
            chunk_base[(size_t)c * E + e] = run;
            run += v;
        }
        counts[e] = run;
    }
    // with a capacity, an expert's rows are its first cap pairs (token order)
    const int kept = (cap > 0 && run > cap) ? cap : run;
    const int nt = own ? (kept + rows_per_tile - 1) / rows_per_tile : 0;
    const int off_incl = block_inclusive_scan(own ? kept : 0, warp_tot);
    const int toff_incl = block_inclusive_scan(nt, warp_tot);
    const int base = off_incl - (own ? kept : 0);
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
            tl.nrows = min(rows_per_tile, kept - j * rows_per_tile);
            tl.pad = 0;
            tiles[tbase + j] = tl;
        }
        if (aux) {
            const float psum = ((psum_s[0][e] + psum_s[1][e]) + psum_s[2][e]) + psum_s[3][e];
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

constexpr int kScatterThreads = 1024;

// Rank of each pair within its expert: chunk_base[c,e] + (tokens of this
// chunk before t that chose e), the last from per-expert token bitmaps; its
// row is offsets[e] + rank, or, with a capacity cap > 0 and rank >= cap, none
// (inv = -1: the pair is dropped).  One CTA per chunk; its threads walk the
// chunk's pairs (token-major), so each thread handles about K / 4 pairs.
__global__ void __launch_bounds__(kScatterThreads) dispatch_scatter_kernel(
    const int32_t* idx, const float* w, int T, int E, int K,
    const int32_t* offsets, const int32_t* chunk_base,
    int32_t* perm_tok, int32_t* perm_slot, int32_t* inv,
    float* w_perm, int cap) {
    __shared__ uint32_t sel[kMaxExperts * kWords];
    __shared__ int base_s[kMaxExperts];
    __shared__ int cb_s[kMaxExperts];
    pdl_trigger();
    for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) sel[i] = 0u;
    pdl_wait();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        base_s[e] = offsets[e];
        cb_s[e] = chunk_base[(size_t)blockIdx.x * E + e];
    }
    __syncthreads();
    const int t0 = blockIdx.x * kChunkTokens;
    const int npairs = min(kChunkTokens, T - t0) * K;
    const int32_t* cidx = idx + (size_t)t0 * K;
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
        const int tl = i / K;
        atomicOr(&sel[cidx[i] * kWords + (tl >> 5)], 1u << (tl & 31));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
        const int tl = i / K, k = i - tl * K, word = tl >> 5, bit = tl & 31;
        const int e = cidx[i];
        const uint32_t* sb = sel + e * kWords;
        int rank = cb_s[e] + __popc(sb[word] & ((1u << bit) - 1u));
        for (int j = 0; j < word; ++j) rank += __popc(sb[j]);
        const int t = t0 + tl;
        if (cap > 0 && rank >= cap) {
            inv[(size_t)t * K + k] = -1;
            continue;
        }
        const int row = base_s[e] + rank;
        perm_tok[row] = t;
        if (perm_slot) perm_slot[row] = k;
        inv[(size_t)t * K + k] = row;
        if (w_perm) w_perm[row] = w[(size_t)t * K + k];
    }
}

constexpr int kSmallThreads = 1024;
static_assert(kSmallThreads == kScanThreads, "block_inclusive_scan's warp_tot size");
static_assert(kRouteDispatchTokens <= kSmallThreads / 32, "one warp per routed token");

// One CTA for T <= kChunkTokens (ROUTE: T <= kRouteDispatchTokens):
//   ROUTE: warp t routes token t from the sum of nparts partial logits (in
//          slice order), writing logits_out (may be null), idx, w and its
//          probability row to shared memory;
//   counts per expert and per-expert token bitmaps (shared-memory atomics);
//   thread e < E: counts, offsets, tile table, aux term (probability sums as
//          the chunked path forms them: from the routing rows in token order
//          (ROUTE) or from p_partial's nrouter rows);
//   scatter: row = offsets[e] + tokens before t that chose e.
template <int EPL, bool ROUTE>
__global__ void __launch_bounds__(kSmallThreads) dispatch_small_kernel(
    const float* parts, int nparts, float* logits_out, int norm, const float* bias,
    int32_t* idx, float* w, const float* p_partial, int nrouter, int T, int E, int K,
    int rows_per_tile,
    int32_t* counts, int32_t* offsets, RowTile* tiles, int32_t* n_tiles, int32_t* perm_tok,
    int32_t* perm_slot, int32_t* inv, float* w_perm, float* aux, const uint4* x,
    uint4* x_perm, int vec_per_row, int cap) {
    // ROUTE: probability rows [T][E]; otherwise [4][kMaxExperts] partial sums
    __shared__ float prob_s[kRouteDispatchTokens * kMaxExperts];
    constexpr int kR = ROUTE ? kRouteDispatchTokens * kMaxTopK : 1;
    __shared__ int tok_s[kR];    // ROUTE: token of each row
    __shared__ int idx_s[kR];    // ROUTE: the selections and weights, kept here
    __shared__ float w_s[kR];    //        for the dispatch (also written out)
    constexpr int kW = ROUTE ? 1 : kWords;  // bitmap words per expert (T <= 32 * kW)
    __shared__ uint32_t sel[kMaxExperts * kW];
    __shared__ int cnt[kMaxExperts];
    __shared__ int base_s[kMaxExperts];
    __shared__ float term_s[kMaxExperts];
    __shared__ int warp_tot[kSmallThreads / 32];
    __shared__ int kept_total_s;
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < E * kW; i += blockDim.x) sel[i] = 0u;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    pdl_wait();
    if (ROUTE) {
        if (warp < T) {  // warp-uniform: one warp per token
            const int t = warp;
            float l[EPL];
#pragma unroll
            for (int q = 0; q < EPL; ++q) {
                const int e = lane + 32 * q;
                if (e < E) {
                    // every slice loaded before the first add, summed in slice order
                    float pv[kRouterMaxSplits];
#pragma unroll
                    for (int sl = 0; sl < kRouterMaxSplits; ++sl)
                        pv[sl] = sl < nparts ? parts[((size_t)sl * T + t) * E + e] : 0.f;
                    float v = pv[0];
#pragma unroll
                    for (int sl = 1; sl < kRouterMaxSplits; ++sl)
                        if (sl < nparts) v += pv[sl];
                    l[q] = v;
                    if (logits_out) logits_out[(size_t)t * E + e] = v;
                } else {
                    l[q] = -INFINITY;
                }
            }
            route_token<EPL>(l, E, K, norm, bias, idx_s + t * K, w_s + t * K, prob_s + t * E);
        }
    } else if (aux) {
        // four threads per expert add up rows j, j+4, ... of p_partial
        const int pe = tid % kMaxExperts, pj = tid / kMaxExperts;
        if (pe < E) prob_s[pj * kMaxExperts + pe] = psum_rows(p_partial, nrouter, E, pe, pj);
    }
    __syncthreads();  // routing results visible to the CTA
    const int P = T * K;
    for (int i = tid; i < P; i += blockDim.x) {
        const int t = i / K;
        const int e = ROUTE ? idx_s[i] : idx[i];
        if (ROUTE) {
            idx[i] = e;
            w[i] = w_s[i];
        }
        atomicAdd(&cnt[e], 1);
        atomicOr(&sel[e * kW + (t >> 5)], 1u << (t & 31));
    }
    __syncthreads();
    const int e = tid;
    const bool own = e < E;
    const int run = own ? cnt[e] : 0;
    const int kept = (cap > 0 && run > cap) ? cap : run;  // first cap pairs in token order
    const int nt = own ? (kept + rows_per_tile - 1) / rows_per_tile : 0;
    const int off_incl = block_inclusive_scan(kept, warp_tot);
    const int toff_incl = block_inclusive_scan(nt, warp_tot);
    const int base = off_incl - kept;
    const int tbase = toff_incl - nt;
    if (own) {
        counts[e] = run;
        offsets[e] = base;
        base_s[e] = base;
        if (e == E - 1) {
            offsets[E] = off_incl;
            *n_tiles = toff_incl;
            kept_total_s = off_incl;
        }
        for (int j = 0; j < nt; ++j) {
            RowTile tl;
            tl.expert = e;
            tl.row0 = base + j * rows_per_tile;
            tl.nrows = min(rows_per_tile, kept - j * rows_per_tile);
            tl.pad = 0;
            tiles[tbase + j] = tl;
        }
        if (aux) {
            float psum;
            if (ROUTE) {
                psum = 0.f;
                for (int t = 0; t < T; ++t) psum += prob_s[t * E + e];
            } else {
                psum = ((prob_s[e] + prob_s[kMaxExperts + e]) + prob_s[2 * kMaxExperts + e]) +
                       prob_s[3 * kMaxExperts + e];
            }
            const float f = (float)run / ((float)T * (float)K);
            term_s[e] = f * (psum / (float)T);
        }
    }
    __syncthreads();
    if (aux && tid < 32) {  // fixed-order reduction over the experts
        float v = 0.f;
        for (int j = tid; j < E; j += 32) v += term_s[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (tid == 0) *aux = (float)E * v;
    }
    for (int i = tid; i < P; i += blockDim.x) {
        const int t = i / K, k = i - t * K, word = t >> 5, bit = t & 31;
        const int ex = ROUTE ? idx_s[i] : idx[i];
        const uint32_t* sb = sel + ex * kW;
        int rank = __popc(sb[word] & ((1u << bit) - 1u));
        for (int j = 0; j < word; ++j) rank += __popc(sb[j]);
        if (cap > 0 && rank >= cap) {  // dropped
            inv[i] = -1;
            continue;
        }
        const int row = base_s[ex] + rank;
        perm_tok[row] = t;
        if (perm_slot) perm_slot[row] = k;
        inv[i] = row;
        if (w_perm) w_perm[row] = ROUTE ? w_s[i] : w[i];
        if (ROUTE) tok_s[row] = t;
    }
    if (ROUTE && x) {
        // Small batches gather here: x_perm[row] = x[token of row].  x is the
        // caller's input, finished before the forward's first kernel passed
        // its dependency wait, so the read-only path is allowed.
        __syncthreads();
        // four vectors loaded before any is stored (the stores may alias the
        // loads as far as the compiler knows)
        const int n = kept_total_s * vec_per_row;
        for (int v0 = tid; v0 < n; v0 += 4 * blockDim.x) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = v0 + j * blockDim.x;
                if (i < n) {
                    const int row = i / vec_per_row, c = i - row * vec_per_row;
                    v[j] = __ldg(x + (size_t)tok_s[row] * vec_per_row + c);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = v0 + j * blockDim.x;
                if (i < n) x_perm[i] = v[j];
            }
        }
    }
}

// x_perm[row, :] = x[perm_tok[row], :]; one warp per row, 16-byte vectors.
// A lane loads all its vectors of the row before storing any (the stores may
// alias the loads as far as the compiler knows, so without the batching every
// load would wait for the previous store), keeping up to kGatherVec loads in
// flight per lane.
constexpr int kGatherVec = 8;

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* x,
                                                          const int32_t* perm_tok,
                                                          const int32_t* n_rows_p, long long P,
                                                          int vec_per_row, uint4* x_perm) {
    pdl_trigger();
    pdl_wait();
    // the dispatch's row count (below P when a capacity dropped pairs)
    if (*n_rows_p < P) P = *n_rows_p;
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = warp; r < P; r += nwarps) {
        const uint4* src = x + (size_t)perm_tok[r] * vec_per_row;
        uint4* dst = x_perm + (size_t)r * vec_per_row;
        for (int c0 = 0; c0 < vec_per_row; c0 += 32 * kGatherVec) {
            // x is the caller's input: whatever wrote it finished before the router
            // (the forward's first kernel) passed its dependency wait, long before
            // this grid launched, so it is constant for this grid's whole lifetime
            // and the read-only path is allowed here.
            uint4 v[kGatherVec];
#pragma unroll
            for (int j = 0; j < kGatherVec; ++j) {
                const int c = c0 + j * 32 + lane;
                if (c < vec_per_row) v[j] = __ldg(src + c);
            }
#pragma unroll
            for (int j = 0; j < kGatherVec; ++j) {
                const int c = c0 + j * 32 + lane;
                if (c < vec_per_row) dst[c] = v[j];
            }
        }
    }
}

// The same rows gathered token by token: one warp per token loads x[t] once and
// stores it to the rows inv[t*K + k] of its kept pairs.  Row order reads each
// token's row K times in scattered order -- from DRAM once x exceeds the L2
// (8 GB/s of re-reads per TB/s of writes at K = 8); token order reads x once.
__global__ void __launch_bounds__(256) gather_tokens_kernel(const uint4* x, const int32_t* inv,
                                                            int T, int K, int vec_per_row,
                                                            uint4* x_perm) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long t = warp; t < T; t += nwarps) {
        // lane k holds the row of pair (t, k) (-1: dropped by a capacity)
        const int my_row = lane < K ? inv[(size_t)t * K + lane] : -1;
        const uint4* src = x + (size_t)t * vec_per_row;
        for (int c0 = 0; c0 < vec_per_row; c0 += 32 * kGatherVec) {
            // x is the caller's input, constant for this grid's lifetime (see
            // gather_rows_kernel): the read-only path is allowed
            uint4 v[kGatherVec];
#pragma unroll
            for (int j = 0; j < kGatherVec; ++j) {
                const int c = c0 + j * 32 + lane;
                if (c < vec_per_row) v[j] = __ldg(src + c);
            }
            for (int k = 0; k < K; ++k) {
                const int row = __shfl_sync(0xffffffffu, my_row, k);
                if (row < 0) continue;
                uint4* dst = x_perm + (size_t)row * vec_per_row;
#pragma unroll
                for (int j = 0; j < kGatherVec; ++j) {
                    const int c = c0 + j * 32 + lane;
                    if (c < vec_per_row) dst[c] = v[j];
                }
            }
        }
    }
}

// x above this size gathers in token order (gather_tokens_kernel): beyond
// about half the L2, the row-order re-reads of x start to come from DRAM.
constexpr size_t kTokenOrderGatherBytes = 48ull << 20;

cudaError_t launch_gather(const __nv_bfloat16* x, const Sizes& s, const Workspace& ws,
                          cudaStream_t st) {
    const long long P = s.P();
    if ((size_t)s.T * s.H * 2 > kTokenOrderGatherBytes) {
        long long blocks = ((long long)s.T + 7) / 8;
        const long long cap = (long long)num_sms() * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        cudaError_t e = launch_pdl(gather_tokens_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                                   reinterpret_cast<const uint4*>(x), (const int32_t*)ws.inv,
                                   s.T, s.K, s.H / 8, reinterpret_cast<uint4*>(ws.x_perm));
        count_launches(1);
        return e;
    }
    long long blocks = (P + 7) / 8;
    const long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                               reinterpret_cast<const uint4*>(x), (const int32_t*)ws.perm_tok,
                               (const int32_t*)(ws.offsets + s.E), P, s.H / 8,
                               reinterpret_cast<uint4*>(ws.x_perm));
    count_launches(1);
    return e;
}

template <int EPL>
cudaError_t launch_small(const float* parts, int nparts, float* logits_out, int norm,
                         const float* bias, int32_t* idx, float* w, const Sizes& s,
                         const Workspace& ws, int rows_per_tile, float* aux,
                         const __nv_bfloat16* x, int cap, cudaStream_t st) {
    // one warp per token and one thread per expert; no more warps than that
    // (each one more party to every barrier), at least eight
    int threads = 32 * s.T > s.E ? 32 * s.T : (s.E + 31) / 32 * 32;
    if (threads < 256) threads = 256;
    if (threads > kSmallThreads) threads = kSmallThreads;
    cudaError_t e = launch_pdl(dispatch_small_kernel<EPL, true>, dim3(1), dim3(threads), 0,
                               st, parts, nparts, logits_out, norm, bias, idx, w,
                               (const float*)nullptr,
                               0, s.T, s.E, s.K, rows_per_tile, ws.counts, ws.offsets, ws.tiles,
                               ws.n_tiles, ws.perm_tok, ws.perm_slot, ws.inv, ws.w_perm, aux,
                               reinterpret_cast<const uint4*>(x),
                               reinterpret_cast<uint4*>(ws.x_perm), s.H / 8, cap);
    count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_dispatch(const int32_t* idx, const float* w, const __nv_bfloat16* x,
                            const Sizes& s, const Workspace& ws, int rows_per_tile,
                            const float* p_partial, int n_partials, float* aux, int cap,
                            cudaStream_t st) {
    const int nch = s.nchunks();
    cudaError_t e;
    if (nch == 1) {
        e = launch_pdl(dispatch_small_kernel<1, false>, dim3(1), dim3(kSmallThreads), 0, st,
                       (const float*)nullptr, 0, (float*)nullptr, 0, (const float*)nullptr,
                       const_cast<int32_t*>(idx),
                       const_cast<float*>(w), p_partial, n_partials, s.T, s.E, s.K,
                       rows_per_tile, ws.counts, ws.offsets, ws.tiles, ws.n_tiles, ws.perm_tok,
                       ws.perm_slot, ws.inv, ws.w_perm, aux, (const uint4*)nullptr,
                       (uint4*)nullptr, 0, cap);
        count_launches(1);
    } else {
        e = launch_pdl(dispatch_count_kernel, dim3(nch), dim3(kChunkTokens), 0, st, idx, s.T, s.E,
                       s.K, ws.chunk_counts);
        if (e != cudaSuccess) return e;
        e = launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kScanThreads), 0, st,
            ws.chunk_counts, ws.chunk_base, nch, s.T, s.E, s.K, ws.counts, ws.offsets, ws.tiles,
            ws.n_tiles, rows_per_tile, p_partial, n_partials, aux, cap);
        if (e != cudaSuccess) return e;
        e = launch_pdl(dispatch_scatter_kernel, dim3(nch), dim3(kScatterThreads), 0, st, idx, w,
                       s.T, s.E, s.K, (const int32_t*)ws.offsets, (const int32_t*)ws.chunk_base,
                       ws.perm_tok, ws.perm_slot, ws.inv, ws.w_perm, cap);
        count_launches(3);
    }
    if (e != cudaSuccess) return e;
    return x ? launch_gather(x, s, ws, st) : cudaSuccess;
}

cudaError_t launch_route_dispatch_small(const float* parts, int nparts, float* logits_out,
                                        int norm, const float* bias, int32_t* idx, float* w,
                                        const __nv_bfloat16* x, const Sizes& s,
                                        const Workspace& ws, int rows_per_tile, float* aux,
                                        int cap, cudaStream_t st) {
    if (s.T > kRouteDispatchTokens || nparts < 1 || nparts > kRouterMaxSplits)
        return cudaErrorInvalidValue;
    // Up to 128 KB of gathered rows are copied by the routing CTA itself (one
    // or two decode tokens); more go to the gather kernel, which spreads them
    // over the SMs.
    const bool in_cta = x && s.P() * s.H * 2 <= (128 << 10);
    const __nv_bfloat16* xk = in_cta ? x : nullptr;
    const int epl = (s.E + 31) / 32;
    cudaError_t e;
    if (epl <= 1) e = launch_small<1>(parts, nparts, logits_out, norm, bias, idx, w, s, ws, rows_per_tile, aux, xk, cap, st);
    else if (epl <= 2) e = launch_small<2>(parts, nparts, logits_out, norm, bias, idx, w, s, ws, rows_per_tile, aux, xk, cap, st);
    else if (epl <= 4) e = launch_small<4>(parts, nparts, logits_out, norm, bias, idx, w, s, ws, rows_per_tile, aux, xk, cap, st);
    else e = launch_small<8>(parts, nparts, logits_out, norm, bias, idx, w, s, ws, rows_per_tile, aux, xk, cap, st);
    if (e != cudaSuccess) return e;
    return x && !in_cta ? launch_gather(x, s, ws, st) : cudaSuccess;
}

}  // namespace moe
