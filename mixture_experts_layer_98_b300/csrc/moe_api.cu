// moe_api.cu -- the C ABI: argument checks, workspace, and the stream-ordered
// sequence of kernels for one forward of the sparse MoE block.
//
//   router (logits, softmax, top-k, renorm, probability sums)
//   -> dispatch (counts, offsets, permutation, row tiles, aux, row gather)
//   -> expert MLPs (tcgen05 grouped GEMMs, or weight streaming for small batches)
//   -> combine (gather-reduce into token order)
//
// No host synchronisation: the expert kernels read the tile count on the device.
#include <atomic>
#include <cmath>
#include <mutex>
#include <unordered_map>

#include "moe_common.cuh"

namespace moe {

static thread_local int g_last_cuda_error = 0;
static int g_expert_path = MOE_PATH_AUTO;
static std::atomic<long long> g_launches{0};

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Stage-boundary events (benchmark instrumentation), MOE_NUM_STAGES + 1 of them.
static bool g_timing = false;
static bool g_timed_once = false;
static cudaEvent_t g_ev[MOE_NUM_STAGES + 1] = {};

static cudaEvent_t g_next_ev[MOE_NUM_STAGES + 1] = {};
static bool g_next_set = false;
static thread_local cudaEvent_t t_cur_ev[MOE_NUM_STAGES + 1] = {};  // events of this forward

// Records the stage-boundary event `boundary` of the current forward, if any.
static void mark(int boundary, cudaStream_t st) {
    if (t_cur_ev[boundary]) cudaEventRecord(t_cur_ev[boundary], st);
}

// Picks the events this forward records: a one-shot caller set, else the
// library's own set when stage timing is on, else none.
static void begin_marks() {
    if (g_next_set) {
        for (int i = 0; i <= MOE_NUM_STAGES; ++i) t_cur_ev[i] = g_next_ev[i];
        g_next_set = false;
    } else {
        for (int i = 0; i <= MOE_NUM_STAGES; ++i) t_cur_ev[i] = g_timing ? g_ev[i] : nullptr;
    }
}

static std::mutex g_attr_mu;

int num_sms() {
    static int cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n < 1) n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

cudaError_t ensure_smem(const void* func, int bytes) {
    static std::unordered_map<unsigned long long, int> done;  // (device, func) -> bytes set
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long key = (unsigned long long)(uintptr_t)func * 64ull + (unsigned)dev;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t layout_workspace(const Sizes& s, char* base, Workspace* ws, bool y_f32) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        char* p = base ? base + off : nullptr;
        off = align_up(off + bytes, 256);
        return p;
    };
    const size_t P = (size_t)s.P();
    const size_t nch = (size_t)s.nchunks();
    Workspace w{};
    w.chunk_counts = (int32_t*)take(nch * s.E * 4);
    w.chunk_base = (int32_t*)take(nch * s.E * 4);
    w.counts = (int32_t*)take((size_t)s.E * 4);
    w.offsets = (int32_t*)take(((size_t)s.E + 1) * 4);
    w.tiles = (RowTile*)take((size_t)s.max_tiles(kStreamRows) * sizeof(RowTile));
    w.n_tiles = (int32_t*)take(4);
    // split-K regions: the weights-as-M plan's or the 4-bit warp-MMA plan's,
    // whichever needs more (a forward runs one of them)
    const WtPlan plan = wt_plan(s);
    const Q4MmaPlan qplan = q4mma_plan(s);
    w.n_clear = 4 + (plan.n_counters > qplan.n_counters ? plan.n_counters : qplan.n_counters);
    w.status = (int32_t*)take((size_t)w.n_clear * 4);
    w.wt_partial = (float*)take(
        (plan.partial_floats > qplan.partial_floats ? plan.partial_floats : qplan.partial_floats) * 4);
    w.p_partial = (float*)take((size_t)s.nrouter() * s.E * 4);
    w.perm_tok = (int32_t*)take(P * 4);
    w.perm_slot = (int32_t*)take(P * 4);
    w.inv = (int32_t*)take(P * 4);
    w.w_perm = (float*)take(P * 4);
    w.logit_parts = (float*)take((size_t)kRouterMaxSplits * s.T * s.E * 4);
    w.topk_idx = (int32_t*)take(P * 4);
    w.topk_w = (float*)take(P * 4);
    w.x_perm = (__nv_bfloat16*)take(P * s.H * 2);
    w.hbuf = (__nv_bfloat16*)take(P * s.I * 2);
    // Y last and unpadded, so that the fp32 form needs exactly P·H·2 bytes more
    w.ybuf = (__nv_bfloat16*)(base ? base + off : nullptr);
    w.ybuf_f32 = y_f32 ? (float*)w.ybuf : nullptr;
    off += P * s.H * (y_f32 ? 4 : 2);
    w.bytes = off;
    if (ws) *ws = w;
    return off;
}

static int check_sizes(int T, int H, int E, int K, int I) {
    if (T < 0 || H < 64 || H % 64 || I < 64 || I % 64) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > kMaxExperts || K < 1 || K > E || K > kMaxTopK) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K > (1LL << 31) - 1) return MOE_ERR_INVALID_ARG;
    if (H > 65536 || I > 65536) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

static bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

static int check_device() {
    static std::mutex mu;
    static std::unordered_map<int, int> ok;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return MOE_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = ok.find(dev);
    if (it == ok.end()) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        it = ok.emplace(dev, (major == 10 && minor == 3) ? 1 : 0).first;
    }
    return it->second ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    g_last_cuda_error = (int)e;
    return MOE_ERR_CUDA;
}

// ---- library-owned workspaces, one per (device, stream) ---------------------
struct OwnedWs {
    void* ptr = nullptr;
    size_t bytes = 0;
    int32_t* counts = nullptr;  // counts of the last forward on this stream
    int32_t* status = nullptr;  // status word of the last forward on this stream
    int E = 0;
};
static std::mutex g_ws_mu;
static std::unordered_map<unsigned long long, OwnedWs> g_ws;

// slot 0: the forwards' workspace (whose counts and status the query calls
// read); slot 1: the stage entry points' private scratch, so that a stage call
// never overwrites what the last forward left for those queries
static unsigned long long ws_key(cudaStream_t st, int slot = 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    return (((unsigned long long)(uintptr_t)st) * 64ull + (unsigned long long)dev) * 2ull +
           (unsigned long long)slot;
}

// Returns a workspace of at least `bytes` for `st` (grown with stream-ordered
// allocation, so earlier work on the stream finishes with the old buffer first).
static int owned_workspace(cudaStream_t st, size_t bytes, void** out, int slot = 0) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    OwnedWs& w = g_ws[ws_key(st, slot)];
    if (w.bytes < bytes) {
        if (w.ptr) {
            cudaError_t e = cudaFreeAsync(w.ptr, st);
            if (e != cudaSuccess) return cuda_status(e);
            w.ptr = nullptr;
            w.bytes = 0;
            w.counts = nullptr;
            w.status = nullptr;
        }
        size_t want = align_up(bytes + bytes / 8, 1 << 20);
        cudaError_t e = cudaMallocAsync(&w.ptr, want, st);
        if (e != cudaSuccess) {
            g_last_cuda_error = (int)e;
            w.ptr = nullptr;
            return MOE_ERR_WORKSPACE;
        }
        w.bytes = want;
    }
    *out = w.ptr;
    return MOE_OK;
}

static void remember_counts(cudaStream_t st, const Workspace& ws, int E) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    OwnedWs& w = g_ws[ws_key(st)];
    w.counts = ws.counts;
    w.status = ws.status;
    w.E = E;
}

enum class ExpertPath { kStreaming, kTokensM, kTokensPair, kWeightsM, kDecodeFused, kWeightsQ4 };

static ExpertPath expert_path(const Sizes& s, bool packed) {
    const bool wt_ok = experts_wt_supported(s);
    // Packed weights exist only for shapes both tensor-core paths tile; the
    // streaming kernels read row-major rows, so packed forwards never use them.
    const ExpertPath small = (wt_ok || packed) ? ExpertPath::kWeightsM : ExpertPath::kStreaming;
    // decode batches: the weights-as-M units and the combine in one kernel --
    // forced up to kDecodeFusedTokens tokens; AUTO up to kDecodeAutoTokens, where
    // it measured faster (4 tokens -6 %, 16 tokens -1.5 %, 64 tokens +6 %)
    const ExpertPath small_fused =
        small == ExpertPath::kWeightsM && experts_decode_supported(s) ? ExpertPath::kDecodeFused
                                                                      : small;
    const ExpertPath small_auto = s.T <= kDecodeAutoTokens ? small_fused : small;
    switch (g_expert_path) {
        case MOE_PATH_STREAMING: return packed ? ExpertPath::kWeightsM : ExpertPath::kStreaming;
        case MOE_PATH_TCGEN05: return ExpertPath::kTokensM;
        case MOE_PATH_TCGEN05_WT: return small;
        case MOE_PATH_TCGEN05_PAIR:
            return experts_pair_supported(s) ? ExpertPath::kTokensPair : ExpertPath::kTokensM;
        case MOE_PATH_TCGEN05_DECODE: return small_fused;
        case MOE_PATH_WARP_MMA: break;  // 4-bit experts only; bf16 weights: AUTO
        default: break;
    }
    // Token rows fill 128-row tiles from ~32 rows per expert on average up;
    // below that the weights go on the MMA's M side (every stage is weights).
    // CTA pairs (256-row tiles) where few experts each receive >= 1024 rows:
    // there an expert's ragged last tile adds little padding (measured faster
    // at E=8, 1024 rows per expert); with 128 experts of 256-1024 rows the
    // single-CTA tiles (128 rows, 64-row tails) pad less and measured faster.
    if (s.P() >= 32LL * s.E) {
        if (experts_pair_supported(s) && s.E <= 32 && s.P() >= 1024LL * s.E)
            return ExpertPath::kTokensPair;
        return ExpertPath::kTokensM;
    }
    return small_auto;
}

// The kernel sequence.  All pointers checked by the caller.
int run_forward(const __nv_bfloat16* x, const __nv_bfloat16* Wr, const ExpertWeights& W,
                const Sizes& s, int norm, const float* bias, int cap, __nv_bfloat16* out,
                float* logits, int32_t* idx, float* w, float* aux, const Workspace& ws,
                cudaStream_t st, cudaEvent_t ev_routed) {
    if (!idx) idx = ws.topk_idx;
    if (!w) w = ws.topk_w;
    // 4-bit experts always run their own kernels (tokens as M, weights
    // dequantised in shared memory); otherwise the path by batch size and setting
    const ExpertPath path = W.q4 ? ExpertPath::kWeightsQ4 : expert_path(s, W.packed != nullptr);
    // 4-bit experts: decode batches on the warp-MMA kernels, larger batches on
    // the tcgen05 kernels
    const bool q4_mma = path == ExpertPath::kWeightsQ4 &&
                        (g_expert_path == MOE_PATH_WARP_MMA ||
                         (g_expert_path != MOE_PATH_TCGEN05 && s.T <= kQ4MmaTokens));
    // The streaming kernels stage kStreamRows rows of H (gate/up) and of I
    // (down) in shared memory; larger layers go to the tensor-core paths.
    if (path == ExpertPath::kStreaming &&
        ((long long)kStreamRows * s.H * 2 > 200 * 1024 ||
         (long long)kStreamRows * s.I * 2 > 200 * 1024))
        return MOE_ERR_INVALID_ARG;
    begin_marks();
    mark(0, st);
    const int tile_rows = path == ExpertPath::kTokensM      ? kTcRows
                          : path == ExpertPath::kTokensPair ? kPairRows
                          : path == ExpertPath::kWeightsM   ? kWtRows
                          : path == ExpertPath::kDecodeFused ? kWtRows
                          : path == ExpertPath::kWeightsQ4  ? (q4_mma ? kQ4MmaRows : kWtRows)
                                                            : kStreamRows;
    // The tensor-core expert paths read gathered rows (x_perm); streaming reads
    // x, and so does the fused decode kernel up to kDecodeDirectTokens tokens.
    const bool x_direct = path == ExpertPath::kStreaming ||
                          (path == ExpertPath::kDecodeFused && s.T <= kDecodeDirectTokens);
    const __nv_bfloat16* gather_x = x_direct ? nullptr : x;
    // Router logits: tensor cores from one full 128-token tile up (E <= 128),
    // else the CUDA-core kernel split over H.  Then routing and dispatch: one
    // CTA for at most 32 tokens, else the routing kernel and the dispatch
    // kernels.
    const bool router_tc = s.T >= 128 && router_tc_supported(s);
    const int n_partials = s.nrouter();
    // Up to kDecodeRouteTokens tokens on the fused decode kernel, that kernel
    // routes and dispatches the batch itself, straight after the router logits.
    const bool route_in_experts = path == ExpertPath::kDecodeFused &&
                                  s.T <= kDecodeRouteTokens && s.K <= kMaxTopK &&
                                  s.E <= kMaxExperts && !router_tc;
    DecodeRouting droute{};
    cudaError_t e;
    if (router_tc) {
        const int nsplit = router_tc_splits(s);
        e = launch_router_tc(x, Wr, s, nsplit, ws.logit_parts, ws.status, ws.n_clear, st);
        if (e == cudaSuccess)
            e = launch_route_from_logits(ws.logit_parts, nsplit, logits, s, norm, bias, idx, w,
                                         ws.p_partial, st);
        if (e != cudaSuccess) return cuda_status(e);
        mark(1, st);
        e = launch_dispatch(idx, w, gather_x, s, ws, tile_rows, ws.p_partial, n_partials, aux, cap,
                            st);
    } else if (s.T <= kRouteDispatchTokens) {
        const int nsplit = router_simt_splits(s);
        e = launch_router_logits(x, Wr, s, nsplit, ws.logit_parts, ws.status, ws.n_clear, st);
        if (e != cudaSuccess) return cuda_status(e);
        mark(1, st);
        if (route_in_experts)
            droute = DecodeRouting{ws.logit_parts, nsplit, logits, norm, bias, idx, w, aux, cap};
        else
            e = launch_route_dispatch_small(ws.logit_parts, nsplit, logits, norm, bias, idx, w,
                                            gather_x, s, ws, tile_rows, aux, cap, st);
    } else {
        e = launch_router(x, Wr, s, norm, bias, logits, ws.logit_parts, idx, w, ws.p_partial,
                          ws.status,
                          ws.n_clear, st);
        if (e != cudaSuccess) return cuda_status(e);
        mark(1, st);
        e = launch_dispatch(idx, w, gather_x, s, ws, tile_rows, ws.p_partial, n_partials, aux, cap,
                            st);
    }
    if (e != cudaSuccess) return cuda_status(e);
    mark(2, st);
    if (ev_routed && !route_in_experts) {
        e = cudaEventRecord(ev_routed, st);
        if (e != cudaSuccess) return cuda_status(e);
    }
    cudaEvent_t mid = t_cur_ev[3];
    switch (path) {
        case ExpertPath::kTokensM: e = launch_experts_tcgen05(W, s, ws, st, mid); break;
        case ExpertPath::kTokensPair: e = launch_experts_pair(W, s, ws, st, mid); break;
        case ExpertPath::kWeightsM: e = launch_experts_wt(W, s, ws, st, mid); break;
        case ExpertPath::kWeightsQ4:
            e = q4_mma ? launch_experts_q4_mma(W.q4, s, ws, st, mid)
                       : launch_experts_q4(W.q4, s, ws, st, mid);
            break;
        case ExpertPath::kDecodeFused: {
            // experts and combine in one kernel: the whole kernel is timed as the
            // gate/up stage; the down and combine stages read zero
            e = launch_experts_decode(W, s, ws, x, cap > 0 ? ws.inv : nullptr, out, st,
                                      route_in_experts ? &droute : nullptr);
            if (e != cudaSuccess) return cuda_status(e);
            // with the routing in the kernel, its outputs are final only now
            if (ev_routed && route_in_experts) {
                e = cudaEventRecord(ev_routed, st);
                if (e != cudaSuccess) return cuda_status(e);
            }
            if (mid) cudaEventRecord(mid, st);
            mark(4, st);
            mark(5, st);
            if (g_timing) g_timed_once = true;
            return MOE_OK;
        }
        default: e = launch_experts_streaming(x, W, s, ws, st, mid); break;
    }
    if (e != cudaSuccess) return cuda_status(e);
    mark(4, st);
    // Y is token-major; with a capacity, inv marks the dropped pairs
    e = launch_combine(ws.ybuf, ws.ybuf_f32, cap > 0 ? ws.inv : nullptr, false, s.T, s.K, s.H,
                       out, st);
    if (e != cudaSuccess) return cuda_status(e);
    mark(5, st);
    if (g_timing) g_timed_once = true;
    return MOE_OK;
}

int check_forward_args(const void* x, int T, int H, const void* Wr, const void* Wg,
                              const void* Wu, const void* Wd, int E, int K, int I, const void* out,
                              const void* logits, const void* idx, const void* w,
                              const void* aux) {
    int rc = check_sizes(T, H, E, K, I);
    if (rc) return rc;
    if (!Wr || !Wg || !Wu || !Wd) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !out)) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {x, Wr, Wg, Wu, Wd, out, logits, idx, w};
    for (const void* p : ps)
        if (misaligned(p)) return MOE_ERR_ALIGNMENT;
    if (aux && (reinterpret_cast<uintptr_t>(aux) & 3u)) return MOE_ERR_ALIGNMENT;
    return check_device();
}

}  // namespace moe

using namespace moe;

// The device-pointer forward behind moe_forward, moe_forward_ws and
// moe_forward_packed: argument checks, T = 0, workspace (library-owned when
// workspace == NULL), kernel sequence.  wg/wu/wd are only null-checked.
static int forward_device(const void* x, int T, int H, const void* W_router,
                          const ExpertWeights& W, const void* wg, const void* wu, const void* wd,
                          int E, int K, int I, int norm, const float* bias, int cap, void* out,
                          float* logits, int32_t* idx, float* w, float* aux, void* workspace,
                          size_t workspace_bytes, cudaStream_t st) {
    int rc = check_forward_args(x, T, H, W_router, wg, wu, wd, E, K, I, out, logits, idx, w, aux);
    if (rc) return rc;
    if (misaligned(bias)) return MOE_ERR_ALIGNMENT;
    if (T == 0) {
        if (aux) return cuda_status(cudaMemsetAsync(aux, 0, sizeof(float), st));
        return MOE_OK;
    }
    Sizes s{T, H, E, K, I};
    // under a capacity the weighted expert outputs stay fp32 until the combine
    const bool y_f32 = cap > 0;
    const size_t need = layout_workspace(s, nullptr, nullptr, y_f32);
    const bool owned = workspace == nullptr;
    if (owned) {
        rc = owned_workspace(st, need, &workspace);
        if (rc) return rc;
    } else {
        if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MOE_ERR_ALIGNMENT;
    }
    Workspace ws;
    layout_workspace(s, (char*)workspace, &ws, y_f32);
    rc = run_forward((const __nv_bfloat16*)x, (const __nv_bfloat16*)W_router, W, s, norm, bias,
                     cap, (__nv_bfloat16*)out, logits, idx, w, aux, ws, st);
    if (rc == MOE_OK && owned) remember_counts(st, ws, E);
    return rc;
}

// A second stream per (device, stream) for the host forward's early copies,
// and the event after the routing that they wait on (created once, kept).
struct SideStream {
    cudaStream_t side = nullptr;
    cudaEvent_t routed = nullptr;
};
static std::mutex g_side_mu;
static std::unordered_map<unsigned long long, SideStream> g_side;

static int side_stream(cudaStream_t st, SideStream* out) {
    std::lock_guard<std::mutex> lk(g_side_mu);
    SideStream& s = g_side[ws_key(st)];
    if (!s.side) {
        cudaError_t e = cudaStreamCreateWithFlags(&s.side, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.routed, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            s.side = nullptr;
            return cuda_status(e);
        }
    }
    *out = s;
    return MOE_OK;
}

// The host-pointer forward behind moe_forward_host and moe_forward_host_packed:
// x is copied in, the forward runs on library-owned scratch, the outputs are
// copied back, and the call returns after the stream has finished them.  The
// routing outputs (logits, top-k, aux) are final after the dispatch: they are
// copied back on a side stream while the expert kernels still run, so only the
// copy of `out` follows the last kernel.  (A decode batch that the fused kernel
// routes itself has them final only when that kernel ends; the side copies
// then follow it, beside the copy of `out`.)
static int forward_host(const void* x_host, int T, int H, const void* W_router,
                        const ExpertWeights& W, const void* wg, const void* wu, const void* wd,
                        int E, int K, int I, int norm, const float* bias, int cap,
                        void* out_host, float* logits_host, int32_t* idx_host, float* w_host,
                        float* aux_host, cudaStream_t st) {
    int rc = check_sizes(T, H, E, K, I);
    if (rc) return rc;
    if (!W_router || !wg || !wu || !wd) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x_host || !out_host)) return MOE_ERR_INVALID_ARG;
    const void* dps[] = {W_router, wg, wu, wd, bias};
    for (const void* p : dps)
        if (misaligned(p)) return MOE_ERR_ALIGNMENT;
    rc = check_device();
    if (rc) return rc;
    if (T == 0) {
        if (aux_host) *aux_host = 0.f;
        return MOE_OK;
    }
    Sizes s{T, H, E, K, I};
    const bool y_f32 = cap > 0;
    const size_t need = layout_workspace(s, nullptr, nullptr, y_f32);
    const size_t xb = (size_t)T * H * 2, lb = (size_t)T * E * 4, kb = (size_t)T * K * 4;
    const size_t stage = align_up(xb, 256) * 2 + align_up(lb, 256) + align_up(kb, 256) * 2 + 256;
    void* base = nullptr;
    rc = owned_workspace(st, need + stage, &base);
    if (rc) return rc;
    Workspace ws;
    layout_workspace(s, (char*)base, &ws, y_f32);
    char* p = (char*)base + align_up(need, 256);  // the +256 of `stage` covers the padding
    __nv_bfloat16* x_d = (__nv_bfloat16*)p;
    p += align_up(xb, 256);
    __nv_bfloat16* out_d = (__nv_bfloat16*)p;
    p += align_up(xb, 256);
    float* logits_d = (float*)p;
    p += align_up(lb, 256);
    int32_t* idx_d = (int32_t*)p;
    p += align_up(kb, 256);
    float* w_d = (float*)p;
    p += align_up(kb, 256);
    float* aux_d = (float*)p;
    SideStream side;
    rc = side_stream(st, &side);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(x_d, x_host, xb, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_status(e);
    rc = run_forward(x_d, (const __nv_bfloat16*)W_router, W, s, norm, bias, cap, out_d,
                     logits_host ? logits_d : nullptr, idx_d, w_d, aux_host ? aux_d : nullptr, ws,
                     st, side.routed);
    if (rc) {
        cudaStreamSynchronize(st);  // nothing of this call left in flight
        return rc;
    }
    remember_counts(st, ws, E);
    // the routing outputs on the side stream, behind the routing
    e = cudaStreamWaitEvent(side.side, side.routed, 0);
    if (e == cudaSuccess && logits_host)
        e = cudaMemcpyAsync(logits_host, logits_d, lb, cudaMemcpyDeviceToHost, side.side);
    if (e == cudaSuccess && idx_host)
        e = cudaMemcpyAsync(idx_host, idx_d, kb, cudaMemcpyDeviceToHost, side.side);
    if (e == cudaSuccess && w_host)
        e = cudaMemcpyAsync(w_host, w_d, kb, cudaMemcpyDeviceToHost, side.side);
    if (e == cudaSuccess && aux_host)
        e = cudaMemcpyAsync(aux_host, aux_d, sizeof(float), cudaMemcpyDeviceToHost, side.side);
    cudaError_t e2 = cudaMemcpyAsync(out_host, out_d, xb, cudaMemcpyDeviceToHost, st);
    // both streams finish before the call returns (and before the next call
    // on st can reuse the staging the side copies read)
    cudaError_t e3 = cudaStreamSynchronize(side.side);
    cudaError_t e4 = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = e3;
    if (e == cudaSuccess) e = e4;
    return cuda_status(e);
}

extern "C" {

const char* moe_strerror(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument (size out of range or NULL pointer)";
        case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case MOE_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (B300)";
        case MOE_ERR_WORKSPACE: return "workspace too small or could not be allocated";
        case MOE_ERR_CUDA: return "CUDA error (see moe_last_cuda_error)";
        case MOE_ERR_TIMEOUT: return "a bounded device-side wait timed out";
        default: return "unknown status";
    }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

long long moe_kernel_launch_count(void) { return g_launches.load(); }

int moe_set_stage_timing(int enable) {
    if (enable && !g_ev[0]) {
        for (int i = 0; i <= MOE_NUM_STAGES; ++i) {
            cudaError_t e = cudaEventCreate(&g_ev[i]);
            if (e != cudaSuccess) return cuda_status(e);
        }
    }
    g_timing = enable != 0;
    return MOE_OK;
}

int moe_set_next_stage_events(void* const* events) {
    if (!events) {
        g_next_set = false;
        return MOE_OK;
    }
    for (int i = 0; i <= MOE_NUM_STAGES; ++i) {
        if (!events[i]) return MOE_ERR_INVALID_ARG;
        g_next_ev[i] = (cudaEvent_t)events[i];
    }
    g_next_set = true;
    return MOE_OK;
}

int moe_stage_times(float* ms, int n) {
    if (!ms || n < 1 || n > MOE_NUM_STAGES || !g_timed_once) return MOE_ERR_INVALID_ARG;
    cudaError_t e = cudaEventSynchronize(g_ev[MOE_NUM_STAGES]);
    if (e != cudaSuccess) return cuda_status(e);
    for (int i = 0; i < n; ++i) {
        e = cudaEventElapsedTime(&ms[i], g_ev[i], g_ev[i + 1]);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return MOE_OK;
}

int moe_set_expert_path(int path) {
    if (path < MOE_PATH_AUTO || path > MOE_PATH_WARP_MMA) return -1;
    const int prev = g_expert_path;
    g_expert_path = path;
    return prev;
}

size_t moe_workspace_bytes(int T, int H, int E, int K, int I) {
    if (check_sizes(T, H, E, K, I)) return 0;
    Sizes s{T, H, E, K, I};
    // enough for every forward of these sizes, including those under a
    // capacity (fp32 expert outputs)
    return layout_workspace(s, nullptr, nullptr, true);
}

int moe_forward_ws(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                   const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down, int E,
                   int K, int I, int norm_topk_prob, moe_bf16* out, float* router_logits,
                   int32_t* topk_idx, float* topk_w, float* aux, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (!workspace) return MOE_ERR_WORKSPACE;
    const ExpertWeights W{(const __nv_bfloat16*)W_gate, (const __nv_bfloat16*)W_up,
                          (const __nv_bfloat16*)W_down, nullptr};
    return forward_device(x, T, H, W_router, W, W_gate, W_up, W_down, E, K, I, norm_topk_prob,
                          nullptr, 0, out, router_logits, topk_idx, topk_w, aux, workspace,
                          workspace_bytes, (cudaStream_t)stream);
}

int moe_forward(const moe_bf16* x, int T, int H, const moe_bf16* W_router, const moe_bf16* W_gate,
                const moe_bf16* W_up, const moe_bf16* W_down, int E, int K, int I,
                int norm_topk_prob, moe_bf16* out, float* router_logits, int32_t* topk_idx,
                float* topk_w, float* aux, void* stream) {
    const ExpertWeights W{(const __nv_bfloat16*)W_gate, (const __nv_bfloat16*)W_up,
                          (const __nv_bfloat16*)W_down, nullptr};
    return forward_device(x, T, H, W_router, W, W_gate, W_up, W_down, E, K, I, norm_topk_prob,
                          nullptr, 0, out, router_logits, topk_idx, topk_w, aux, nullptr, 0,
                          (cudaStream_t)stream);
}

size_t moe_packed_experts_bytes(int H, int E, int I) {
    if (H < 64 || H % 64 || I < 64 || I % 64 || E < 1 || E > kMaxExperts) return 0;
    if (!packed_supported(H, E, I)) return 0;
    return 3 * packed_matrix_bytes(H, E, I);
}

int moe_pack_experts(const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down, int H,
                     int E, int I, void* packed, void* stream) {
    if (!moe_packed_experts_bytes(H, E, I)) return MOE_ERR_INVALID_ARG;
    if (!W_gate || !W_up || !W_down || !packed) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {W_gate, W_up, W_down, packed};
    for (const void* p : ps)
        if (misaligned(p)) return MOE_ERR_ALIGNMENT;
    int rc = check_device();
    if (rc) return rc;
    return cuda_status(launch_pack_experts((const __nv_bfloat16*)W_gate,
                                           (const __nv_bfloat16*)W_up,
                                           (const __nv_bfloat16*)W_down, H, E, I,
                                           (char*)packed, (cudaStream_t)stream));
}

int moe_forward_packed(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                       const void* packed_experts, int E, int K, int I, int norm_topk_prob,
                       moe_bf16* out, float* router_logits, int32_t* topk_idx, float* topk_w,
                       float* aux, void* workspace, size_t workspace_bytes, void* stream) {
    if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
    if (!packed_supported(H, E, I)) return MOE_ERR_INVALID_ARG;
    const ExpertWeights W{nullptr, nullptr, nullptr, (const char*)packed_experts};
    return forward_device(x, T, H, W_router, W, packed_experts, packed_experts, packed_experts,
                          E, K, I, norm_topk_prob, nullptr, 0, out, router_logits, topk_idx,
                          topk_w, aux, workspace, workspace_bytes, (cudaStream_t)stream);
}

size_t moe_q4_experts_bytes(int H, int E, int I) {
    if (H < 64 || H % 64 || I < 64 || I % 64 || E < 1 || E > kMaxExperts) return 0;
    if (!q4_supported(H, E, I)) return 0;
    return q4_experts_bytes(H, E, I);
}

int moe_quantize_experts_q4(const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                            int H, int E, int I, void* q4_experts, void* stream) {
    if (!moe_q4_experts_bytes(H, E, I)) return MOE_ERR_INVALID_ARG;
    if (!W_gate || !W_up || !W_down || !q4_experts) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {W_gate, W_up, W_down, q4_experts};
    for (const void* p : ps)
        if (misaligned(p)) return MOE_ERR_ALIGNMENT;
    int rc = check_device();
    if (rc) return rc;
    return cuda_status(launch_quantize_q4((const __nv_bfloat16*)W_gate,
                                          (const __nv_bfloat16*)W_up,
                                          (const __nv_bfloat16*)W_down, H, E, I,
                                          (char*)q4_experts, (cudaStream_t)stream));
}

int moe_dequantize_experts_q4(const void* q4_experts, int H, int E, int I, moe_bf16* W_gate,
                              moe_bf16* W_up, moe_bf16* W_down, void* stream) {
    if (!moe_q4_experts_bytes(H, E, I)) return MOE_ERR_INVALID_ARG;
    if (!W_gate || !W_up || !W_down || !q4_experts) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {W_gate, W_up, W_down, q4_experts};
    for (const void* p : ps)
        if (misaligned(p)) return MOE_ERR_ALIGNMENT;
    int rc = check_device();
    if (rc) return rc;
    return cuda_status(launch_dequantize_q4((const char*)q4_experts, H, E, I,
                                            (__nv_bfloat16*)W_gate, (__nv_bfloat16*)W_up,
                                            (__nv_bfloat16*)W_down, (cudaStream_t)stream));
}

int moe_forward_q4(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                   const void* q4_experts, int E, int K, int I, int norm_topk_prob,
                   moe_bf16* out, float* router_logits, int32_t* topk_idx, float* topk_w,
                   float* aux, void* workspace, size_t workspace_bytes, void* stream) {
    if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
    if (!moe_q4_experts_bytes(H, E, I)) return MOE_ERR_INVALID_ARG;
    if (misaligned(q4_experts)) return MOE_ERR_ALIGNMENT;
    ExpertWeights W{nullptr, nullptr, nullptr, nullptr};
    W.q4 = (const char*)q4_experts;
    return forward_device(x, T, H, W_router, W, q4_experts, q4_experts, q4_experts, E, K, I,
                          norm_topk_prob, nullptr, 0, out, router_logits, topk_idx, topk_w, aux,
                          workspace, workspace_bytes, (cudaStream_t)stream);
}

int moe_forward_opts(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                     const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down, int E,
                     int K, int I, int norm_topk_prob, moe_bf16* out, float* router_logits,
                     int32_t* topk_idx, float* topk_w, float* aux, const moe_forward_options* opts,
                     void* stream) {
    const moe_forward_options none{};
    const moe_forward_options& o = opts ? *opts : none;
    if (!(o.capacity_factor >= 0.f) || o.capacity_factor > 1e6f) return MOE_ERR_INVALID_ARG;
    if (E < 1 || T < 0 || K < 1) return MOE_ERR_INVALID_ARG;
    // capacity in pairs: ceil(cf * T * K / E); 0 = none
    const double cf_pairs = (double)o.capacity_factor * T * K / E;
    const int cap = o.capacity_factor > 0.f ? (int)(cf_pairs < 1.0 ? 1.0 : std::ceil(cf_pairs)) : 0;
    if (o.packed_experts && o.q4_experts) return MOE_ERR_INVALID_ARG;
    if (o.q4_experts) {
        if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
        if (!moe_q4_experts_bytes(H, E, I)) return MOE_ERR_INVALID_ARG;
        if (misaligned(o.q4_experts)) return MOE_ERR_ALIGNMENT;
        ExpertWeights W{nullptr, nullptr, nullptr, nullptr};
        W.q4 = (const char*)o.q4_experts;
        return forward_device(x, T, H, W_router, W, o.q4_experts, o.q4_experts, o.q4_experts, E,
                              K, I, norm_topk_prob, o.expert_bias, cap, out, router_logits,
                              topk_idx, topk_w, aux, o.workspace, o.workspace_bytes,
                              (cudaStream_t)stream);
    }
    if (o.packed_experts) {
        if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
        if (!packed_supported(H, E, I)) return MOE_ERR_INVALID_ARG;
        const ExpertWeights W{nullptr, nullptr, nullptr, (const char*)o.packed_experts};
        return forward_device(x, T, H, W_router, W, o.packed_experts, o.packed_experts,
                              o.packed_experts, E, K, I, norm_topk_prob, o.expert_bias, cap, out,
                              router_logits, topk_idx, topk_w, aux, o.workspace,
                              o.workspace_bytes, (cudaStream_t)stream);
    }
    const ExpertWeights W{(const __nv_bfloat16*)W_gate, (const __nv_bfloat16*)W_up,
                          (const __nv_bfloat16*)W_down, nullptr};
    return forward_device(x, T, H, W_router, W, W_gate, W_up, W_down, E, K, I, norm_topk_prob,
                          o.expert_bias, cap, out, router_logits, topk_idx, topk_w, aux,
                          o.workspace, o.workspace_bytes, (cudaStream_t)stream);
}

int moe_forward_host(const moe_bf16* x_host, int T, int H, const moe_bf16* W_router,
                     const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down, int E,
                     int K, int I, int norm_topk_prob, moe_bf16* out_host,
                     float* router_logits_host, int32_t* topk_idx_host, float* topk_w_host,
                     float* aux_host, void* stream) {
    const ExpertWeights W{(const __nv_bfloat16*)W_gate, (const __nv_bfloat16*)W_up,
                          (const __nv_bfloat16*)W_down, nullptr};
    return forward_host(x_host, T, H, W_router, W, W_gate, W_up, W_down, E, K, I, norm_topk_prob,
                        nullptr, 0, out_host, router_logits_host, topk_idx_host, topk_w_host,
                        aux_host, (cudaStream_t)stream);
}

int moe_forward_host_packed(const moe_bf16* x_host, int T, int H, const moe_bf16* W_router,
                            const void* packed_experts, int E, int K, int I, int norm_topk_prob,
                            moe_bf16* out_host, float* router_logits_host,
                            int32_t* topk_idx_host, float* topk_w_host, float* aux_host,
                            void* stream) {
    if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
    if (!packed_supported(H, E, I)) return MOE_ERR_INVALID_ARG;
    const ExpertWeights W{nullptr, nullptr, nullptr, (const char*)packed_experts};
    return forward_host(x_host, T, H, W_router, W, packed_experts, packed_experts,
                        packed_experts, E, K, I, norm_topk_prob, nullptr, 0, out_host,
                        router_logits_host, topk_idx_host, topk_w_host, aux_host,
                        (cudaStream_t)stream);
}

int moe_forward_host_q4(const moe_bf16* x_host, int T, int H, const moe_bf16* W_router,
                        const void* q4_experts, int E, int K, int I, int norm_topk_prob,
                        moe_bf16* out_host, float* router_logits_host, int32_t* topk_idx_host,
                        float* topk_w_host, float* aux_host, void* stream) {
    if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
    if (!moe_q4_experts_bytes(H, E, I)) return MOE_ERR_INVALID_ARG;
    if (misaligned(q4_experts)) return MOE_ERR_ALIGNMENT;
    ExpertWeights W{nullptr, nullptr, nullptr, nullptr};
    W.q4 = (const char*)q4_experts;
    return forward_host(x_host, T, H, W_router, W, q4_experts, q4_experts, q4_experts, E, K, I,
                        norm_topk_prob, nullptr, 0, out_host, router_logits_host, topk_idx_host,
                        topk_w_host, aux_host, (cudaStream_t)stream);
}

int moe_last_expert_counts(int32_t* counts_host, int E, void* stream) {
    if (!counts_host || E < 1) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t* src = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find(ws_key(st));
        if (it == g_ws.end() || !it->second.counts || it->second.E != E)
            return MOE_ERR_INVALID_ARG;
        src = it->second.counts;
    }
    cudaError_t e = cudaMemcpyAsync(counts_host, src, (size_t)E * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

int moe_device_status(const void* workspace, int T, int H, int E, int K, int I, void* stream) {
    cudaStream_t st = (cudaStream_t)stream;
    int32_t* status = nullptr;
    if (workspace) {
        if (check_sizes(T, H, E, K, I)) return MOE_ERR_INVALID_ARG;
        Sizes s{T, H, E, K, I};
        Workspace ws;
        layout_workspace(s, (char*)workspace, &ws, false);  // the status word's offset
        status = ws.status;
    } else {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        auto it = g_ws.find(ws_key(st));
        if (it == g_ws.end() || !it->second.status) return MOE_OK;
        status = it->second.status;
    }
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, status, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    return v == 0 ? MOE_OK : v;
}

int moe_dbg_route_from_logits(const float* logits, int T, int E, int K, int norm_topk_prob,
                              const float* expert_bias, int32_t* topk_idx, float* topk_w,
                              void* stream) {
    if (T < 0 || E < 1 || E > kMaxExperts || K < 1 || K > E || K > kMaxTopK)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
    if (misaligned(logits) || misaligned(topk_idx) || misaligned(topk_w) ||
        misaligned(expert_bias))
        return MOE_ERR_ALIGNMENT;
    int rc = check_device();
    if (rc) return rc;
    if (T == 0) return MOE_OK;
    Sizes s{T, 64, E, K, 64};
    return cuda_status(launch_route_from_logits(logits, 1, nullptr, s, norm_topk_prob,
                                                expert_bias, topk_idx, topk_w, nullptr,
                                                (cudaStream_t)stream));
}

int moe_dbg_permute(const int32_t* topk_idx, int T, int E, int K, int capacity, int32_t* counts,
                    int32_t* offsets, int32_t* perm_tok, int32_t* perm_slot, int32_t* inv,
                    void* stream) {
    if (T < 0 || E < 1 || E > kMaxExperts || K < 1 || K > E || K > kMaxTopK)
        return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || (T > 0 && (!topk_idx || !perm_tok || !perm_slot || !inv)))
        return MOE_ERR_INVALID_ARG;
    const void* ps[] = {topk_idx, counts, offsets, perm_tok, perm_slot, inv};
    for (const void* p : ps)
        if (misaligned(p)) return MOE_ERR_ALIGNMENT;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, (size_t)E * 4, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, ((size_t)E + 1) * 4, st);
        return cuda_status(e);
    }
    Sizes s{T, 64, E, K, 64};
    // Private scratch for the chunk tables and tiles (small), stream-ordered,
    // apart from the forwards' workspace.
    const size_t nch = (size_t)(s.nchunks() > 0 ? s.nchunks() : 1);
    const size_t tb = (size_t)s.max_tiles(kStreamRows) * sizeof(RowTile);
    const size_t bytes = align_up(nch * E * 4, 256) * 2 + align_up(tb, 256) + 256;
    void* base = nullptr;
    rc = owned_workspace(st, bytes, &base, 1);
    if (rc) return rc;
    Workspace ws{};
    char* p = (char*)base;
    ws.chunk_counts = (int32_t*)p;
    p += align_up(nch * E * 4, 256);
    ws.chunk_base = (int32_t*)p;
    p += align_up(nch * E * 4, 256);
    ws.tiles = (RowTile*)p;
    p += align_up(tb, 256);
    ws.n_tiles = (int32_t*)p;
    ws.counts = counts;
    ws.offsets = offsets;
    ws.perm_tok = perm_tok;
    ws.perm_slot = perm_slot;
    ws.inv = inv;
    ws.w_perm = nullptr;
    return cuda_status(
        launch_dispatch(topk_idx, nullptr, nullptr, s, ws, kStreamRows, nullptr, 0, nullptr,
                        capacity > 0 ? capacity : 0, st));
}

int moe_dbg_combine(const moe_bf16* Y, const int32_t* inv, int T, int K, int H, moe_bf16* out,
                    void* stream) {
    if (T < 0 || K < 1 || K > kMaxTopK || H < 8 || H % 8) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!Y || !inv || !out)) return MOE_ERR_INVALID_ARG;
    if (misaligned(Y) || misaligned(inv) || misaligned(out)) return MOE_ERR_ALIGNMENT;
    int rc = check_device();
    if (rc) return rc;
    if (T == 0) return MOE_OK;
    return cuda_status(launch_combine((const __nv_bfloat16*)Y, nullptr, inv, true, T, K, H,
                                      (__nv_bfloat16*)out,
                                      (cudaStream_t)stream));
}

}  // extern "C"
