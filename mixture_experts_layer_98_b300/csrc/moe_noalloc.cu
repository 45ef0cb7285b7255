// moe_noalloc.cu -- the block forward for callers that cannot allocate device
// memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocator) on the
// path where they run the layer: code that runs inside a memory budget fixed
// up front, host code that must not take the allocator's locks or trigger its
// synchronisation, and integrations whose device memory is owned entirely by
// another runtime.  For them, moe_forward_noalloc runs the same kernels as
// moe_forward but takes its scratch from one array that is part of the loaded
// library itself, so nothing is allocated at call time.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads the library holds that much memory for it
// until the process exits, whether or not this entry point is ever called.
#include <mutex>

#include "moe_common.cuh"

namespace moe {

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code must not use the name as a device address:
// it only names the symbol; the address on each device comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress((void**)&p, g_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        if (!p) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_forward_noalloc(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                                   const moe_bf16* W_gate, const moe_bf16* W_up,
                                   const moe_bf16* W_down, int E, int K, int I,
                                   int norm_topk_prob, moe_bf16* out, float* router_logits,
                                   int32_t* topk_idx, float* topk_w, float* aux, void* stream) {
    int rc = check_forward_args(x, T, H, W_router, W_gate, W_up, W_down, E, K, I, out,
                                router_logits, topk_idx, topk_w, aux);
    if (rc) return rc;
    Sizes s{T, H, E, K, I};
    const size_t need = T > 0 ? layout_workspace(s, nullptr, nullptr, false) : 0;
    if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;  // before any work or set-up
    void* base = nullptr;
    rc = scratch_address(&base);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        if (aux) return cuda_status(cudaMemsetAsync(aux, 0, sizeof(float), st));
        return MOE_OK;
    }
    // Nothing in the scratch has to start at zero: the forward's first kernel
    // clears the status word, and every other region is written before it is
    // read within the same call.
    Workspace ws;
    layout_workspace(s, (char*)base, &ws, false);
    const ExpertWeights W{(const __nv_bfloat16*)W_gate, (const __nv_bfloat16*)W_up,
                          (const __nv_bfloat16*)W_down, nullptr};
    return run_forward((const __nv_bfloat16*)x, (const __nv_bfloat16*)W_router, W, s,
                       norm_topk_prob, nullptr, 0, (__nv_bfloat16*)out, router_logits, topk_idx, topk_w, aux,
                       ws, st);
}
