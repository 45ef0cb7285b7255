/*
 * moe_b300.h -- C ABI of the B300 (sm_103a) sparse Mixture-of-Experts block
 * forward.
 *
 * The operation is the forward method of the Qwen3-style sparse MoE block as
 * printed on the cnblogs page "大模型-qwen3 MoE 详细解读" (class
 * Qwen3MoeSparseMoeBlock): router logits x·W_routerᵀ (a bias-free Linear),
 * softmax in fp32, top-k, optional renormalisation of the k kept weights
 * (norm_topk_prob), dispatch of the tokens to their experts, the SwiGLU expert
 * MLP down(silu(gate(x)) ⊙ up(x)) (the gate_proj / up_proj / down_proj expert
 * of the csdn page "MoE架构深度解析：128专家与8激活的智能路由", section
 * "128个专家网络的组织结构与参数分布"), and the routing-weight-scaled combine back
 * into token order (the index_add_ of the forward).  It also produces the
 * load-balance statistic aux = n · Σ_i f_i · P_i of the csdn page's section
 * "负载均衡机制".
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - bf16 tensors are passed as uint16_t bit patterns (moe_bf16).
 *  - Every pointer is DEVICE memory unless the name ends in _host; arrays are
 *    contiguous, row-major, and must be 16-byte aligned.  The caller owns them;
 *    the library never frees or keeps them after the call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    enqueue work on it and return without waiting (except moe_forward_host);
 *    outputs are valid once that work completes.  No call synchronises the
 *    host with the device.
 *  - Every call returns a moe_status.  All argument checks happen before any
 *    work is enqueued: a call that returns an error other than MOE_ERR_CUDA
 *    has enqueued nothing.  No C++ exception crosses this interface.
 *  - Sizes: T >= 0 tokens, H hidden size, E experts, K experts per token, I
 *    expert intermediate size.  H and I must be multiples of 64 and at most
 *    65536, 1 <= E <= 256, 1 <= K <= min(E, 16).  T = 0 is a no-op that writes
 *    aux = 0.  Shapes the tensor-core kernels cannot tile at decode sizes
 *    (I % 128 != 0 or H % 256 != 0 with T*K < 32*E) run on the weight-streaming
 *    kernels, which also need H <= 12800 and I <= 12800 (MOE_ERR_INVALID_ARG
 *    otherwise, before any work).
 *  - Only NVIDIA Blackwell datacenter GPUs of compute capability 10.3 (B300)
 *    are supported; other devices give MOE_ERR_UNSUPPORTED_DEVICE.
 *  - Results are deterministic: the same inputs give bitwise identical outputs
 *    on every call (no floating-point atomics anywhere).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* a size out of range or a required pointer NULL  */
    MOE_ERR_ALIGNMENT = 2,          /* a pointer not 16-byte aligned                   */
    MOE_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3   */
    MOE_ERR_WORKSPACE = 4,          /* workspace too small, or it could not be grown    */
    MOE_ERR_CUDA = 5,               /* a CUDA call failed; see moe_last_cuda_error()    */
    MOE_ERR_TIMEOUT = 6             /* a bounded device-side wait gave up               */
};

/*
 * moe_forward -- the whole block forward on the current device.
 *
 *   x              [T, H]     bf16   hidden states, one row per token
 *   W_router       [E, H]     bf16   router weight (nn.Linear(H, E, bias=False))
 *   W_gate, W_up   [E, I, H]  bf16   per-expert gate_proj / up_proj weights
 *   W_down         [E, H, I]  bf16   per-expert down_proj weights
 *   norm_topk_prob            0/1    renormalise the K kept weights to sum to 1
 *   out            [T, H]     bf16   block output Σ_k w_k · MLP_{idx_k}(x_t)
 *   router_logits  [T, E]     fp32   x·W_routerᵀ (not rounded to bf16); may be NULL
 *   topk_idx       [T, K]     int32  selected experts, by descending logit, ties
 *                                    to the lower expert index; may be NULL
 *   topk_w         [T, K]     fp32   routing weights (softmax probabilities of
 *                                    the selected experts, renormalised if
 *                                    norm_topk_prob); may be NULL
 *   aux            [1]        fp32   E · Σ_e (counts_e/(T·K)) · mean_t p[t,e];
 *                                    may be NULL
 *
 * Scratch memory comes from a workspace the library owns: one per (device,
 * stream), grown on demand with stream-ordered allocation and kept until the
 * process exits.  Use moe_forward_ws to supply your own.
 */
int moe_forward(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                int E, int K, int I, int norm_topk_prob, moe_bf16* out,
                float* router_logits, int32_t* topk_idx, float* topk_w, float* aux,
                void* stream);

/* moe_forward for callers that cannot allocate device memory.  The pages have
 * no counterpart of this entry point; it exists for integrations where
 * allocating on the call path is not allowed: a runtime that fixed its memory
 * budget up front, host code that must not take the allocator's locks or wait
 * on its implicit synchronisation, or an embedding whose device memory belongs
 * to another runtime.  Arguments and results are exactly those of
 * moe_forward; the caller still provides every input and output buffer.
 *
 * Scratch: a 32 MiB array that is part of the loaded library (a __device__
 * variable), so nothing is allocated by the call.  Every GPU that loads the
 * library holds those 32 MiB until the process exits.  This call takes no
 * expert capacity, so it needs the scratch of a forward without one:
 * moe_workspace_bytes(T,H,E,K,I) less the T·K·H·2 bytes that only a capacity
 * forward uses.  Sizes whose need exceeds 32 MiB are rejected with
 * MOE_ERR_WORKSPACE before any work (e.g. the H=4096, E=128, K=8, I=1536
 * layer fits up to T = 212 tokens).
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture.  All calls on a device share the one array and it keeps the last
 * call's contents (nothing in it needs to start at zero: each call writes
 * every part before reading it).  Calls whose work overlaps on the GPU --
 * concurrent streams, or host threads racing on one device -- race on the
 * array; serialise them. */
int moe_forward_noalloc(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                        const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                        int E, int K, int I, int norm_topk_prob, moe_bf16* out,
                        float* router_logits, int32_t* topk_idx, float* topk_w, float* aux,
                        void* stream);

/* Bytes of device workspace moe_forward_ws needs for these sizes (0 on a size
 * error).  The requirement grows with T·K·(H+I); it does not depend on data.
 * It covers every forward of these sizes, including one under an expert
 * capacity (moe_forward_opts), which keeps the weighted expert outputs in
 * fp32 (T·K·H·2 bytes more than a forward without a capacity needs). */
size_t moe_workspace_bytes(int T, int H, int E, int K, int I);

/* moe_forward with caller-provided scratch: `workspace` is device memory of at
 * least moe_workspace_bytes(T,H,E,K,I) bytes, 256-byte aligned, that no other
 * work uses until this call's work has completed on `stream`.  Too small ->
 * MOE_ERR_WORKSPACE.  Every other argument is as for moe_forward. */
int moe_forward_ws(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                   const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                   int E, int K, int I, int norm_topk_prob, moe_bf16* out,
                   float* router_logits, int32_t* topk_idx, float* topk_w, float* aux,
                   void* workspace, size_t workspace_bytes, void* stream);

/* End-to-end call with host activations: copies x_host [T,H] to the device,
 * runs moe_forward, copies out_host [T,H] (and, when not NULL,
 * router_logits_host [T,E], topk_idx_host / topk_w_host [T,K], aux_host [1])
 * back, and waits for the stream, so the host buffers hold the results when
 * it returns.  The weights are device pointers (a loaded model).  Host buffers
 * should be page-locked for the copies to run at full speed.  Device staging
 * for x and the outputs lives in the library-owned workspace of `stream`. */
int moe_forward_host(const moe_bf16* x_host, int T, int H, const moe_bf16* W_router,
                     const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                     int E, int K, int I, int norm_topk_prob, moe_bf16* out_host,
                     float* router_logits_host, int32_t* topk_idx_host, float* topk_w_host,
                     float* aux_host, void* stream);

/* ---- packed expert weights ------------------------------------------------
 * No counterpart on the pages: a one-time layout transform of the expert
 * weights (done when a model is loaded) that lets the expert GEMMs stream them
 * as contiguous 16 KB blocks instead of 128 row pieces per tile.  Every
 * 128-row x 64-column block of each expert's W_gate [I,H], W_up [I,H] and
 * W_down [H,I] becomes one contiguous 16 KB block holding element (r, k) at
 * byte r*128 + (((k/8) ^ (r%8))*16) + (k%8)*2; blocks are ordered (expert,
 * row block, column block); the buffer holds W_gate's blocks, then W_up's,
 * then W_down's (3*E*I*H*2 bytes).  The forward computes exactly the same
 * products in the same order as with row-major weights, so its results are
 * bitwise identical to moe_forward's. */

/* Bytes of the packed weights for (H, E, I), or 0 when the shape cannot be
 * packed (packing needs I % 128 == 0 and H % 256 == 0, 1 <= E <= 256). */
size_t moe_packed_experts_bytes(int H, int E, int I);

/* Packs W_gate, W_up [E,I,H] and W_down [E,H,I] (row-major, device) into
 * `packed` (device, moe_packed_experts_bytes(H,E,I) bytes, 16-byte aligned,
 * owned by the caller) on `stream`.  MOE_ERR_INVALID_ARG for a shape that
 * cannot be packed or a NULL pointer; MOE_ERR_ALIGNMENT for a misaligned
 * pointer.  The row-major weights are not modified and are not needed by
 * moe_forward_packed. */
int moe_pack_experts(const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                     int H, int E, int I, void* packed, void* stream);

/* moe_forward with packed expert weights (from moe_pack_experts with the same
 * H, E, I).  workspace == NULL uses the library-owned workspace of `stream`
 * (as moe_forward); otherwise it is the caller's scratch of at least
 * moe_workspace_bytes(T,H,E,K,I) bytes, 256-byte aligned (as moe_forward_ws).
 * MOE_ERR_INVALID_ARG for a shape that cannot be packed.  With packed
 * weights the expert MLPs always run on the tensor cores (the
 * MOE_PATH_STREAMING setting selects the weights-as-M kernels instead). */
int moe_forward_packed(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                       const void* packed_experts, int E, int K, int I, int norm_topk_prob,
                       moe_bf16* out, float* router_logits, int32_t* topk_idx, float* topk_w,
                       float* aux, void* workspace, size_t workspace_bytes, void* stream);

/* moe_forward_host with packed expert weights. */
int moe_forward_host_packed(const moe_bf16* x_host, int T, int H, const moe_bf16* W_router,
                            const void* packed_experts, int E, int K, int I,
                            int norm_topk_prob, moe_bf16* out_host, float* router_logits_host,
                            int32_t* topk_idx_host, float* topk_w_host, float* aux_host,
                            void* stream);

/* ---- 4-bit group-quantised experts ----------------------------------------
 *
 * Weight-only quantisation of the expert projections as the csdn page
 * "MoE架构深度解析：128专家与8激活的智能路由" describes it (section
 * "参数量化与存储优化": 4-bit values, groups of 128 parameters, a scale and a
 * bias per group; the page gives no formula).  Reading implemented: a group is
 * 128 consecutive entries of a weight row (along H for W_gate / W_up, along I
 * for W_down); with lo / hi its minimum / maximum (a zero minimum as +0),
 * s = bf16((hi - lo) / 15), b = lo, and each weight's code
 * q = clamp(rint((w - b) / s), 0, 15) in fp32 (q = 0 when s = 0).  A forward
 * with 4-bit experts is exactly the bf16 forward with the dequantised weights
 * w' = bf16(q·s + b) (rounded once); it reads 4.25 bits per weight.
 *
 * Buffer layout (device, from moe_quantize_experts_q4), per matrix -- W_gate
 * [E,I,H], W_up [E,I,H], W_down [E,H,I], R rows per expert, C columns -- a code
 * section then a scale section, in the order gate, up, down:
 *   codes  (E·R·C/2 bytes): 4096-byte blocks of 128 rows x 64 columns ordered
 *          (expert, row block, column block); in a block, row r is 8 32-bit
 *          words from byte r·32; word c holds columns 8c..8c+7: column 8c+2j
 *          in bits 4j..4j+3 and column 8c+2j+1 in bits 16+4j..19+4j (j=0..3);
 *   scales (E·R·(C/128)·4 bytes): 512-byte blocks of 128 rows x one 128-column
 *          group ordered (expert, row block, group); word r = bf16 s (bits
 *          0-15) | bf16 b (bits 16-31) of row r.
 * Shapes: I % 128 == 0 and H % 256 == 0 (else 0 bytes / MOE_ERR_INVALID_ARG).
 */

/* Bytes of the 4-bit buffer for (H, E, I); 0 for an unsupported shape. */
size_t moe_q4_experts_bytes(int H, int E, int I);

/* Quantises row-major bf16 expert weights (device) into `q4_experts` (device,
 * moe_q4_experts_bytes bytes, 16-byte aligned, owned by the caller) on
 * `stream`: a one-time model-load step.  MOE_ERR_INVALID_ARG for an
 * unsupported shape or a NULL pointer, MOE_ERR_ALIGNMENT for a misaligned one. */
int moe_quantize_experts_q4(const moe_bf16* W_gate, const moe_bf16* W_up,
                            const moe_bf16* W_down, int H, int E, int I, void* q4_experts,
                            void* stream);

/* The dequantised weights w' = bf16(q·s + b) of a 4-bit buffer, written as
 * row-major bf16 W_gate [E,I,H], W_up [E,I,H], W_down [E,H,I] (device, caller
 * owned) on `stream`.  Errors as moe_quantize_experts_q4. */
int moe_dequantize_experts_q4(const void* q4_experts, int H, int E, int I, moe_bf16* W_gate,
                              moe_bf16* W_up, moe_bf16* W_down, void* stream);

/* moe_forward with 4-bit expert weights (moe_quantize_experts_q4 with the
 * same H, E, I); workspace as for moe_forward_packed.  Decode batches (T <= 64
 * under MOE_PATH_AUTO) run the expert MLPs on warp-level tensor-core MMAs whose
 * weight operands are dequantised straight into registers (row tiles of <= 16
 * tokens); larger batches on tcgen05 kernels with a row tile's tokens (<= 64)
 * on the MMA's M side and 256 weight rows, dequantised in shared memory, on its
 * N side (MOE_PATH_WARP_MMA / MOE_PATH_TCGEN05 force either).  Either way the
 * results are those of the bf16 forward on the dequantised weights up to the
 * order of fp32 sums.  4 bits pay at decode, where the expert weights' bytes
 * bound the forward; at prefill sizes the bf16 forward is faster. */
int moe_forward_q4(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                   const void* q4_experts, int E, int K, int I, int norm_topk_prob,
                   moe_bf16* out, float* router_logits, int32_t* topk_idx, float* topk_w,
                   float* aux, void* workspace, size_t workspace_bytes, void* stream);

/* moe_forward_host with 4-bit expert weights (q4_experts on the device, from
 * moe_quantize_experts_q4 with the same H, E, I); host buffers and errors as
 * moe_forward_host, shapes and kernels as moe_forward_q4. */
int moe_forward_host_q4(const moe_bf16* x_host, int T, int H, const moe_bf16* W_router,
                        const void* q4_experts, int E, int K, int I, int norm_topk_prob,
                        moe_bf16* out_host, float* router_logits_host, int32_t* topk_idx_host,
                        float* topk_w_host, float* aux_host, void* stream);

/* ---- forward with options ------------------------------------------------ */

/* Optional inputs of moe_forward_opts; a zero-initialised struct (or a NULL
 * pointer) gives moe_forward. */
typedef struct moe_forward_options {
    /* [E] fp32 device, or NULL.  Selection-only expert bias for
     * auxiliary-loss-free load balancing (the DeepSeek scheme named on the
     * sshipanoo.com page "项目 17：稀疏性的调度艺术：实现双专家 MoE 路由（MoE
     * Router）", section "第四阶段：更先进的路由方案：DeepSeek 的突破"): experts
     * are ranked by the fp32 key router_logits + expert_bias (ties to the lower
     * index) while topk_w are the unbiased softmax probabilities of the kept
     * experts (renormalised when norm_topk_prob); aux counts the biased
     * selection.  router_logits stay unbiased.  The bias's update rule (a
     * training-time controller) is the caller's. */
    const float* expert_bias;
    /* Packed expert weights from moe_pack_experts, or NULL for the row-major
     * W_gate / W_up / W_down (then ignored when packed_experts is set). */
    const void* packed_experts;
    /* Caller scratch of at least moe_workspace_bytes(T,H,E,K,I) bytes,
     * 256-byte aligned, or NULL for the library-owned workspace of `stream`. */
    void* workspace;
    size_t workspace_bytes;
    /* Expert capacity factor cf >= 0 (0: no capacity).  The capacity of the
     * csdn page "MoE架构深度解析：128专家与8激活的智能路由", section "容量因子设计"
     * (batch tokens / experts × factor), counted in token-expert pairs: each
     * expert keeps the first C = ceil(cf·T·K/E) pairs routed to it, in token
     * order (C >= 1), and the others are dropped: they add nothing to `out`.
     * topk_idx / topk_w, router_logits, aux and the expert counts stay the
     * router's.  A negative or non-finite cf gives MOE_ERR_INVALID_ARG. */
    float capacity_factor;
    /* 4-bit quantised expert weights from moe_quantize_experts_q4 (the row-major
     * W_gate / W_up / W_down are then ignored), or NULL.  Not together with
     * packed_experts (MOE_ERR_INVALID_ARG). */
    const void* q4_experts;
} moe_forward_options;

/* moe_forward with the options above; every other argument as for
 * moe_forward.  A misaligned expert_bias gives MOE_ERR_ALIGNMENT. */
int moe_forward_opts(const moe_bf16* x, int T, int H, const moe_bf16* W_router,
                     const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                     int E, int K, int I, int norm_topk_prob, moe_bf16* out,
                     float* router_logits, int32_t* topk_idx, float* topk_w, float* aux,
                     const moe_forward_options* opts, void* stream);

/* Per-expert pair counts ("expert utilisation histogram") of the last
 * forward on `stream` that used the library-owned workspace (moe_forward,
 * moe_forward_host, moe_forward_host_packed, moe_forward_host_q4, and
 * moe_forward_packed / moe_forward_q4 without a workspace), copied into counts_host[E]
 * (waits for the stream).  MOE_ERR_INVALID_ARG if there was no such call. */
int moe_last_expert_counts(int32_t* counts_host, int E, void* stream);

/* Device-side status of the last forward that used `workspace` (the
 * caller's workspace of moe_forward_ws or moe_forward_packed, with the sizes
 * of that call), or, with workspace == NULL, of the last forward on `stream`
 * that used the library-owned workspace.
 * Waits for the stream.  Returns MOE_OK, or MOE_ERR_TIMEOUT if a bounded
 * device-side wait of that forward gave up (its outputs are then invalid). */
int moe_device_status(const void* workspace, int T, int H, int E, int K, int I, void* stream);

/* Human-readable name of a status code (static string). */
const char* moe_strerror(int status);

/* The cudaError_t value behind the last MOE_ERR_CUDA on this host thread. */
int moe_last_cuda_error(void);

/* Kernel-path selection for the expert MLPs (process-wide):
 *   MOE_PATH_AUTO         tcgen05 grouped GEMMs with token rows on the MMA's
 *                         M side when the average expert receives >= 32 rows
 *                         (P >= 32*E) -- on CTA pairs (256-row tiles) when
 *                         E <= 32 experts average >= 1024 rows and
 *                         I % 128 == 0, H % 256 == 0, else on single CTAs
 *                         (128-row tiles); below that the tcgen05 kernels with
 *                         the expert weights on the M side (for 1 <= T <= 16
 *                         fused with the combine into one kernel), or, for
 *                         shapes those cannot tile, the weight-streaming
 *                         kernels;
 *   MOE_PATH_STREAMING    always the weight-streaming CUDA-core kernels;
 *   MOE_PATH_TCGEN05      always the single-CTA token-rows-as-M tcgen05
 *                         grouped GEMMs;
 *   MOE_PATH_TCGEN05_PAIR always the CTA-pair token-rows-as-M grouped GEMMs
 *                         where the shape allows, else MOE_PATH_TCGEN05;
 *   MOE_PATH_TCGEN05_WT   always the weights-as-M tcgen05 kernels where the
 *                         shape allows (I % 128 == 0 and H % 256 == 0), else
 *                         the weight-streaming kernels; gate/up, down and
 *                         the combine as three kernels;
 *   MOE_PATH_TCGEN05_DECODE  as MOE_PATH_TCGEN05_WT, but with 1 <= T <= 64
 *                         the three run as one cooperative kernel (AUTO's
 *                         choice for T <= 16; bitwise the same results);
 *   MOE_PATH_WARP_MMA     4-bit experts (moe_forward_q4): always the kernels
 *                         that dequantise the weights into the registers of
 *                         warp-level MMAs (AUTO's choice for T <= 64); with
 *                         bf16 weights the same as MOE_PATH_AUTO.
 * With 4-bit experts, MOE_PATH_TCGEN05 selects the tcgen05 4-bit kernels (AUTO's
 * choice for T > 64) and every other value acts as MOE_PATH_AUTO.
 * Every path computes the same function; results agree within the fp32
 * accumulation-order tolerance (not bitwise across paths).
 * Returns the previous setting, or -1 for an unknown value. */
enum moe_path {
    MOE_PATH_AUTO = 0,
    MOE_PATH_STREAMING = 1,
    MOE_PATH_TCGEN05 = 2,
    MOE_PATH_TCGEN05_WT = 3,
    MOE_PATH_TCGEN05_PAIR = 4,
    MOE_PATH_TCGEN05_DECODE = 5,
    MOE_PATH_WARP_MMA = 6
};
int moe_set_expert_path(int path);

/* ---- benchmark instrumentation ------------------------------------------ */

/* Stages of one forward, in launch order. */
enum moe_stage {
    MOE_STAGE_ROUTER = 0,   /* router GEMM + softmax + top-k + renorm            */
    MOE_STAGE_DISPATCH = 1, /* histogram, scan, permutation, aux, row gather      */
    MOE_STAGE_GATE_UP = 2,  /* expert gate/up projections + SiLU·mul             */
    MOE_STAGE_DOWN = 3,     /* expert down projection × routing weight           */
    MOE_STAGE_COMBINE = 4,  /* gather-reduce into token order                     */
    MOE_NUM_STAGES = 5
};

/* enable != 0: every following forward records a CUDA event at each stage
 * boundary on its own stream (process-wide; meant for one benchmarking
 * stream at a time).  Returns MOE_OK, or MOE_ERR_CUDA if the events could not
 * be created. */
int moe_set_stage_timing(int enable);

/* Benchmark variant of stage timing without host waits: `events` points to
 * MOE_NUM_STAGES + 1 cudaEvent_t created by the caller; the next forward (and
 * only that one) records them at its stage boundaries on its stream.  Pass a
 * fresh set before each forward and read them with cudaEventElapsedTime
 * after synchronising.  NULL cancels a pending set. */
int moe_set_next_stage_events(void* const* events);

/* Waits for the events of the last forward recorded with stage timing and
 * writes the device time of each stage in milliseconds to ms[0..n) (n <=
 * MOE_NUM_STAGES).  MOE_ERR_INVALID_ARG if no forward was timed. */
int moe_stage_times(float* ms, int n);

/* Number of kernels this library has launched in this process. */
long long moe_kernel_launch_count(void);

/* ---- stage entry points (used by the stage-parity tests) --------------- */

/* Steps softmax -> top-k -> renormalise on given fp32 logits [T,E]:
 * topk_idx [T,K] int32 and topk_w [T,K] fp32, exactly as moe_forward
 * computes them from its own logits (expert_bias as in moe_forward_options,
 * or NULL). */
int moe_dbg_route_from_logits(const float* logits, int T, int E, int K, int norm_topk_prob,
                              const float* expert_bias, int32_t* topk_idx, float* topk_w,
                              void* stream);

/* Self-test of the bounded device-side waits (no counterpart on the pages):
 * one thread waits, for at most timeout_ns (1 ns .. 1 s), on an mbarrier that
 * nothing arrives on, then writes MOE_ERR_TIMEOUT to *status (device int32).
 * The same limit-and-record path ends every wait of the forward's kernels;
 * the context stays usable afterwards.  MOE_ERR_INVALID_ARG for a limit out
 * of range or a NULL status. */
int moe_dbg_wait_timeout(long long timeout_ns, int32_t* status, void* stream);

/* Dispatch of given selections topk_idx [T,K] (each row holds K distinct
 * experts in [0,E)): counts [E], offsets [E+1] (exclusive prefix sum),
 * perm_tok / perm_slot [T·K] (token and k-slot of each row, rows ordered by
 * expert then token) and inv [T,K] (row of each pair).  With capacity > 0,
 * each expert keeps its first `capacity` pairs in token order: offsets count
 * the kept pairs, only they get rows, inv = -1 for the others, and counts stay
 * the routed pairs.  Out-of-range experts are not checked on the device. */
int moe_dbg_permute(const int32_t* topk_idx, int T, int E, int K, int capacity, int32_t* counts,
                    int32_t* offsets, int32_t* perm_tok, int32_t* perm_slot, int32_t* inv,
                    void* stream);

/* Combine: out[t,:] = bf16( Σ_{k=0..K-1} Y[inv[t,k], :] ) with fp32 sums in
 * k order.  Y [T·K, H] bf16 holds the already weighted expert outputs in
 * dispatch order; inv [T,K]. */
int moe_dbg_combine(const moe_bf16* Y, const int32_t* inv, int T, int K, int H,
                    moe_bf16* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
