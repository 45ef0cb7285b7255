// quant.cu -- 4-bit group-quantised expert weights: the one-time quantiser and
// a dequantiser.
//
// The csdn page "MoE架构深度解析：128专家与8激活的智能路由" (section
// "参数量化与存储优化") stores the experts' weights as 4-bit values in groups of
// 128 parameters, each group with its own scale and bias.  Reading taken (the
// page gives no formula): a group is 128 consecutive entries of a weight row
// (along the projection's input dimension); with lo, hi its minimum and
// maximum (a zero minimum taken as +0), s = bf16((hi - lo) / 15) and b = lo; a
// weight's code is q = clamp(rint((w - b) / s), 0, 15), all in fp32 (q = 0
// when s = 0); the dequantised weight is w' = bf16(q·s + b), rounded once
// (fma.rn.bf16x2).
//
// Layout (moe_b300.h, moe_q4_experts_bytes): per matrix (W_gate [E,I,H],
// W_up [E,I,H], W_down [E,H,I]; R rows per expert, C columns) a code section
// and a scale section:
//   codes: 4 KB blocks of 128 rows x 64 columns, ordered (expert, row block,
//          column block); in a block, row r holds 8 words of 32 bits (bytes
//          r*32 ..), word c the columns 8c..8c+7 with column 8c+2j in bits
//          4j..4j+3 and column 8c+2j+1 in bits 16+4j..19+4j (j = 0..3), so that
//          (word >> 4j) & 0x000F000F holds one bf16 pair's codes;
//   scales: 512-byte blocks of 128 rows x one 128-column group, ordered
//          (expert, row block, group); word r = bf16 s (low half) | bf16 b
//          (high half) of row r.
// Sections in the order gate codes, gate scales, up codes, up scales, down
// codes, down scales.
#include "moe_common.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float bf16_bits_f32(uint16_t v) {
    return __uint_as_float((uint32_t)v << 16);
}

// One warp per (row, 128-column group): lane l holds columns 4l..4l+3.
__global__ void __launch_bounds__(256) quantize_q4_kernel(const uint16_t* W, long long rows,
                                                          int R, int C, uint32_t* codes,
                                                          uint32_t* scales) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int groups = C / 128;
    for (long long item = warp; item < rows * groups; item += nwarps) {
        const long long gr = item / groups;
        const int g = (int)(item % groups);
        const uint2 raw = *reinterpret_cast<const uint2*>(W + gr * C + (long long)g * 128 + 4 * lane);
        float v[4] = {bf16_bits_f32((uint16_t)(raw.x & 0xFFFFu)), bf16_bits_f32((uint16_t)(raw.x >> 16)),
                      bf16_bits_f32((uint16_t)(raw.y & 0xFFFFu)), bf16_bits_f32((uint16_t)(raw.y >> 16))};
        float lo = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
        float hi = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
        }
        if (lo == 0.0f) lo = 0.0f;  // a zero minimum is stored as +0
        const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
        const __nv_bfloat16 bb = __float2bfloat16_rn(lo);
        const float sf = __bfloat162float(sb), bf = __bfloat162float(bb);
        // this lane's four codes at their places in the shared 8-column word:
        // lane 2c holds columns 8c..8c+3 (element j), lane 2c+1 columns 8c+4..8c+7
        uint32_t part = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t code = 0;
            if (sf != 0.0f) {
                const float t = rintf(__fdiv_rn(__fsub_rn(v[j], bf), sf));
                code = t < 0.0f ? 0u : (t > 15.0f ? 15u : (uint32_t)t);
            }
            const int e = (lane & 1) * 4 + j;  // column within the word
            part |= code << ((e & 1) * 16 + (e >> 1) * 4);
        }
        const uint32_t word = part | __shfl_down_sync(0xffffffffu, part, 1);
        const long long e_ = gr / R;
        const int r = (int)(gr % R);
        const long long rb = (long long)e_ * (R / kPackRows) + r / kPackRows;
        if ((lane & 1) == 0) {
            const int c = lane >> 1;  // word 0..15 of the group: block 2g + c/8, word c%8
            const long long blk = rb * (C / kPackCols) + 2 * g + c / 8;
            codes[blk * (kQ4CodeBlockBytes / 4) + (r % kPackRows) * 8 + (c % 8)] = word;
        }
        if (lane == 0) {
            const uint32_t sbw = (uint32_t)__bfloat16_as_ushort(sb) |
                                 ((uint32_t)__bfloat16_as_ushort(bb) << 16);
            scales[(rb * groups + g) * kPackRows + (r % kPackRows)] = sbw;
        }
    }
}

// One thread per code word: eight bf16 weights of row-major W'.
__global__ void __launch_bounds__(256) dequantize_q4_kernel(const uint32_t* codes,
                                                            const uint32_t* scales,
                                                            long long rows, int R, int C,
                                                            uint4* W) {
    const long long words = rows * (C / 8);
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride) {
        const long long gr = i / (C / 8);
        const int col8 = (int)(i % (C / 8));  // word index along the row
        const long long e_ = gr / R;
        const int r = (int)(gr % R);
        const long long rb = (long long)e_ * (R / kPackRows) + r / kPackRows;
        const long long blk = rb * (C / kPackCols) + col8 / 8;
        const uint32_t w = codes[blk * (kQ4CodeBlockBytes / 4) + (r % kPackRows) * 8 + col8 % 8];
        const uint32_t sbw = scales[(rb * (C / 128) + col8 / 16) * kPackRows + (r % kPackRows)];
        W[i] = q4_dequant8(w, sbw);
    }
}

long long blocks_for(long long work, int per_block) {
    long long b = (work + per_block - 1) / per_block;
    const long long cap = (long long)num_sms() * 16;
    if (b > cap) b = cap;
    return b < 1 ? 1 : b;
}

size_t q4_code_bytes(int R, int C, int E) { return (size_t)E * R * C / 2; }
size_t q4_scale_bytes(int R, int C, int E) { return (size_t)E * R * (C / 128) * 4; }

}  // namespace

bool q4_supported(int H, int E, int I) { return E >= 1 && I % 128 == 0 && H % 256 == 0; }

Q4Sections q4_sections(const char* base, int H, int E, int I) {
    Q4Sections q;
    const size_t gc = q4_code_bytes(I, H, E), gs = q4_scale_bytes(I, H, E);
    const size_t dc = q4_code_bytes(H, I, E);
    q.codes[0] = base;
    q.scales[0] = base + gc;
    q.codes[1] = base + gc + gs;
    q.scales[1] = base + 2 * gc + gs;
    q.codes[2] = base + 2 * (gc + gs);
    q.scales[2] = base + 2 * (gc + gs) + dc;
    return q;
}

size_t q4_experts_bytes(int H, int E, int I) {
    return 2 * (q4_code_bytes(I, H, E) + q4_scale_bytes(I, H, E)) + q4_code_bytes(H, I, E) +
           q4_scale_bytes(H, I, E);
}

cudaError_t launch_quantize_q4(const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                               const __nv_bfloat16* Wd, int H, int E, int I, char* q4,
                               cudaStream_t st) {
    const Q4Sections q = q4_sections(q4, H, E, I);
    const __nv_bfloat16* src[3] = {Wg, Wu, Wd};
    const int R[3] = {I, I, H}, C[3] = {H, H, I};
    for (int m = 0; m < 3; ++m) {
        const long long rows = (long long)E * R[m];
        const long long items = rows * (C[m] / 128);
        quantize_q4_kernel<<<(unsigned)blocks_for(items * 32, 256), 256, 0, st>>>(
            reinterpret_cast<const uint16_t*>(src[m]), rows, R[m], C[m],
            reinterpret_cast<uint32_t*>(const_cast<char*>(q.codes[m])),
            reinterpret_cast<uint32_t*>(const_cast<char*>(q.scales[m])));
        count_launches(1);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_dequantize_q4(const char* q4, int H, int E, int I, __nv_bfloat16* Wg,
                                 __nv_bfloat16* Wu, __nv_bfloat16* Wd, cudaStream_t st) {
    const Q4Sections q = q4_sections(q4, H, E, I);
    __nv_bfloat16* dst[3] = {Wg, Wu, Wd};
    const int R[3] = {I, I, H}, C[3] = {H, H, I};
    for (int m = 0; m < 3; ++m) {
        const long long rows = (long long)E * R[m];
        dequantize_q4_kernel<<<(unsigned)blocks_for(rows * (C[m] / 8), 256), 256, 0, st>>>(
            reinterpret_cast<const uint32_t*>(q.codes[m]),
            reinterpret_cast<const uint32_t*>(q.scales[m]), rows, R[m], C[m],
            reinterpret_cast<uint4*>(dst[m]));
        count_launches(1);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
