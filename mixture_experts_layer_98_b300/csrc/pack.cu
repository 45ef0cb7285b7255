// pack.cu -- expert weights in the tile-major layout the expert GEMMs stream.
//
// The expert projections gate_proj / up_proj [I,H] and down_proj [H,I] (csdn
// page "MoE架构深度解析：128专家与8激活的智能路由", section
// "128个专家网络的组织结构与参数分布") are row-major in the caller's memory.
// A 128x64 tile of such a matrix is 128 separate 128-byte row pieces, and
// streaming the weights as tiled TMA boxes made the expert GEMMs' loads about
// a quarter slower than streaming the same bytes as contiguous 16 KB blocks.
// The packed layout stores every 128-row x 64-column block of each
// expert's matrix as one contiguous 16 KB block, already in the 128-byte
// swizzled K-major arrangement the tcgen05 shared-memory descriptors read:
//
//   element (r, k) of a block (r < 128, k < 64) sits at byte
//       r*128 + (((k/8) ^ (r%8)) * 16) + (k%8)*2
//
// (8-row, 1024-byte swizzle atoms stacked along the rows).  Blocks of one
// matrix are ordered (expert, 128-row block, 64-column block); the packed
// buffer holds W_gate's blocks, then W_up's, then W_down's.  Packing is a
// one-time transform of the weights (model load), not part of a forward.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kPackThreads = 256;

// One CTA per 16 KB block: 128 rows x 8 chunks of 16 bytes, 4 chunks a thread.
// src is row-major [E * R, C] (R rows per expert); dst gets blocks ordered
// (expert, row block, column block).
__global__ void __launch_bounds__(kPackThreads) pack_blocks_kernel(const uint4* src, int R,
                                                                   int C, uint4* dst) {
    const int kbs = C / kPackCols;                       // column blocks per row block
    const long long blk = blockIdx.x;                    // (e * R/128 + rb) * kbs + kb
    const long long row_blk = blk / kbs;                 // global 128-row block
    const int kb = (int)(blk % kbs);
    const int vpr = C / 8;                               // 16-byte chunks per source row
    for (int i = threadIdx.x; i < kPackRows * 8; i += blockDim.x) {
        const int r = i >> 3, c = i & 7;
        const uint4 v = src[(size_t)(row_blk * kPackRows + r) * vpr + (size_t)kb * 8 + c];
        dst[(size_t)blk * (kPackBlockBytes / 16) + r * 8 + (c ^ (r & 7))] = v;
    }
}

cudaError_t pack_matrix(const __nv_bfloat16* src, int E, int R, int C, char* dst,
                        cudaStream_t st) {
    const long long blocks = (long long)E * (R / kPackRows) * (C / kPackCols);
    pack_blocks_kernel<<<(unsigned)blocks, kPackThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(src), R, C, reinterpret_cast<uint4*>(dst));
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool packed_supported(int H, int E, int I) {
    return E >= 1 && I % 128 == 0 && H % 256 == 0;
}

size_t packed_matrix_bytes(int H, int E, int I) { return (size_t)E * I * H * 2; }

cudaError_t launch_pack_experts(const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                                const __nv_bfloat16* Wd, int H, int E, int I, char* packed,
                                cudaStream_t st) {
    const size_t mb = packed_matrix_bytes(H, E, I);
    cudaError_t e = pack_matrix(Wg, E, I, H, packed, st);
    if (e == cudaSuccess) e = pack_matrix(Wu, E, I, H, packed + mb, st);
    if (e == cudaSuccess) e = pack_matrix(Wd, E, H, I, packed + 2 * mb, st);
    return e;
}

}  // namespace moe
