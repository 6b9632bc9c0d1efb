// copy_blocks: the copy-on-write block copy issued at a fork.
//
// "LLM 推理引擎内部原理" §3.1 / §3.3 (blocks_to_copy, Copy-on-Write) and
// "vLLM核心概念" §4.2.2: before a sequence writes into a block it shares, the
// block is copied to a private one.  A physical block of one layer's pool is
// block_size * num_kv_heads * head_dim contiguous elements, so each (pair,
// layer) is two contiguous memcpy's of that size (K and V), done here with
// 16-byte vector loads spread over several CTAs per block.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(const CopyArgs a) {
    const int layer = blockIdx.z;
    const uint4* kbase = a.key[layer];
    const uint4* vbase = a.value[layer];
    uint4* kout = a.key[layer];
    uint4* vout = a.value[layer];
    const int64_t bv = a.block_vecs;
    for (int64_t i = blockIdx.y; i < a.num_pairs; i += gridDim.y) {
        const int64_t src = a.pairs[2 * i];
        const int64_t dst = a.pairs[2 * i + 1];
        if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
            if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(a.err, kErrBounds);
            continue;
        }
        const uint4* ks = kbase + src * bv;
        const uint4* vs = vbase + src * bv;
        uint4* kd = kout + dst * bv;
        uint4* vd = vout + dst * bv;
        for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < bv;
             v += static_cast<int64_t>(gridDim.x) * kThreads) {
            const uint4 x = ks[v];
            const uint4 y = vs[v];
            kd[v] = x;
            vd[v] = y;
        }
    }
}
}  // namespace

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t s) {
    if (a.num_pairs <= 0 || a.num_layers <= 0) return cudaSuccess;
    const int64_t per_block = (a.block_vecs + kThreads - 1) / kThreads;
    const unsigned gx = static_cast<unsigned>(per_block < 16 ? per_block : 16);
    const unsigned gy = static_cast<unsigned>(a.num_pairs < 65535 ? a.num_pairs : 65535);
    dim3 grid(gx, gy, static_cast<unsigned>(a.num_layers));
    copy_blocks_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
