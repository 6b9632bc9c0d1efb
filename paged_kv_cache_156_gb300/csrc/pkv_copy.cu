// Block copies: the copy-on-write copy issued at a fork, and the swap of
// blocks between the device pool and a pinned host pool.
//
// "LLM 推理引擎内部原理" §3.1 (the scheduler output's blocks_to_copy,
// blocks_to_swap_in, blocks_to_swap_out), §3.2 (preemption by swapping:
// blocks move to CPU memory and back) and §3.3 (Copy-on-Write); "vLLM核心概念"
// §4.2.2: before a sequence writes into a block it shares, the block is
// copied to a private one.  A physical block of one layer's pool is
// block_size * num_kv_heads * head_dim contiguous elements, so each (pair,
// layer) is two contiguous copies of that size (K and V), done with 16-byte
// vector loads spread over several CTAs per block; each thread issues all of
// its loads (kUnroll vectors of K and of V) before its stores, so a fork's
// few megabytes of copies are in flight at once in one wave of CTAs.  Pinned host memory is
// addressed directly by the kernel (unified addressing), so a swap is the
// same gather as a copy.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {
constexpr int kThreads = 256;
constexpr int kUnroll = 4;                          // 16-byte vectors per thread and pool in flight
constexpr int64_t kSpan = static_cast<int64_t>(kThreads) * kUnroll;   // vectors of a block per CTA pass

__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(const CopyArgs a) {
    // This grid may have launched early: it waits for the previous one before
    // touching memory; then the next kernel (which waits for this grid) may
    // start launching.
    grid_dependency_wait();
    launch_dependents();
    const int layer = blockIdx.z;
    const uint4* kbase = a.src_key[layer];
    const uint4* vbase = a.src_value[layer];
    uint4* kout = a.dst_key[layer];
    uint4* vout = a.dst_value[layer];
    const int64_t bv = a.block_vecs;
    for (int64_t i = blockIdx.y; i < a.num_pairs; i += gridDim.y) {
        const int64_t src = a.pairs[2 * i];
        const int64_t dst = a.pairs[2 * i + 1];
        if (src < 0 || src >= a.src_num_blocks || dst < 0 || dst >= a.dst_num_blocks) {
            if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(a.err, kErrBounds);
            continue;
        }
        const uint4* ks = kbase + src * bv;
        const uint4* vs = vbase + src * bv;
        uint4* kd = kout + dst * bv;
        uint4* vd = vout + dst * bv;
        for (int64_t base = static_cast<int64_t>(blockIdx.x) * kSpan; base < bv;
             base += static_cast<int64_t>(gridDim.x) * kSpan) {
            uint4 x[kUnroll], y[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t v = base + u * kThreads + threadIdx.x;
                if (v < bv) {
                    x[u] = ks[v];
                    y[u] = vs[v];
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t v = base + u * kThreads + threadIdx.x;
                if (v < bv) {
                    kd[v] = x[u];
                    vd[v] = y[u];
                }
            }
        }
    }
}
}  // namespace

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t s) {
    if (a.num_pairs <= 0 || a.num_layers <= 0) return cudaSuccess;
    const int64_t per_block = (a.block_vecs + kSpan - 1) / kSpan;
    const unsigned gx = static_cast<unsigned>(per_block < 16 ? per_block : 16);
    const unsigned gy = static_cast<unsigned>(a.num_pairs < 65535 ? a.num_pairs : 65535);
    // programmatic stream serialization: the grid may become resident while
    // the previous kernel finishes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, gy, static_cast<unsigned>(a.num_layers));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, a);
}

}  // namespace pkv
