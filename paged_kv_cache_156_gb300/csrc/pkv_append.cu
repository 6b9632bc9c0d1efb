// paged_kv_append: scatter each new token's K/V row into its slot.
//
// The slot arithmetic is the one of the block manager's append_slot
// ("LLM 推理引擎内部原理" §2.3): slot = physical_block * block_size + offset, so
// a slot indexes the pool viewed as [num_blocks * block_size] rows of
// num_kv_heads * head_dim elements.  One warp moves one token: its K row and V
// row are each num_kv_heads * head_dim * 2 contiguous bytes in both the input
// and the pool, copied with 16-byte vector loads and stores.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {
constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) append_kernel(const AppendArgs a) {
    // This grid may have launched early: it waits for the previous one before
    // touching memory; then the next kernel (a plan or decode grid, which waits
    // for this one) may start launching.
    grid_dependency_wait();
    launch_dependents();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= a.num_tokens) return;
    const int64_t slot = a.slots[t];
    if (slot < 0) return;                       // padding entry: nothing to write
    if (slot >= a.num_slots) {                  // never write outside the pool
        if (lane == 0) raise_error(a.err, kErrBounds);
        return;
    }
    const uint4* ks = a.k + t * a.row_vecs;
    const uint4* vs = a.v + t * a.row_vecs;
    uint4* kd = a.key_cache + slot * a.row_vecs;
    uint4* vd = a.value_cache + slot * a.row_vecs;
    for (int i = lane; i < a.row_vecs; i += 32) {
        const uint4 x = __ldg(ks + i);
        const uint4 y = __ldg(vs + i);
        kd[i] = x;
        vd[i] = y;
    }
}

// ---------------------------------------------------------------- E4M3 pools
// The same scatter into an 8-bit pool (the KV quantization of "LLM 推理优化深度实战"
// §6.2: attention then reads low-precision K/V).  Each lane converts 8
// elements per step with quantize8 (pkv_device.cuh).
template <bool BF16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) append_fp8_kernel(const AppendFp8Args a) {
    grid_dependency_wait();
    launch_dependents();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= a.num_tokens) return;
    const int64_t slot = a.slots[t];
    if (slot < 0) return;
    if (slot >= a.num_slots) {
        if (lane == 0) raise_error(a.err, kErrBounds);
        return;
    }
    const uint4* ks = a.k + t * a.row_vecs;
    const uint4* vs = a.v + t * a.row_vecs;
    uint2* kd = a.key_cache + slot * a.row_vecs;
    uint2* vd = a.value_cache + slot * a.row_vecs;
    for (int i = lane; i < a.row_vecs; i += 32) {
        const int h = i / a.head_vecs;
        const uint4 x = __ldg(ks + i);
        const uint4 y = __ldg(vs + i);
        kd[i] = quantize8<BF16>(x, __ldg(a.k_scale + h));
        vd[i] = quantize8<BF16>(y, __ldg(a.v_scale + h));
    }
}

// Launched with programmatic stream serialization: the grid may become
// resident while the previous kernel (a decode) finishes, and waits for it.
template <typename Kern, typename Args>
cudaError_t launch_dependent(Kern kern, const Args& a, int64_t tokens, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((tokens + kWarpsPerBlock - 1) / kWarpsPerBlock));
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}
}  // namespace

cudaError_t launch_append_fp8(const AppendFp8Args& a, cudaStream_t s) {
    if (a.num_tokens <= 0) return cudaSuccess;
    return a.bf16 ? launch_dependent(append_fp8_kernel<true>, a, a.num_tokens, s)
                  : launch_dependent(append_fp8_kernel<false>, a, a.num_tokens, s);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
    if (a.num_tokens <= 0) return cudaSuccess;
    return launch_dependent(append_kernel, a, a.num_tokens, s);
}

}  // namespace pkv
