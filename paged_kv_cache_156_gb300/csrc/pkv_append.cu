// paged_kv_append: scatter each new token's K/V row into its slot.
//
// The slot arithmetic is the one of the block manager's append_slot
// ("LLM 推理引擎内部原理" §2.3): slot = physical_block * block_size + offset, so
// a slot indexes the pool viewed as [num_blocks * block_size] rows of
// num_kv_heads * head_dim elements.  One warp moves one token: its K row and V
// row are each num_kv_heads * head_dim * 2 contiguous bytes in both the input
// and the pool, copied with 16-byte vector loads and stores.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {
constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) append_kernel(const AppendArgs a) {
    // a following decode call's plan kernel may start launching; it waits for
    // this grid to finish before it reads anything
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
}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
    if (a.num_tokens <= 0) return cudaSuccess;
    const int64_t blocks = (a.num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
    append_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
