// Decode work plan: a small kernel that runs before the decode kernel and
// turns the batch's sequence lengths into the decode grid's work list.
//
// The page "vLLM核心概念" §4.2 and the tbr8.org PagedAttention article §2.2
// make a decode step one pass over every sequence's blocks; split-K cuts a
// long sequence into partitions.  A grid of (KV head group, partition,
// sequence) sized by the longest sequence leaves most CTAs of a mixed-length
// batch with nothing to do (past their sequence's end), and each still costs a
// dispatch and a load.  The plan instead lists exactly the (sequence,
// partition) items that exist, in an order that starts long sequences first:
//
//  * partition size: at least the host's choice; when the call asks for the
//    automatic size, about 0.85 x the positions per resident CTA slot
//    (sum_s L_s * KV head groups / slots; twice that for an E4M3 pool, whose
//    positions are half the bytes), in multiples of 512, capped by the
//    longest sequence and by the staged table, raised when the item count
//    would spill a quarter wave or less past one full wave, then shrunk to
//    the smallest multiple of 64 that splits the longest sequence into as
//    many partitions when that adds no work items (equal partitions on the
//    critical path);
//  * order: groups of adjacent sequences that share their first physical
//    block (forks of one prompt, "LLM 推理引擎内部原理" §3.3) stay together, so
//    their shared prefix is read while it is still in L2; groups are ordered
//    by their longest member, longest first, ties by sequence index;
//  * the list is padded to the grid's size with entries whose sequence is -1;
//  * the split-K merge tickets are zeroed.
//
// Every CTA of the plan kernel (one thread per sequence) derives the same
// partition size and order from the same lengths; each then ranks and writes
// the items of its own 64 sequences, 16 threads per sequence.  The
// merge sums partitions in partition order, so the decode output does not
// depend on the order chosen here.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPlanThreads = kPlanMaxSeqs;          // one thread per sequence in the batch-wide phases
constexpr int kRankSeqs = 64;                       // sequences each CTA ranks and writes
constexpr int kRankLanes = kPlanThreads / kRankSeqs;   // threads cooperating on one sequence's rank
constexpr int kWarps = kPlanThreads / 32;
constexpr int kGranule = 512;                       // automatic partition sizes: multiples of 512 positions

// Block-wide reductions with one barrier each: warp shuffles, one partial per
// warp in `buf`, then every warp reduces the partials with shuffles.  Callers
// alternate two buffers, so a buffer is rewritten only after a later barrier.
__device__ __forceinline__ long long block_sum(long long v, long long* buf) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) buf[threadIdx.x >> 5] = v;
    __syncthreads();
    v = buf[lane];                                  // kWarps == 32
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ int block_max(int v, long long* buf) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (lane == 0) buf[threadIdx.x >> 5] = v;
    __syncthreads();
    v = static_cast<int>(buf[lane]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Inclusive prefix maximum over the block (thread order).
__device__ __forceinline__ int block_scan_max(int v, long long* buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v = max(v, o);
    }
    if (lane == 31) buf[warp] = v;
    __syncthreads();
    int c = static_cast<int>(buf[lane]);            // scan of the warp maxima
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, c, off);
        if (lane >= off) c = max(c, o);
    }
    const int carry = __shfl_sync(0xffffffffu, c, warp > 0 ? warp - 1 : 0);
    return warp > 0 ? max(v, carry) : v;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const DecodeArgs a) {
    static_assert(kWarps == 32, "the second reduction stage reads one partial per lane");
    __shared__ int sB0[kPlanMaxSeqs];               // first physical block (-1: empty sequence)
    __shared__ int sGmax[kPlanMaxSeqs];             // per group start: the group's longest length
    __shared__ int sNp[kPlanMaxSeqs];               // partitions of each sequence
    __shared__ int sL[kPlanMaxSeqs];                // lengths, clamped to [0, max_seq_len]
    __shared__ long long sOrd[kPlanMaxSeqs];        // order key: group length << 11 | (2047 - index)
    __shared__ long long buf[2][kWarps];
    const int B = a.num_seqs;
    const int t = threadIdx.x;
    const int nh = a.num_kv_heads * a.head_groups;
    int nb = 0;                                     // next reduction buffer
    auto next = [&]() { long long* b = buf[nb]; nb ^= 1; return b; };
    grid_dependency_wait();                         // lengths and tables may come from the previous kernel
    launch_dependents();                            // the decode grid may launch now; it waits for this grid

    // ---- this thread's sequence: length (clamped to [0, max_seq_len]) and first block
    int L = 0, b0 = -1;
    if (t < B) {
        L = __ldg(a.seq_lens + t);
        const int first =
            a.max_blocks_per_seq > 0 ? __ldg(a.block_tables + static_cast<int64_t>(t) * a.max_blocks_per_seq) : -1;
        if (L > a.max_seq_len) {                    // precondition broken: attend over max_seq_len
            if (blockIdx.x == 0) raise_error(a.err, kErrBounds);
            L = a.max_seq_len;
        }
        L = max(L, 0);
        b0 = L > 0 ? first : -1;
        sB0[t] = b0;
        sGmax[t] = 0;
    }

    // ---- the caller's sum of the lengths, when given, must be the real one (it sized the grid)
    long long W = 0;
    if (a.part_auto || a.sum_seq_lens > 0) {
        W = block_sum(L, next());
        if (a.sum_seq_lens > 0 && W != a.sum_seq_lens && blockIdx.x == 0 && t == 0) raise_error(a.err, kErrBounds);
    }

    // ---- partition size
    int P = a.part_tokens;
    if (a.part_auto) {
        const int lmax = block_max(L, next());
        const long long slots = a.slots > 0 ? a.slots : 1;
        // 0.85 x the positions per slot, counted in 16-bit-pool bytes: an E4M3
        // position is half the bytes, so its partitions are twice as long
        const long long target = (W * nh * (a.kv8 ? 34 : 17)) / (slots * 20);
        long long p = ((target + kGranule / 2) / kGranule) * kGranule;       // nearest multiple of 512
        p = max(p, static_cast<long long>(kGranule));
        const int table_cap = dec::kMaxTable * a.block_size;
        const int cap = max(a.part_tokens, min(table_cap, (lmax + 63) / 64 * 64));
        P = static_cast<int>(min(max(p, static_cast<long long>(a.part_tokens)), static_cast<long long>(cap)));
        // a quarter wave or less past one full wave: take the next size that fits one wave
        const long long n = block_sum(t < B ? max(1, (L + P - 1) / P) : 0, next()) * nh;
        if (n > slots && n * 4 <= slots * 5) {
            int q = P;
            while (q < cap) {
                q = min(q + kGranule, cap);
                if (block_sum(t < B ? max(1, (L + q - 1) / q) : 0, next()) * nh <= slots) {
                    P = q;
                    break;
                }
            }
        }
        // balance the longest sequence's partitions: the smallest multiple of 64 that still
        // covers it in as many partitions, when that adds no work items (the critical path
        // shortens; more items cost more than they save)
        if (lmax > 0) {
            const int parts = (lmax + P - 1) / P;
            const int q = max(a.part_tokens, ((lmax + parts - 1) / parts + 63) / 64 * 64);
            if (q < P && block_sum(t < B ? max(1, (L + q - 1) / q) : 0, next()) <=
                             block_sum(t < B ? max(1, (L + P - 1) / P) : 0, next()))
                P = q;
        }
    } else {
        __syncthreads();                            // sB0 complete
    }

    // ---- partitions; prefix groups: a group starts at a sequence that does not
    // continue its predecessor's first block; its key is its longest member
    const int np = t < B ? max(1, (L + P - 1) / P) : 0;
    const bool start = t < B && (t == 0 || b0 < 0 || b0 != sB0[t - 1]);
    const int gid = block_scan_max(start ? t : -1, next());
    if (t < B) atomicMax(&sGmax[gid], L);
    const long long n_live = block_sum(np, next());  // its barrier also completes the atomics
    // more entries than the grid covers (only a wrong sum_seq_lens does this): the rest are
    // dropped below, and the error word says so
    if (n_live > a.plan_capacity && blockIdx.x == 0 && t == 0) raise_error(a.err, kErrBounds);
    if (t < B) {
        sNp[t] = np;
        sL[t] = L;
        sOrd[t] = (static_cast<long long>(sGmax[gid]) << 11) | (2047 - t);
    }
    __syncthreads();

    // ---- rank: the items of every sequence ordered before this CTA's sequences
    const int my = blockIdx.x * kRankSeqs + t / kRankLanes;
    const int sub = t % kRankLanes;
    int off = 0;
    if (my < B) {
        const long long key = sOrd[my];
#pragma unroll 4
        for (int u = sub; u < B; u += kRankLanes) off += sOrd[u] > key ? sNp[u] : 0;
    }
#pragma unroll
    for (int o = kRankLanes / 2; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
    if (my < B) {
        for (int p = sub; p < sNp[my]; p += kRankLanes) {
            const int y = off + p;
            if (y < a.plan_capacity) a.plan[y] = make_int4(my, p, sL[my], P);
        }
    }

    // ---- padding entries and tickets, spread over every CTA
    const int gt = blockIdx.x * kPlanThreads + t, gstride = gridDim.x * kPlanThreads;
    for (long long y = n_live + gt; y < a.plan_capacity; y += gstride) a.plan[y] = make_int4(-1, 0, 0, P);
    const long long nt = static_cast<long long>(B) * nh;
    for (long long i = gt; i < nt; i += gstride) a.tickets[i] = 0u;
}

}  // namespace

cudaError_t launch_decode_plan(const DecodeArgs& a, cudaStream_t s) {
    if (a.num_seqs <= 0 || a.num_seqs > kPlanMaxSeqs || !a.plan) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.num_seqs + kRankSeqs - 1) / kRankSeqs));
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, a);
}

}  // namespace pkv
