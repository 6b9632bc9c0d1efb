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
//    (sum_s L_s * KV head groups / slots; 1.4 times that for an E4M3 pool,
//    whose positions are half the bytes), in multiples of 512, capped by the
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
// Every CTA of the plan kernel (one thread per sequence, the block sized to
// the batch: the next power of two, at least 64) derives the same partition
// size and order from the same lengths; each then ranks and writes the items
// of its own 64 sequences.  The plan is latency-bound (a few bytes per
// sequence), so its block-wide phases are merged: one barrier for the sum,
// maximum and prefix-group scan of the lengths, one for the item counts at
// the candidate partition sizes, one before ranking.  The merge sums
// partitions in partition order, so the decode output does not depend on
// the order chosen here.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kRankSeqs = 64;                       // sequences each CTA ranks and writes
constexpr int kMaxWarps = kPlanMaxSeqs / 32;
constexpr int kGranule = kPlanGranule;              // automatic partition sizes: multiples of 512 positions

template <typename V>
__device__ __forceinline__ V warp_sum(V v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Block sum with one barrier (the rare wave-size search): warp partials in
// `buf`, then every warp reduces them.  Callers alternate two buffers, so a
// buffer is rewritten only after a later barrier.
__device__ __forceinline__ long long block_sum(long long v, long long* buf) {
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    v = warp_sum(v);
    if (lane == 0) buf[threadIdx.x >> 5] = v;
    __syncthreads();
    return warp_sum(lane < nw ? buf[lane] : 0ll);
}

// Items of one sequence of length L at partition size P (every sequence has one).
__device__ __forceinline__ int parts_of(int L, int P) { return max(1, (L + P - 1) / P); }

// The smallest multiple of 64 (at least `floor`) that splits lmax into as many
// partitions as P does.
__device__ __forceinline__ int balanced(int lmax, int P, int floor) {
    const int parts = (lmax + P - 1) / P;
    return max(floor, ((lmax + parts - 1) / parts + 63) / 64 * 64);
}

__global__ void __launch_bounds__(kPlanMaxSeqs) plan_kernel(const DecodeArgs a) {
    __shared__ int sGmax[kPlanMaxSeqs];             // per group start: the group's longest length
    __shared__ int sNp[kPlanMaxSeqs];               // partitions of each sequence
    __shared__ int sL[kPlanMaxSeqs];                // lengths, clamped to [0, max_seq_len]
    __shared__ long long sOrd[kPlanMaxSeqs];        // order key: group length << 11 | (2047 - index)
    __shared__ long long sW[kMaxWarps];             // per warp: sum of lengths
    __shared__ int sMax[kMaxWarps], sScan[kMaxWarps], sC0[kMaxWarps], sC1[kMaxWarps];
    __shared__ long long buf[2][kMaxWarps];         // the rare search's reductions
    const int B = a.num_seqs;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = blockDim.x >> 5;
    const int nh = a.num_kv_heads * a.head_groups;
    grid_dependency_wait();                         // lengths and tables may come from the previous kernel
    launch_dependents();                            // the decode grid may launch now; it waits for this grid

    // ---- this thread's sequence and its predecessor (for the prefix-group test):
    // length clamped to [0, max_seq_len], first physical block (-1: empty).  The
    // lengths and the first table entries are loaded together (one round trip);
    // an entry counts only for a non-empty sequence.
    auto first_entry = [&](int s) {
        return a.max_blocks_per_seq > 0 ? __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq) : -1;
    };
    int L = 0, b0 = -1, bp = -1;
    if (t < B) {
        L = __ldg(a.seq_lens + t);
        const int Lp_raw = t > 0 ? __ldg(a.seq_lens + t - 1) : 0;
        const int e0 = first_entry(t);
        const int ep = t > 0 ? first_entry(t - 1) : -1;
        const int Lp = min(max(Lp_raw, 0), a.max_seq_len);
        if (L > a.max_seq_len) {                    // precondition broken: attend over max_seq_len
            if (blockIdx.x == 0) raise_error(a.err, kErrBounds);
            L = a.max_seq_len;
        }
        L = max(L, 0);
        b0 = L > 0 ? e0 : -1;
        bp = Lp > 0 ? ep : -1;
        sGmax[t] = 0;
    }
    // a group starts at a sequence that does not continue its predecessor's first block
    const bool start = t < B && (t == 0 || b0 < 0 || b0 != bp);

    // ---- phase 1: sum and maximum of the lengths, prefix-group scan (group id = its first index)
    long long W = warp_sum(static_cast<long long>(L));
    int lmax = warp_max(L);
    int gid = start ? t : -1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, gid, off);
        if (lane >= off) gid = max(gid, o);
    }
    if (lane == 31) {
        sW[warp] = W;
        sMax[warp] = lmax;
        sScan[warp] = gid;
    }
    __syncthreads();
    W = warp_sum(lane < nw ? sW[lane] : 0ll);
    lmax = warp_max(lane < nw ? sMax[lane] : 0);
    gid = max(gid, warp_max(lane < warp ? sScan[lane] : -1));   // carry from the warps before this one
    if (t < B) atomicMax(&sGmax[gid], L);
    // the caller's sum of the lengths, when given, must be the real one (it sized the grid)
    if (a.sum_seq_lens > 0 && W != a.sum_seq_lens && blockIdx.x == 0 && t == 0) raise_error(a.err, kErrBounds);

    // ---- partition size: the rule's size P0 and its balanced size q0
    const long long slots = a.slots > 0 ? a.slots : 1;
    int P0 = a.part_tokens, q0 = a.part_tokens;
    int cap = a.part_tokens;
    if (a.part_auto) {
        // 0.85 x the positions per slot (an E4M3 position counts 1.4 times)
        const long long p = plan_rule_tokens(W, nh, a.kv8 != 0, slots);
        const int table_cap = dec::kMaxTable * a.block_size;
        cap = max(a.part_tokens, min(table_cap, (lmax + 63) / 64 * 64));
        P0 = static_cast<int>(min(max(p, static_cast<long long>(a.part_tokens)), static_cast<long long>(cap)));
        q0 = lmax > 0 ? balanced(lmax, P0, a.part_tokens) : P0;
    }

    // ---- phase 2: item counts at P0 and q0 (its barrier also completes the group maxima)
    int c0 = warp_sum(t < B ? parts_of(L, P0) : 0);
    int c1 = warp_sum(t < B ? parts_of(L, q0) : 0);
    if (lane == 0) {
        sC0[warp] = c0;
        sC1[warp] = c1;
    }
    __syncthreads();
    const long long n0 = warp_sum(lane < nw ? sC0[lane] : 0);
    const long long n1 = warp_sum(lane < nw ? sC1[lane] : 0);

    int P = P0;
    long long n_live = n0;
    if (a.part_auto) {
        const long long n = n0 * nh;
        // a quarter wave or less past one full wave: take the next size that fits one
        // wave (none can when every sequence alone fills the slots)
        if (n > slots && n * 4 <= slots * 5 && static_cast<long long>(B) * nh <= slots) {
            int nb = 0;
            int q = P0;
            while (q < cap) {
                q = min(q + kGranule, cap);
                if (block_sum(t < B ? parts_of(L, q) : 0, buf[nb]) * nh <= slots) {
                    P = q;
                    break;
                }
                nb ^= 1;
            }
            n_live = P == P0 ? n0 : block_sum(t < B ? parts_of(L, P) : 0, buf[nb ^ 1]);
            nb ^= 1;
            // balance the longest sequence's partitions at the final size
            if (lmax > 0) {
                const int q2 = balanced(lmax, P, a.part_tokens);
                if (q2 < P) {
                    const long long nq = block_sum(t < B ? parts_of(L, q2) : 0, buf[nb ^ 1]);
                    if (nq <= n_live) {
                        P = q2;
                        n_live = nq;
                    }
                }
            }
        } else if (lmax > 0 && q0 < P0 && n1 <= n0) {
            // balance the longest sequence's partitions: the smallest multiple of 64 that still
            // covers it in as many partitions, when that adds no work items (the critical path
            // shortens; more items cost more than they save)
            P = q0;
            n_live = n1;
        }
    }
    // more entries than the grid covers (only a wrong sum_seq_lens does this): the rest are
    // dropped below, and the error word says so
    if (n_live > a.plan_capacity && blockIdx.x == 0 && t == 0) raise_error(a.err, kErrBounds);
    if (t < B) {
        sNp[t] = parts_of(L, P);
        sL[t] = L;
        sOrd[t] = (static_cast<long long>(sGmax[gid]) << 11) | (2047 - t);
    }
    __syncthreads();

    // ---- rank: the items of every sequence ordered before this CTA's sequences
    const int lanes = blockDim.x / kRankSeqs;        // threads per ranked sequence (a power of two)
    const int my = blockIdx.x * kRankSeqs + t / lanes;
    const int sub = t % lanes;
    int off = 0;
    if (my < B) {
        const long long key = sOrd[my];
#pragma unroll 4
        for (int u = sub; u < B; u += lanes) off += sOrd[u] > key ? sNp[u] : 0;
    }
    for (int o = lanes / 2; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
    if (my < B) {
        for (int p = sub; p < sNp[my]; p += lanes) {
            const int y = off + p;
            if (y < a.plan_capacity) a.plan[y] = make_int4(my, p, sL[my], P);
        }
    }

    // ---- padding entries and tickets, spread over every CTA
    const int gt = blockIdx.x * blockDim.x + t, gstride = gridDim.x * blockDim.x;
    for (long long y = n_live + gt; y < a.plan_capacity; y += gstride) a.plan[y] = make_int4(-1, 0, 0, P);
    const long long nt = static_cast<long long>(B) * nh;
    for (long long i = gt; i < nt; i += gstride) a.tickets[i] = 0u;
}

}  // namespace

cudaError_t launch_decode_plan(const DecodeArgs& a, cudaStream_t s) {
    if (a.num_seqs <= 0 || a.num_seqs > kPlanMaxSeqs || !a.plan) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    unsigned threads = kRankSeqs;                   // one per sequence, a power of two >= 64
    while (threads < static_cast<unsigned>(a.num_seqs)) threads *= 2;
    cfg.gridDim = dim3(static_cast<unsigned>((a.num_seqs + kRankSeqs - 1) / kRankSeqs));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, a);
}

}  // namespace pkv
