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
//    automatic size, a kernel-specific fraction of the positions per resident
//    CTA slot (sum_s L_s * KV head groups / slots: 0.85 of it for the 16-bit
//    decode kernel, 1.2 for an E4M3 pool, whose positions are half the bytes,
//    1.1 for the tensor-core verify kernel), in multiples of 512, capped by the
//    longest sequence and by the staged table, raised when the item count
//    would spill a quarter wave or less past one full wave, then shrunk to
//    the smallest multiple of 64 that splits the longest sequence into as
//    many partitions when that adds no work items (equal partitions on the
//    critical path);
//  * order: groups of adjacent sequences that share their first physical
//    block (forks of one prompt, "LLM 推理引擎内部原理" §3.3) stay together, so
//    their shared prefix is read while it is still in L2; groups are ordered
//    by their longest member, longest first, ties by sequence index;
//  * shared-prefix units (when the call allows them): a sequence whose first
//    block is its predecessor's has its table row compared with the
//    predecessor's, entry by entry (a warp per pair, four pairs in flight),
//    giving the run of leading blocks the two share.  Runs of sequences that
//    share at least kUnitMinShare positions with their predecessor are cut
//    into units of at most 8 / (query heads per KV head) members, each unit
//    with at most as many partitions (at the host's smallest partition size)
//    as the workspace holds per sequence.  A unit is one work item per
//    partition of its stream: the shared prefix (the members' common blocks,
//    up to the shortest member's length) once, then each member's blocks
//    past the prefix, every segment starting on a block boundary.  Its items
//    are written at its first sequence, with the member count and the
//    shared length; the size rule still uses the lengths' sum, so the grid
//    bound the host derives from it holds;
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

// Stream positions of a unit: the shared prefix (ceil(sh / bs) blocks), then
// each member whose length exceeds sh from block floor(sh / bs) to its last
// block.  With one member it is the member's length.
__device__ __forceinline__ int unit_stream(const int* len, int n, int sh, int bs) {
    if (n == 1) return len[0];
    const int fb = sh / bs;
    int blocks = (sh + bs - 1) / bs;
    for (int j = 0; j < n; ++j)
        if (len[j] > sh) blocks += (len[j] + bs - 1) / bs - fb;
    return blocks * bs;
}

__global__ void __launch_bounds__(kPlanMaxSeqs) plan_kernel(const DecodeArgs a) {
    __shared__ int sGmax[kPlanMaxSeqs];             // per group start: the group's longest length
    __shared__ int sNp[kPlanMaxSeqs];               // partitions of each work unit (0: not a unit's first)
    __shared__ int sL[kPlanMaxSeqs];                // lengths, clamped to [0, max_seq_len]
    __shared__ int sT[kPlanMaxSeqs];                // stream length of the unit a sequence starts
    __shared__ int sUn[kPlanMaxSeqs];               // members of the unit a sequence starts (0: a member)
    __shared__ int sUsh[kPlanMaxSeqs];              // shared prefix length of that unit
    __shared__ int sCrun[kPlanMaxSeqs];             // leading table entries equal to the predecessor's
    __shared__ long long sOrd[kPlanMaxSeqs];        // order key: group length << 11 | (2047 - index)
    __shared__ long long sW[kMaxWarps];             // per warp: sum of lengths
    __shared__ int sMax[kMaxWarps], sScan[kMaxWarps], sC0[kMaxWarps], sC1[kMaxWarps], sC2[kMaxWarps];
    __shared__ long long buf[2][kMaxWarps];         // the rare search's reductions
    __shared__ int sJn;                             // joined sequences listed (in sNp, before it is used)
    const int B = a.num_seqs;
    const int bs = a.block_size;
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
        sL[t] = L;
    }
    // a group starts at a sequence that does not continue its predecessor's first block
    const bool start = t < B && (t == 0 || b0 < 0 || b0 != bp);
    // a sequence that may join its predecessor's unit
    const int max_members = a.units ? dec::kHeadsPerCta / max(a.qgroup, 1) : 1;
    const bool joined = max_members > 1 && t < B && !start;

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
    if (t == 0) sJn = 0;
    const int any_joined = __syncthreads_or(joined);
    W = warp_sum(lane < nw ? sW[lane] : 0ll);
    lmax = warp_max(lane < nw ? sMax[lane] : 0);
    gid = max(gid, warp_max(lane < warp ? sScan[lane] : -1));   // carry from the warps before this one
    if (t < B) atomicMax(&sGmax[gid], L);
    // the caller's sum of the lengths, when given, must be the real one (it sized the grid)
    if (a.sum_seq_lens > 0 && W != a.sum_seq_lens && blockIdx.x == 0 && t == 0) raise_error(a.err, kErrBounds);

    // ---- shared-prefix units (only when some sequence continues its predecessor's first block)
    bool lead = t < B;                              // this thread's sequence starts a work unit
    int Tu = L;                                     // the unit's stream length
    int lmax_u = lmax;
    if (any_joined) {
        if (t < B) {
            sCrun[t] = 0;
            sUn[t] = 1;
            sT[t] = L;
            sUsh[t] = L;
        }
        // leading equal entries of the rows of each joined sequence and its predecessor:
        // the joined sequences are listed, then every warp takes four at a time, a
        // lane comparing four entries of each pair (16-byte loads when the rows allow)
        int* sJ = sNp;                              // the list (sNp is written after this phase)
        const unsigned jm = __ballot_sync(0xffffffffu, joined);
        int jbase = 0;
        if (lane == 0 && jm) jbase = atomicAdd(&sJn, __popc(jm));
        jbase = __shfl_sync(0xffffffffu, jbase, 0);
        if (joined) sJ[jbase + __popc(jm & ((1u << lane) - 1u))] = t;
        __syncthreads();
        const int nj = sJn;
        const int64_t Wt = a.max_blocks_per_seq;
        const bool vec = (Wt & 3) == 0 && (reinterpret_cast<uintptr_t>(a.block_tables) & 15u) == 0;
        constexpr int kPairs = 4;
        for (int base = warp * kPairs; base < nj; base += nw * kPairs) {
            int tk[kPairs], first[kPairs];
            int mm = 0;
#pragma unroll
            for (int k = 0; k < kPairs; ++k) {
                tk[k] = base + k < nj ? sJ[base + k] : -1;
                first[k] = tk[k] >= 0 ? min((sL[tk[k] - 1] + bs - 1) / bs, (sL[tk[k]] + bs - 1) / bs) : 0;
                mm = max(mm, first[k]);
            }
            for (int e0 = 0; e0 < mm; e0 += 128) {
                const int j = e0 + 4 * lane;            // this lane's four entries
                int4 xa[kPairs], xb[kPairs];
#pragma unroll
                for (int k = 0; k < kPairs; ++k) {
                    xa[k] = xb[k] = make_int4(0, 0, 0, 0);
                    if (j < first[k]) {
                        const int32_t* ra = a.block_tables + static_cast<int64_t>(tk[k] - 1) * Wt + j;
                        const int32_t* rb = a.block_tables + static_cast<int64_t>(tk[k]) * Wt + j;
                        if (vec) {                      // j + 3 < Wt: Wt is a multiple of 4
                            xa[k] = __ldg(reinterpret_cast<const int4*>(ra));
                            xb[k] = __ldg(reinterpret_cast<const int4*>(rb));
                        } else {
                            const int n = min(4, first[k] - j);
                            xa[k].x = __ldg(ra);
                            xb[k].x = __ldg(rb);
                            if (n > 1) { xa[k].y = __ldg(ra + 1); xb[k].y = __ldg(rb + 1); }
                            if (n > 2) { xa[k].z = __ldg(ra + 2); xb[k].z = __ldg(rb + 2); }
                            if (n > 3) { xa[k].w = __ldg(ra + 3); xb[k].w = __ldg(rb + 3); }
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < kPairs; ++k) {
                    // first differing entry of this lane's four that lies before first[k]
                    unsigned d = 0x7fffffffu;
                    if (xa[k].w != xb[k].w && j + 3 < first[k]) d = j + 3;
                    if (xa[k].z != xb[k].z && j + 2 < first[k]) d = j + 2;
                    if (xa[k].y != xb[k].y && j + 1 < first[k]) d = j + 1;
                    if (xa[k].x != xb[k].x && j < first[k]) d = j;
                    first[k] = min(first[k], static_cast<int>(__reduce_min_sync(0xffffffffu, d)));
                }
            }
            if (lane == 0)
#pragma unroll
                for (int k = 0; k < kPairs; ++k)
                    if (tk[k] >= 0) sCrun[tk[k]] = first[k];
        }
        __syncthreads();
        // positions sequence u shares with its predecessor (0: not joined)
        auto share = [&](int u) {
            return sCrun[u] > 0 ? min(sCrun[u] * bs, min(sL[u - 1], sL[u])) : 0;
        };
        auto linked = [&](int u) { return u < B && u > 0 && share(u) >= kUnitMinShare; };
        // the first sequence of each run of linked sequences cuts the run into units
        if (t < B && !linked(t) && linked(t + 1)) {
            int u0 = t;
            for (;;) {
                int len[dec::kHeadsPerCta];
                len[0] = sL[u0];
                int n = 1, sh = sL[u0], T = sL[u0];
                while (n < max_members && linked(u0 + n)) {
                    len[n] = sL[u0 + n];
                    const int sh2 = min(sh, share(u0 + n));
                    const int T2 = unit_stream(len, n + 1, sh2, bs);
                    if ((T2 + a.part_tokens - 1) / a.part_tokens > a.max_parts) break;
                    sh = sh2;
                    T = T2;
                    ++n;
                }
                sUn[u0] = n;
                sT[u0] = T;
                sUsh[u0] = sh;
                for (int j = 1; j < n; ++j) sUn[u0 + j] = 0;
                u0 += n;
                if (!linked(u0)) break;             // the run ended
            }
        }
        __syncthreads();
        lead = t < B && sUn[t] > 0;
        Tu = lead ? sT[t] : 0;
        const int mu = warp_max(Tu);
        if (lane == 0) sMax[warp] = mu;
        __syncthreads();
        lmax_u = warp_max(lane < nw ? sMax[lane] : 0);
    }

    // ---- partition size: the rule's size P0 and its balanced size q0
    const long long slots = a.slots > 0 ? a.slots : 1;
    int P0 = a.part_tokens, q0 = a.part_tokens;
    int cap = a.part_tokens;
    if (a.part_auto) {
        // the kernel's share of the positions per slot (plan_rule_tokens), from the lengths' sum
        const long long p = plan_rule_tokens(W, nh, a.rule_weight, slots);
        const int table_cap = dec::kMaxTable * bs;
        cap = max(a.part_tokens, min(table_cap, (lmax_u + 63) / 64 * 64));
        P0 = static_cast<int>(min(max(p, static_cast<long long>(a.part_tokens)), static_cast<long long>(cap)));
        q0 = lmax_u > 0 ? balanced(lmax_u, P0, a.part_tokens) : P0;
    }

    // ---- phase 2: item counts at P0 and q0, and the unit count (its barrier also
    // completes the group maxima)
    int c0 = warp_sum(lead ? parts_of(Tu, P0) : 0);
    int c1 = warp_sum(lead ? parts_of(Tu, q0) : 0);
    int c2 = warp_sum(lead ? 1 : 0);
    if (lane == 0) {
        sC0[warp] = c0;
        sC1[warp] = c1;
        sC2[warp] = c2;
    }
    __syncthreads();
    const long long n0 = warp_sum(lane < nw ? sC0[lane] : 0);
    const long long n1 = warp_sum(lane < nw ? sC1[lane] : 0);
    const long long nunits = warp_sum(lane < nw ? sC2[lane] : 0);

    int P = P0;
    long long n_live = n0;
    if (a.part_auto) {
        const long long n = n0 * nh;
        // a quarter wave or less past one full wave: take the next size that fits one
        // wave (none can when every unit alone fills the slots)
        if (n > slots && n * 4 <= slots * 5 && nunits * nh <= slots) {
            int nb = 0;
            int q = P0;
            while (q < cap) {
                q = min(q + kGranule, cap);
                if (block_sum(lead ? parts_of(Tu, q) : 0, buf[nb]) * nh <= slots) {
                    P = q;
                    break;
                }
                nb ^= 1;
            }
            n_live = P == P0 ? n0 : block_sum(lead ? parts_of(Tu, P) : 0, buf[nb ^ 1]);
            nb ^= 1;
            // balance the longest unit's partitions at the final size
            if (lmax_u > 0) {
                const int q2 = balanced(lmax_u, P, a.part_tokens);
                if (q2 < P) {
                    const long long nq = block_sum(lead ? parts_of(Tu, q2) : 0, buf[nb ^ 1]);
                    if (nq <= n_live) {
                        P = q2;
                        n_live = nq;
                    }
                }
            }
        } else if (lmax_u > 0 && q0 < P0 && n1 <= n0) {
            // balance the longest unit's partitions: the smallest multiple of 64 that still
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
        sNp[t] = lead ? parts_of(Tu, P) : 0;
        sT[t] = Tu;
        if (!any_joined) {
            sUn[t] = 1;
            sUsh[t] = L;
        }
        sOrd[t] = (static_cast<long long>(sGmax[gid]) << 11) | (2047 - t);
    }
    __syncthreads();

    // ---- rank: the items of every unit ordered before this CTA's units
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
            if (y < a.plan_capacity) {
                a.plan[kPlanEntryInts * y] = make_int4(my, p, sT[my], P);
                // (members, shared length, lengths of the first two members)
                a.plan[kPlanEntryInts * y + 1] =
                    make_int4(sUn[my], sUsh[my], sL[my], sUn[my] > 1 ? sL[my + 1] : 0);
            }
        }
    }

    // ---- padding entries and tickets, spread over every CTA
    const int gt = blockIdx.x * blockDim.x + t, gstride = gridDim.x * blockDim.x;
    for (long long y = n_live + gt; y < a.plan_capacity; y += gstride) {
        a.plan[kPlanEntryInts * y] = make_int4(-1, 0, 0, P);
        a.plan[kPlanEntryInts * y + 1] = make_int4(0, 0, 0, 0);
    }
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
