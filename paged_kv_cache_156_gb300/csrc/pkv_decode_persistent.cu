// paged_attention_decode, persistent variant: same arithmetic as the grid
// kernel (pkv_decode_common.cuh), different scheduling.
//
//  * A one-CTA plan kernel zeroes the work counter and the merge tickets and
//    writes the call's work items, (sequence, partition) pairs, sorted by size
//    (chunks of 64 positions) largest first with a counting sort; empty
//    sequences get their zero output here.
//  * Decode CTAs stay resident (as many per SM as fit) and pull work units
//    (item, KV-head group) from an atomic counter, largest items first, so the
//    last wave is made of the smallest items.
//  * A scheduler warp claims and resolves the next unit (list entry, sequence
//    length, block-table slice) while the TMA warp streams the current one and
//    bulk-copies each unit's query rows into shared memory with its first
//    chunk, so a CTA pays no start-up latency between units.
//  * Shared memory is almost all ring (each stage's K and V contiguous): the
//    consumers keep the stage of a unit's last chunk and use it as the
//    epilogue's scratch, releasing it afterwards, so the other stages keep
//    streaming the next unit meanwhile.
#include <stdlib.h>

#include "pkv_decode_common.cuh"

namespace pkv {

namespace {

using dec::Geo;
using dec::kHeadsPerCta;
using dec::kMaxTable;

constexpr int kPartBits = 9;                     // item = sequence << 9 | partition (partition < 512)
constexpr int kPlanThreads = 1024;
constexpr int kMaxBuckets = 4096 / 64;           // chunk-count buckets (partition <= 4096 positions)
constexpr int kFirst = 1, kLast = 2;

// ---------------------------------------------------------------- plan kernel
template <typename T, int D>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const DecodeArgs a) {
    __shared__ unsigned hist[kMaxBuckets];
    __shared__ unsigned cursor[kMaxBuckets];
    const int tid = threadIdx.x;
    const int P = a.part_tokens;
    const int nbk = P / 64;                      // items have 1..nbk chunks of 64
    const int64_t ntk = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * a.head_groups;
    for (int64_t i = tid; i < ntk; i += kPlanThreads) a.tickets[i] = 0u;
    if (tid == 0) *a.work_counter = 0u;
    for (int b = tid; b < kMaxBuckets; b += kPlanThreads) hist[b] = 0u;
    __syncthreads();
    for (int s = tid; s < a.num_seqs; s += kPlanThreads) {
        const int L = a.seq_lens[s];
        if (L <= 0) continue;
        const int nfull = L / P, rem = L - nfull * P;
        if (nfull) atomicAdd(&hist[nbk - 1], static_cast<unsigned>(nfull));
        if (rem) atomicAdd(&hist[(rem - 1) / 64], 1u);
    }
    __syncthreads();
    if (tid == 0) {
        unsigned acc = 0;
        for (int b = nbk - 1; b >= 0; --b) {
            cursor[b] = acc;
            acc += hist[b];
        }
        *a.n_items = acc;
    }
    __syncthreads();
    T* out = reinterpret_cast<T*>(a.out);
    for (int s = tid; s < a.num_seqs; s += kPlanThreads) {
        const int L = a.seq_lens[s];
        if (L <= 0) {                            // empty sequence: zeros for every head
            uint4* o = reinterpret_cast<uint4*>(out + static_cast<int64_t>(s) * a.num_heads * D);
            for (int i = 0; i < a.num_heads * D * 2 / 16; ++i) o[i] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const int nfull = L / P, rem = L - nfull * P;
        for (int j = 0; j < nfull; ++j) {
            const unsigned pos = atomicAdd(&cursor[nbk - 1], 1u);
            a.items[pos] = (static_cast<unsigned>(s) << kPartBits) | static_cast<unsigned>(j);
        }
        if (rem) {
            const unsigned pos = atomicAdd(&cursor[(rem - 1) / 64], 1u);
            a.items[pos] = (static_cast<unsigned>(s) << kPartBits) | static_cast<unsigned>(nfull);
        }
    }
}

// ---------------------------------------------------------------- persistent decode kernel
// Descriptor of the chunk a ring stage holds; written by the producer before
// it arms the stage, read by the consumers after the stage's wait.
struct ChunkInfo {
    int s;        // sequence; -1 marks the end of the work
    int hh;       // KV head * head_groups + query-head group
    int part;     // partition index
    int nvalid;   // positions of the chunk below seq_len
    int flags;    // kFirst / kLast chunk of its unit
    int nparts;   // partitions of the sequence
    int tok0w;    // position of the chunk's first row
    int L;        // sequence length
};

template <int D, int CW, int STAGES>
struct PSmem {
    using G = Geo<D, CW>;
    static constexpr size_t kQSlot = kHeadsPerCta * D * 2;          // query rows of one unit
    static constexpr size_t kStagePair = 2 * G::kStage;             // K then V of one stage, contiguous
    static constexpr size_t kRing = STAGES * kStagePair;
    static_assert(size_t(G::kScratch) <= kStagePair, "the epilogue scratch lives in one held stage");
    static constexpr size_t kQ = kRing;
    static constexpr size_t kInfo = kQ + STAGES * kQSlot;
    static constexpr size_t kBars = kInfo + STAGES * sizeof(ChunkInfo);
    static constexpr size_t kTable = kBars + (2 * STAGES + 1) * sizeof(uint64_t);   // two table slices
    static constexpr size_t kQueue = kTable + 2 * kMaxTable * sizeof(int);              // two resolved units
    static constexpr size_t kQBars = kQueue + 2 * 8 * sizeof(int);                       // their full/empty barriers
    static constexpr size_t kMisc = kQBars + 4 * sizeof(uint64_t);
    static constexpr size_t kBytes = kMisc + 16;
};

// Threads of the persistent kernel: consumers, the TMA warp, the scheduler warp.
template <int D, int CW>
constexpr int persistent_threads() { return Geo<D, CW>::kThreads + 32; }

template <typename T, int D, int CW, int STAGES>
__global__ void __launch_bounds__(persistent_threads<D, CW>()) decode_persistent_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
    using G = Geo<D, CW>;
    using S = PSmem<D, CW, STAGES>;
    constexpr int kChunk = G::kChunk;
    constexpr int kConsumers = G::kConsumers;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* qslots = smem + S::kQ;
    ChunkInfo* info = reinterpret_cast<ChunkInfo*>(smem + S::kInfo);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
    uint64_t* empty = full + STAGES;
    uint64_t* epi = empty + STAGES;
    int* tbl = reinterpret_cast<int*>(smem + S::kTable);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc);
    volatile int* merge_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NH = a.num_kv_heads * a.head_groups;
    const int bs = a.block_size;
    const int P = a.part_tokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CW);
        }
        mbar_init(epi, kConsumers);
        uint64_t* qb = reinterpret_cast<uint64_t*>(smem + S::kQBars);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qb[i], 32);                // queue slot i filled (every scheduler lane)
            mbar_init(&qb[2 + i], 1);             // queue slot i consumed (TMA warp)
        }
        const bool misaligned = (smem_u32(smem) & 1023u) != 0;
        if (misaligned) raise_error(a.err, kErrTimeout);
        *abort_flag = misaligned;
        *merge_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    int* qdesc = reinterpret_cast<int*>(smem + S::kQueue);       // [2][8]: s, hh, part, L, valid
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + S::kQBars);
    uint64_t* qempty = qfull + 2;

    // ================================================================ scheduler warp
    // Claims one work unit at a time from the atomic counter and resolves it
    // (item entry -> sequence length and block-table slice) into the free slot
    // of a two-slot queue.  A slot frees when the TMA warp has issued the unit
    // it held, so a unit is claimed about one unit ahead of its use: late
    // enough to balance, early enough to hide the dependent loads.
    if (warp == CW + 1) {
        const unsigned units = *a.n_items * static_cast<unsigned>(NH);
        for (unsigned j = 0;; ++j) {
            const int slot = j & 1;
            if (!dec::wait_or_abort(&qempty[slot], ((j >> 1) & 1) ^ 1, abort_flag)) {
                if (lane == 0) dec::raise_abort(a.err, abort_flag);
                break;
            }
            unsigned v = 0;
            if (lane == 0) v = atomicAdd(a.work_counter, 1u);
            v = __shfl_sync(0xffffffffu, v, 0);
            int* d = qdesc + slot * 8;
            if (v >= units) {
                if (lane == 0) d[4] = 0;
                __syncwarp();
                mbar_arrive(&qfull[slot]);
                break;
            }
            const unsigned it = __ldg(a.items + v / NH);
            const int su = static_cast<int>(it >> kPartBits);
            const int pu = static_cast<int>(it & ((1u << kPartBits) - 1));
            const int first = pu * P / bs;
            const int tcount = min(P / bs, a.max_blocks_per_seq - first);
            const int32_t* row = a.block_tables + static_cast<int64_t>(su) * a.max_blocks_per_seq + first;
            const int L = __ldg(a.seq_lens + su);
            const int nblk = min(tcount, (min(L, pu * P + P) - pu * P + bs - 1) / bs);
            for (int i = lane; i < nblk; i += 32) {
                int b = __ldg(row + i);
                if (b < 0 || static_cast<int64_t>(b) >= a.num_blocks) {
                    raise_error(a.err, kErrBounds);
                    b = -1;                       // outside the tensor map: TMA fills zeros, reads nothing
                }
                tbl[slot * kMaxTable + i] = b;
            }
            if (lane == 0) {
                d[0] = su;
                d[1] = static_cast<int>(v % NH);
                d[2] = pu;
                d[3] = L;
                d[4] = 1;
            }
            __syncwarp();
            mbar_arrive(&qfull[slot]);            // every lane releases its table entries and the descriptor
        }
        return;
    }

    // ================================================================ TMA warp
    // Takes resolved units from the queue and streams their chunks into the ring.
    if (warp == CW) {
        if (lane != 0) return;
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        unsigned c = 0;                                            // chunks handed over
        for (unsigned j = 0; !*abort_flag; ++j) {
            const int slot = j & 1;
            if (!dec::wait_or_abort(&qfull[slot], (j >> 1) & 1, abort_flag)) {
                dec::raise_abort(a.err, abort_flag);
                break;
            }
            const int* d = qdesc + slot * 8;
            if (!d[4]) break;
            const int s = d[0], hh = d[1], part = d[2], L = d[3];
            const int start = part * P;
            const int end = min(L, start + P);
            const int nparts = (L + P - 1) / P;
            const int nch = (end - start + kChunk - 1) / kChunk;
            const int hg = hh % a.head_groups;
            const int kvh = hh / a.head_groups;
            const int h0 = kvh * a.qgroup + hg * kHeadsPerCta;   // one query token: rows are heads
            const int gc = min(kHeadsPerCta, a.group - hg * kHeadsPerCta);
            const int per_chunk = kChunk / bs;
            const int* tb = tbl + slot * kMaxTable;
            for (int ci = 0; ci < nch; ++ci, ++c) {
                const int st = c % STAGES;
                const unsigned ph = (c / STAGES) & 1;
                if (!dec::wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                    dec::raise_abort(a.err, abort_flag);
                    break;
                }
                const int tok0 = start + ci * kChunk;
                const int nv = min(kChunk, end - tok0);
                const int nb = (nv + bs - 1) / bs;
                ChunkInfo& in = info[st];
                in.s = s;
                in.hh = hh;
                in.part = part;
                in.nvalid = nv;
                in.flags = (ci == 0 ? kFirst : 0) | (ci == nch - 1 ? kLast : 0);
                in.nparts = nparts;
                in.tok0w = tok0;
                in.L = L;
                const unsigned qbytes = ci == 0 ? static_cast<unsigned>(gc * D * 2) : 0u;
                mbar_arrive_expect_tx(&full[st], static_cast<unsigned>(nb * bs * D * 2 * 2) + qbytes);
                if (ci == 0)
                    bulk_copy_g2s(qslots + st * S::kQSlot,
                                  reinterpret_cast<const T*>(a.q) + (static_cast<int64_t>(s) * a.num_heads + h0) * D,
                                  qbytes, &full[st]);
                for (int jb = 0; jb < nb; ++jb) {
                    const int pb = tb[ci * per_chunk + jb];
#pragma unroll
                    for (int hf = 0; hf < G::kHalves; ++hf) {
                        uint8_t* kdst = smem + st * S::kStagePair + hf * G::kPlane + jb * bs * 128;
                        tma_load_4d(kdst, &tmk, hf * 64, kvh, 0, pb, &full[st]);
                        tma_load_4d(kdst + G::kStage, &tmv, hf * 64, kvh, 0, pb, &full[st]);
                    }
                }
            }
            mbar_arrive(&qempty[slot]);                            // the slot's table is no longer read
        }
        // end marker: one more stage carrying s = -1
        if (!*abort_flag) {
            const int st = c % STAGES;
            const unsigned ph = (c / STAGES) & 1;
            if (dec::wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                info[st].s = -1;
                mbar_arrive(&full[st]);
            } else {
                dec::raise_abort(a.err, abort_flag);
            }
        }
        return;
    }

    // ================================================================ consumer warps
    dec::WarpState<D> ws;
    unsigned c = 0;
    unsigned epi_uses = 0;
    auto epi_sync = [&]() -> bool {               // all consumer threads, bounded
        mbar_arrive(epi);
        const bool r = dec::wait_or_abort(epi, epi_uses & 1, abort_flag);
        ++epi_uses;
        return r;
    };
    for (;;) {
        const int st = c % STAGES;
        const unsigned ph = (c / STAGES) & 1;
        bool got = dec::wait_or_abort(&full[st], ph, abort_flag);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
            if (lane == 0) dec::raise_abort(a.err, abort_flag);
            break;
        }
        const ChunkInfo ci = info[st];
        if (ci.s < 0) break;
        ++c;
        const int hg = ci.hh % a.head_groups;
        const int kvh = ci.hh / a.head_groups;
        const int vh0 = hg * kHeadsPerCta;
        const int gc = min(kHeadsPerCta, a.group - vh0);
        const int64_t sh0 = dec::item_row0<false>(a, ci.s, kvh, vh0);
        if (ci.flags & kFirst) {
            // Q^T fragments from the unit's query rows (rows of absent heads are zero)
            const uint32_t* qs = reinterpret_cast<const uint32_t*>(qslots + st * S::kQSlot);
            const int n = lane >> 2;
            const int kq = (lane & 3) * 2;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                ws.qb[ks][0] = n < gc ? qs[(n * D + ks * 16 + kq) / 2] : 0u;
                ws.qb[ks][1] = n < gc ? qs[(n * D + ks * 16 + 8 + kq) / 2] : 0u;
            }
            dec::reset_state(ws);
        }
        const int nv = min(16, ci.nvalid - warp * 16);
        uint8_t* stage = smem + st * S::kStagePair;
        if (nv > 0)
            dec::consume_chunk<T, D, CW, false>(ws, smem_u32(stage), smem_u32(stage + G::kStage), nv, warp, lane,
                                         a.scale_log2, ci.tok0w + warp * 16, ci.L, ci.L);
        __syncwarp();
        if (!(ci.flags & kLast)) {
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }

        // ---- unit epilogue in the held stage (the other stages stream the next unit)
        float* scratch = reinterpret_cast<float*>(stage);
        if (!epi_sync()) break;                   // every warp is done reading this stage
        dec::warp_state_to_smem<D, CW>(ws, scratch, warp, lane);
        if (!epi_sync()) break;
        dec::combine_warps<T, D, CW, false>(a, scratch, sh0, ci.s, kvh, vh0, gc, ci.part, ci.nparts, threadIdx.x);
        if (ci.nparts > 1) {
            // the group barrier orders every thread's partial writes before thread
            // 0's gpu-scope fence, which releases them all before the ticket
            if (!epi_sync()) break;
            if (threadIdx.x == 0) {
                __threadfence();
                const unsigned t = atomicAdd(a.tickets + static_cast<int64_t>(ci.s) * NH + ci.hh, 1u);
                __threadfence();
                *merge_flag = (t == static_cast<unsigned>(ci.nparts - 1));
            }
            if (!epi_sync()) break;
            if (*merge_flag) {
                if (!dec::merge_partitions<T, D, CW, false>(a, scratch, sh0, ci.s, kvh, vh0, gc, ci.nparts, warp, lane,
                                                           threadIdx.x, epi_sync))
                    break;
            }
        }
        if (!epi_sync()) break;                   // scratch and flag are read: release the stage
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (*abort_flag) {
        // give copies still in flight a bounded moment to land before the CTA exits
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 10000000ull) __nanosleep(100000);
    }
}

template <typename T, int D, int CW, int STAGES>
cudaError_t launch_p(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    constexpr size_t smem = PSmem<D, CW, STAGES>::kBytes;
    static_assert(smem <= 232448, "shared memory budget");
    auto kern = decode_persistent_kernel<T, D, CW, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, persistent_threads<D, CW>(), smem)) != cudaSuccess)
        return e;
    plan_kernel<T, D><<<1, kPlanThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.head_groups * a.max_parts * a.num_seqs;
    int64_t grid = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    if (grid > units) grid = units;
    kern<<<static_cast<unsigned>(grid), persistent_threads<D, CW>(), smem, s>>>(tmk, tmv, a);
    return cudaGetLastError();
}

int env_int(const char* name, int dflt) {
    const char* e = getenv(name);
    return e ? atoi(e) : dflt;
}

template <typename T, int D>
cudaError_t launch_p_cfg(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    static const int cw = env_int("PKV_DECODE_WARPS", 4) == 2 ? 2 : 4;
    static const int st = env_int("PKV_DECODE_STAGES", 3) == 2 ? 2 : 3;
    if (cw == 2) return st == 3 ? launch_p<T, D, 2, 3>(a, tmk, tmv, s) : launch_p<T, D, 2, 2>(a, tmk, tmv, s);
    return st == 3 ? launch_p<T, D, 4, 3>(a, tmk, tmv, s) : launch_p<T, D, 4, 2>(a, tmk, tmv, s);
}

}  // namespace

cudaError_t launch_decode_persistent(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                                     int head_dim, cudaStream_t s) {
    if (a.num_seqs <= 0) return cudaSuccess;
    if (dtype == 0)
        return head_dim == 128 ? launch_p_cfg<__half, 128>(a, tmk, tmv, s) : launch_p_cfg<__half, 64>(a, tmk, tmv, s);
    return head_dim == 128 ? launch_p_cfg<__nv_bfloat16, 128>(a, tmk, tmv, s)
                           : launch_p_cfg<__nv_bfloat16, 64>(a, tmk, tmv, s);
}

}  // namespace pkv
