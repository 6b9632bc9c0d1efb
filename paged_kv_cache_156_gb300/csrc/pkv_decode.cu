// paged_attention_decode: one query token per sequence over its paged K/V.
//
// What is computed ("tbr8.org PagedAttention article" §2.2; "LLM 推理引擎内部原理"
// §2.4): for each sequence s and query head h, walk the logical blocks of s,
// look each one up in the block table, read K/V rows of KV head
// g = h / group up to seq_len, and return softmax(scale * q.K) V.
//
// How (sm_103a):
//  * One CTA per work item = (KV head, group of <= 8 query heads sharing it,
//    partition of P positions, sequence).  All query heads of a KV head are
//    served from the same K/V bytes, so every byte of the pool is read from
//    HBM once per step.  Two or three CTAs share an SM so one CTA's start-up
//    (table and q fetch, first loads in flight) hides behind the others'
//    streaming.  The items come from the plan kernel's work list (only the
//    partitions that exist, long sequences first, P chosen from the batch's
//    lengths); a batch too large to plan runs the full grid instead, whose
//    CTAs past their sequence's end return at once.
//  * The CTA's slice of the block table is staged in shared memory once; a
//    producer warp then streams the partition's K and V tiles with TMA
//    (cp.async.bulk.tensor; one box = one (physical block, KV head) tile of
//    block_size rows x 64 elements, 128B-swizzled, loaded with an L2
//    evict-first policy: K/V bytes are read once per step) into a ring of
//    STAGES chunks of 64 positions, handing each chunk over with an mbarrier.
//  * With the step's slot write fused in (pkv_paged_kv_append_decode), the
//    producer warp of the CTA that holds position seq_len - 1 first stores
//    the sequence's new K and V rows for its KV head into that slot (after
//    checking the slot against the table) and fences them against its own
//    tile loads ("LLM 推理引擎内部原理" §2.3: append_slot gives the slot).
//  * Four consumer warps each own 16 positions of every chunk.  Scores are a
//    small dense contraction over the query-head group, done on the tensor
//    cores with keys as the M dimension: S^T[16 pos x 8 heads] = K Q^T
//    (mma.m16n8k16, fp32 accumulate).  Each warp keeps an fp32 online softmax
//    (running max and sum per head, log2 domain), rounds the weights to the
//    input type, transposes them in registers (movmatrix) and accumulates
//    O^T[d x 8 heads] += V^T P^T on the tensor cores.
//  * Positions past seq_len are masked: their scores become -inf and their V
//    rows in shared memory are zeroed (the slots hold no token and may be
//    NaN), so nothing beyond seq_len contributes.
//  * After the last chunk the four warps' states are merged through shared
//    memory.  A sequence that fits one partition writes its output directly.
//    Otherwise the partition writes (max, sum, unnormalised output) to the
//    workspace and takes a ticket; the CTA that takes the last ticket of its
//    (sequence, head group) merges all partitions in the same launch
//    (split-K over the sequence):
//        M = max_p m_p,  out = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p.
//  * Every wait is an mbarrier wait bounded in wall time; a wait that gives
//    up raises the error word and the CTA winds down.
#include <atomic>
#include <type_traits>

#include "pkv_decode_common.cuh"

namespace pkv {

namespace {

using dec::Geo;
using dec::kHeadsPerCta;
using dec::kMaxTable;

template <int D, int CW, int STAGES, int EB = 2, bool UNITS = false>
struct Smem {
    using G = Geo<D, CW, EB>;
    static constexpr size_t kRing = 2 * STAGES * G::kStage;
    static constexpr size_t kArena = kRing > size_t(G::kScratch) ? kRing : size_t(G::kScratch);  // scratch aliases the ring
    static constexpr size_t kBars = kArena;
    static constexpr size_t kTable = kBars + (2 * STAGES + 1) * sizeof(uint64_t);
    static constexpr size_t kDesc = kTable + kMaxTable * sizeof(int);   // shared-prefix unit: per staged block
    static constexpr size_t kUnit = kDesc + (UNITS ? kMaxTable : 0) * sizeof(int);   // unit layout
    static constexpr size_t kMisc = kUnit + (UNITS ? 2 * kHeadsPerCta + 2 : 0) * sizeof(int);
    static constexpr size_t kBytes = kMisc + 16;
};

// A query pair (two elements of T) as the f16 pair the E4M3 path multiplies with.
template <typename T>
__device__ __forceinline__ uint32_t q_as_f16x2(uint32_t x);
template <>
__device__ __forceinline__ uint32_t q_as_f16x2<__half>(uint32_t x) { return x; }
template <>
__device__ __forceinline__ uint32_t q_as_f16x2<__nv_bfloat16>(uint32_t x) {
    return Mma<__half>::pack(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

// KV8: the pools hold E4M3 codes (head_dim 128); the tensor cores run in f16.
// UNITS: the work list may hold shared-prefix units (16-bit decode only; the
// host launches this form when the plan may make them).
// Register caps: an SM's four sub-partitions each hold a quarter of the register
// file (16384) and take the resident warps in turn, so the 5-warp CTAs that shared
// memory allows 3 to an SM (head_dim 128, 16-bit or E4M3) fit at 128 registers, and
// the 6 of head_dim 64 at 64.
template <typename T, int D, int CW, int STAGES, bool MQ, bool KV8 = false, bool UNITS = false>
__global__ void __maxnreg__(D == 64 ? 64 : 128) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                     const __grid_constant__ CUtensorMap tmv,
                                                                     const DecodeArgs a) {
    static_assert(!KV8 || D == 128, "E4M3 pools: head_dim 128");
    constexpr int kEB = KV8 ? 1 : 2;                // bytes of a pool element
    constexpr bool kUnits = UNITS && !MQ && !KV8;   // shared-prefix units: 16-bit decode
    using G = Geo<D, CW, kEB>;
    using S = Smem<D, CW, STAGES, kEB, kUnits>;
    constexpr int kChunk = G::kChunk;
    constexpr int kConsumers = G::kConsumers;
    constexpr int kThreads = G::kThreads;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* kring = smem;
    uint8_t* vring = smem + STAGES * G::kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
    uint64_t* empty = full + STAGES;
    uint64_t* epi = empty + STAGES;               // consumer-group barrier (all consumer threads)
    int* tbl = reinterpret_cast<int*>(smem + S::kTable);
    // a unit's staged blocks: segment + 1 (0: the shared prefix) | first valid offset << 8 | end offset << 16
    int* udesc = reinterpret_cast<int*>(smem + S::kDesc);
    int* useg = reinterpret_cast<int*>(smem + S::kUnit);   // members' first stream blocks; [members]: the total
    int* ulen = useg + kHeadsPerCta + 1;                   // members' lengths; [kHeadsPerCta]: layout refused
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc);
    volatile int* merge_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the plan and the pools come from earlier kernels; with the caller's guarantee that
    // nothing still running writes them (a.early), the wait moves below the work item,
    // the table slice and the first tile loads, before anything else is read
    if (!a.early) grid_dependency_wait();
    // Work item: from the plan (one entry per (unit, partition), KV head
    // groups innermost in the 1-D grid) or, without one, the 3-D grid itself.
    // A unit is one sequence, or (16-bit decode) `un` adjacent sequences that
    // share their first `ush` positions, whose stream is Lp positions long.
    int hh, part, s, P, Lp;
    int un = 1, ush = 0, ul0 = 0, ul1 = 0;          // (units: the first two members' lengths)
    if (a.plan) {
        const int nh = a.num_kv_heads * a.head_groups;
        const unsigned y = blockIdx.x / static_cast<unsigned>(nh);
        hh = static_cast<int>(blockIdx.x - y * static_cast<unsigned>(nh));
        const int4 it = __ldg(a.plan + kPlanEntryInts * y);
        const int4 iu = __ldg(a.plan + kPlanEntryInts * y + 1);
        s = it.x;
        part = it.y;
        Lp = it.z;
        P = it.w;
        un = iu.x;
        ush = iu.y;
        ul0 = iu.z;
        ul1 = iu.w;
        if (s < 0) return;                          // padding entry
        // a plan made for other batch arguments (a run-only call's misuse): never index out of range
        bool bad = s >= a.num_seqs || part < 0 || Lp < 0 || P < 64 || P > kMaxTable * a.block_size ||
                   part * P >= max(Lp, 1) || (Lp + P - 1) / P > a.max_parts || un < 1;
        if (un == 1)
            bad = bad || Lp > a.max_seq_len;
        else
            bad = bad || !kUnits || un * a.group > kHeadsPerCta || a.head_groups != 1 || s + un > a.num_seqs ||
                  ush < 1 || ush > a.max_seq_len || Lp % a.block_size != 0 ||
                  static_cast<int64_t>(Lp) > static_cast<int64_t>(un) * (a.max_seq_len + a.block_size);
        if (bad) {
            if (threadIdx.x == 0) raise_error(a.err, kErrBounds);
            return;
        }
    } else {
        hh = blockIdx.x;                            // KV head * head_groups + query-head group
        part = blockIdx.y;
        s = blockIdx.z;
        P = a.part_tokens;
        Lp = -1;
    }
    const bool grouped = kUnits && un > 1;          // a shared-prefix unit (CTA-uniform)
    // (CTA-uniform; compiled only into the unit-free 16-bit decode form, the one whole-step
    // batches without forks use)
    const bool early = !kUnits && !MQ && !KV8 && a.early && a.plan && !grouped;
    if (a.early && !early) grid_dependency_wait();
    const int hg = hh % a.head_groups;
    const int kvh = hh / a.head_groups;
    const int vh0 = hg * kHeadsPerCta;                // first query row of this CTA within the KV head's rows
    // columns: the rows of this CTA (a unit's column c is head c % group of member c / group)
    const int gc = grouped ? un * a.group : min(kHeadsPerCta, a.group - vh0);
    const int64_t sh0 = dec::item_row0<MQ>(a, s, kvh, vh0);
    const dec::ItemRows rows{sh0, s, kvh, vh0, grouped ? un : 1};
    const int bs = a.block_size;
    const int start = part * P;
    T* out = reinterpret_cast<T*>(a.out);

    // Issue the loads that depend only on the work item before the sequence
    // length is known: this warp's slice of the block table (producer) or the
    // query fragments (consumers).
    constexpr int kTePerLane = (kMaxTable + 31) / 32;
    int te[kTePerLane];
    dec::WarpState<D> ws;
    const int first_blk = start / bs;
    const int tcount = min(P / bs, a.max_blocks_per_seq - first_blk);
    // Fused slot write: the new token's row (K in the first D/8 lanes, V in the
    // next D/8, 16 bytes each) for a CTA that may hold position seq_len - 1.
    constexpr int kHV = D / 8;
    uint4 nrow = make_uint4(0u, 0u, 0u, 0u);
    int64_t nslot = -1;
    float nscale = 1.0f;
    const bool maybe_put = !MQ && !grouped && a.k_new != nullptr && (Lp <= 0 || part == (Lp + P - 1) / P - 1);
    if (warp == CW) {
        if (!grouped) {                             // (a unit's blocks are staged once its lengths are known)
            const int32_t* row = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + first_blk;
#pragma unroll
            for (int k = 0; k < kTePerLane; ++k) {
                const int i = lane + 32 * k;
                te[k] = (32 * k < tcount && i < tcount) ? __ldg(row + i) : 0;
            }
            if (maybe_put && !early) {              // (early: after the wait, below)
                nslot = __ldg(a.slot_mapping + s);
                if (lane < 2 * kHV) {
                    const uint4* src = lane < kHV ? a.k_new : a.v_new;
                    nrow = __ldg(src + (static_cast<int64_t>(s) * a.num_kv_heads + kvh) * kHV + lane % kHV);
                    if constexpr (KV8) nscale = __ldg((lane < kHV ? a.k_scale : a.v_scale) + kvh);
                }
            }
        }
    } else if constexpr (KV8) {
        // Q^T in consume_chunk_fp8's order: lane holds q[n = lane/4][32*t + 4*ks + {0,1}]
        // and [.. + {2,3}] (t = lane % 4), as f16 (exact for |q| < 65504)
        const int n = lane >> 2;
        const int nq = min(n, gc - 1);
        const T* qrow = reinterpret_cast<const T*>(a.q) + dec::qo_row<MQ>(a, sh0, s, kvh, vh0, nq) * D + 32 * (lane & 3);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(qrow + 4 * ks));
            ws.qb[ks][0] = n < gc ? q_as_f16x2<T>(raw.x) : 0u;
            ws.qb[ks][1] = n < gc ? q_as_f16x2<T>(raw.y) : 0u;
        }
    } else {
        if (early) grid_dependency_wait();          // q comes from the preceding kernel
        // Q^T as the B operand (k = head_dim, n = query head): lane holds
        // q[n = lane/4][k = 16*ks + 2*(lane%4) + {0,1}] and the same at k + 8.
        const int n = lane >> 2;
        const int kq = (lane & 3) * 2;
        const int nq = min(n, gc - 1);      // lanes of absent rows read a present row, then drop it
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(a.q) +
                                                                 rows.out<MQ>(a, nq) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            ws.qb[ks][0] = n < gc ? __ldg(qrow + (ks * 16 + kq) / 2) : 0u;
            ws.qb[ks][1] = n < gc ? __ldg(qrow + (ks * 16 + 8 + kq) / 2) : 0u;
        }
    }

    int L = Lp;
    if (Lp < 0) {
        L = __ldg(a.seq_lens + s);
        if (L > a.max_seq_len) {                    // precondition broken: attend over max_seq_len
            if (threadIdx.x == 0 && part == 0 && hh == 0) raise_error(a.err, kErrBounds);
            L = a.max_seq_len;
        }
    }
    if (L <= 0) {                                   // empty sequence: zeros
        // a fused slot write needs a position for its token
        if (maybe_put && warp == CW && lane == 0 && part == 0 && hh == 0 && nslot >= 0) raise_error(a.err, kErrBounds);
        if (part == 0)
            for (int i = threadIdx.x; i < gc * D; i += kThreads)
                out[dec::qo_row<MQ>(a, sh0, s, kvh, vh0, i / D) * D + i % D] = T(0.0f);
        return;
    }
    if (start >= L) return;                         // partition past the end of this sequence
    const int end = min(L, start + P);
    const int nparts = (L + P - 1) / P;
    const int nchunks = (end - start + kChunk - 1) / kChunk;
    const int lbs = 31 - __clz(bs);                 // block sizes are powers of two
    const int sb0 = start >> lbs;                   // a unit's first stream block of this partition
    const int nblk = (end - start + bs - 1) >> lbs;
    // a unit's fused slot writes: member `lane`'s slot, and the new rows of its first
    // two members (lanes < 2 * D / 8), loaded with its lengths (they depend on nothing else)
    constexpr int kUnitRows = 2;
    int64_t uslot = -1;
    uint4 urow[kUnitRows];
#pragma unroll
    for (int j = 0; j < kUnitRows; ++j) urow[j] = make_uint4(0u, 0u, 0u, 0u);

    if (grouped && warp == CW) {
        if (a.k_new != nullptr) {
            if (lane < un) uslot = __ldg(a.slot_mapping + s + lane);
            if (lane < 2 * kHV) {
                const uint4* src = lane < kHV ? a.k_new : a.v_new;
#pragma unroll
                for (int j = 0; j < kUnitRows; ++j)
                    if (j < un) urow[j] = __ldg(src + (static_cast<int64_t>(s + j) * a.num_kv_heads + kvh) * kHV + lane % kHV);
            }
        }
        // The unit's stream: the shared prefix (blocks [0, nsb) of the first member,
        // positions < ush), then each member j whose length exceeds ush: its blocks
        // from fb = ush / bs on, positions [ush, L_j).  Staged here (before the CTA
        // barrier, so every warp sees it): each block of this partition with its
        // physical id, its segment and the valid offsets within it.
        const int fb = ush >> lbs, nsb = (ush + bs - 1) >> lbs;
        // member lengths: the first two come with the work item
        int Lj = lane == 0 ? ul0 : lane == 1 ? ul1 : 0;
        if (lane >= 2 && lane < un) Lj = __ldg(a.seq_lens + s + lane);
        Lj = lane < un ? min(max(Lj, 0), a.max_seq_len) : 0;
        const int cnt = (lane < un && Lj > ush) ? ((Lj + bs - 1) >> lbs) - fb : 0;
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const int total = nsb + __shfl_sync(0xffffffffu, incl, 31);
        // the plan's stream must be this one: lengths changed since the plan otherwise
        const bool layout_ok = (static_cast<int64_t>(total) << lbs) == Lp;
        if (lane < un) {
            useg[lane] = nsb + incl - cnt;
            ulen[lane] = Lj;
        }
        if (lane == 0) {
            useg[un] = total;
            ulen[kHeadsPerCta] = !layout_ok;
            if (!layout_ok) raise_error(a.err, kErrBounds);
        }
        __syncwarp();
        for (int i = lane; i < nblk && layout_ok; i += 32) {
            const int sb = sb0 + i;
            int j = -1, lb = sb, lo = 0, hi = ush;
            if (sb >= nsb) {
                j = 0;
                while (j + 1 < un && useg[j + 1] <= sb) ++j;
                lb = fb + (sb - useg[j]);
                lo = ush;
                hi = ulen[j];
            }
            int b = __ldg(a.block_tables + static_cast<int64_t>(s + max(j, 0)) * a.max_blocks_per_seq + lb);
            if (b < 0 || static_cast<int64_t>(b) >= a.num_blocks) {
                raise_error(a.err, kErrBounds);
                b = -1;                             // outside the tensor map: TMA fills zeros, reads nothing
            }
            tbl[i] = b;
            const int vlo = min(max(lo - (lb << lbs), 0), bs), vhi = min(max(hi - (lb << lbs), 0), bs);
            udesc[i] = (j + 1) | (vlo << 8) | (vhi << 16);
        }
        __syncwarp();
        if (a.k_new != nullptr && layout_ok) {
            // Fused slot writes of the unit: member j's new token goes to position L_j - 1,
            // which must lie in its own segment (a block holding it is private after
            // copy-on-write) and be staged by this partition; a slot in the shared prefix is
            // refused.  Done before the CTA barrier; one proxy fence orders them all before
            // the tile loads.
            bool stored = false;
            for (int j = 0; j < un; ++j) {
                const int64_t slot = __shfl_sync(0xffffffffu, uslot, j);
                if (slot < 0) continue;
                const int pos = __shfl_sync(0xffffffffu, Lj, j) - 1;
                if (pos < ush) {
                    if (lane == 0) raise_error(a.err, kErrBounds);
                    continue;
                }
                const int i = useg[j] + ((pos >> lbs) - fb) - sb0;
                if (i < 0 || i >= nblk) continue;   // another partition of the unit holds it
                const int pb = tbl[i];
                if (pb < 0 || slot != static_cast<int64_t>(pb) * bs + (pos & (bs - 1))) {
                    if (lane == 0) raise_error(a.err, kErrBounds);
                    continue;
                }
                if (lane < 2 * kHV) {
                    uint4 r = urow[0];
#pragma unroll
                    for (int jj = 1; jj < kUnitRows; ++jj)
                        if (j == jj) r = urow[jj];
                    if (j >= kUnitRows) {
                        const uint4* src = lane < kHV ? a.k_new : a.v_new;
                        r = __ldg(src + (static_cast<int64_t>(s + j) * a.num_kv_heads + kvh) * kHV + lane % kHV);
                    }
                    const int64_t at = (slot * a.num_kv_heads + kvh) * kHV + lane % kHV;
                    reinterpret_cast<uint4*>(lane < kHV ? a.key_cache : a.value_cache)[at] = r;
                    stored = true;
                }
            }
            if (stored) fence_proxy_async_global();
        }
    }

    auto init_barriers = [&]() {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CW);
        }
        mbar_init(epi, kConsumers);
        // the 128B swizzle assumes a 1 KB aligned ring; refuse to run otherwise
        const bool misaligned = (smem_u32(smem) & 1023u) != 0;
        if (misaligned) raise_error(a.err, kErrTimeout);
        *abort_flag = misaligned;
        *merge_flag = 0;
        fence_barrier_init();
    };
    // K/V bytes are read once per step: evict them first, so the small data every
    // CTA and layer reuses (tables, q, work items, partials) stays in L2
    auto issue_chunk = [&](int c, uint64_t pol) {
        const int st = c % STAGES;
        const int tok0 = start + c * kChunk;
        const int nb = (min(end, tok0 + kChunk) - tok0 + bs - 1) / bs;
        mbar_arrive_expect_tx(&full[st], static_cast<unsigned>(nb * bs * D * kEB * 2));
        for (int j = 0; j < nb; ++j) {
            const int pb = tbl[c * (kChunk / bs) + j];
#pragma unroll
            for (int hf = 0; hf < G::kHalves; ++hf) {
                const int off = st * G::kStage + hf * G::kPlane + j * bs * 128;
                tma_load_4d_hint(kring + off, &tmk, hf * 64, kvh, 0, pb, &full[st], pol);
                tma_load_4d_hint(vring + off, &tmv, hf * 64, kvh, 0, pb, &full[st], pol);
            }
        }
    };
    auto stage_table = [&]() {                      // the producer warp's table slice into shared memory
#pragma unroll
        for (int k = 0; k < kTePerLane; ++k) {
            const int i = lane + 32 * k;
            if (32 * k < nblk && i < nblk) {
                int b = te[k];
                if (b < 0 || static_cast<int64_t>(b) >= a.num_blocks) {
                    raise_error(a.err, kErrBounds);
                    b = -1;                         // outside the tensor map: TMA fills zeros, reads nothing
                }
                tbl[i] = b;
            }
        }
        __syncwarp();
    };
    // chunks whose tile loads the producer issued before the wait (early only): the ring's
    // first stages, up to the chunk that receives the new token (written after the wait)
    int c_first = 0;
    if (early && warp == CW) {
        stage_table();
        if (lane == 0) {
            init_barriers();
            if (!*abort_flag) {
                prefetch_tensormap(&tmk);
                prefetch_tensormap(&tmv);
                const uint64_t pol = l2_policy_evict_first();
                for (; c_first < min(STAGES, nchunks); ++c_first) {
                    const int tok0 = start + c_first * kChunk;
                    if (maybe_put && L - 1 >= tok0 && L - 1 < tok0 + kChunk) break;
                    issue_chunk(c_first, pol);
                }
            }
        }
        c_first = __shfl_sync(0xffffffffu, c_first, 0);
    } else if (!early && threadIdx.x == 0) {
        init_barriers();
    }
    __syncthreads();
    if (grouped && ulen[kHeadsPerCta]) return;      // a unit whose layout the plan did not make

    // ================================================================ producer warp
    if (warp == CW) {
        // (a unit's blocks were staged before the barrier; early: with the first tile loads)
        if (!grouped && !early) stage_table();
        if (early) {
            grid_dependency_wait();                 // the new token comes from the preceding kernel
            if (maybe_put) {
                nslot = __ldg(a.slot_mapping + s);
                if (lane < 2 * kHV) {
                    const uint4* src = lane < kHV ? a.k_new : a.v_new;
                    nrow = __ldg(src + (static_cast<int64_t>(s) * a.num_kv_heads + kvh) * kHV + lane % kHV);
                }
            }
        }
        __syncwarp();
        // The fused slot write goes to the slot of position L - 1, which only
        // this partition reads in this call (and any other head group of the
        // same KV head, which writes the same bytes); anything else is refused.
        bool put = false;
        if (maybe_put && part == nparts - 1 && nslot >= 0) {
            const int pb = tbl[(L - 1) / bs - first_blk];
            put = pb >= 0 && nslot == static_cast<int64_t>(pb) * bs + (L - 1) % bs;
            if (!put && lane == 0) raise_error(a.err, kErrBounds);
        }
        // Each storing lane orders its stores before the tile loads (async
        // proxy) that lane 0 issues after the warp barrier.
        if (put && lane < 2 * kHV) {
            const int64_t at = (nslot * a.num_kv_heads + kvh) * kHV + lane % kHV;
            if constexpr (KV8)
                reinterpret_cast<uint2*>(lane < kHV ? a.key_cache : a.value_cache)[at] =
                    quantize8<std::is_same<T, __nv_bfloat16>::value>(nrow, nscale);
            else
                reinterpret_cast<uint4*>(lane < kHV ? a.key_cache : a.value_cache)[at] = nrow;
            fence_proxy_async_global();
        }
        __syncwarp();
        if (lane == 0 && !*abort_flag) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            const uint64_t pol = l2_policy_evict_first();
            for (int c = c_first; c < nchunks; ++c) {
                const int st = c % STAGES;
                const unsigned ph = (c / STAGES) & 1;
                if (!dec::wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                    dec::raise_abort(a.err, abort_flag);
                    break;
                }
                issue_chunk(c, pol);
            }
        }
        return;
    }

    // ================================================================ consumer warps
    dec::reset_state(ws);
    // an E4M3 pool's K scale multiplies every score of this KV head
    float sl2 = a.scale_log2;
    if constexpr (KV8) sl2 *= __ldg(a.k_scale + kvh);
    // causal limits of this lane's two query-row columns (all L for decode)
    const int lim0 = vh0 + 2 * (lane & 3) < a.group ? dec::causal_limit<MQ>(a, L, vh0 + 2 * (lane & 3)) : L;
    const int lim1 = vh0 + 2 * (lane & 3) + 1 < a.group ? dec::causal_limit<MQ>(a, L, vh0 + 2 * (lane & 3) + 1) : L;
    // a unit: the members of this lane's two columns
    const int mem0 = (2 * (lane & 3)) / a.group, mem1 = (2 * (lane & 3) + 1) / a.group;
    bool ok = !*abort_flag;
    unsigned epi_uses = 0;
    auto epi_sync = [&]() -> bool {               // all consumer threads, bounded
        mbar_arrive(epi);
        const bool r = dec::wait_or_abort(epi, epi_uses & 1, abort_flag);
        ++epi_uses;
        return r;
    };

    for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c % STAGES;
        const unsigned ph = (c / STAGES) & 1;
        bool got = dec::wait_or_abort(&full[st], ph, abort_flag);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
            if (lane == 0) dec::raise_abort(a.err, abort_flag);
            ok = false;
            break;
        }
        const int tokw = start + c * kChunk + warp * 16;
        const int nv = min(16, end - tokw);
        if (nv > 0) {
            if constexpr (KV8) {
                dec::consume_chunk_fp8<CW, MQ>(ws, smem_u32(kring + st * G::kStage), smem_u32(vring + st * G::kStage),
                                               nv, warp, lane, sl2, tokw, lim0, lim1);
            } else {
                const int r0 = lane >> 2;
                unsigned vis, zr;
                if (grouped) {
                    // row r of this tile: valid within its block's segment; seen by the
                    // columns of every member (shared prefix) or of its own member
                    auto row_seg = [&](int r) -> int {  // segment (-1: prefix) or -2: no token
                        if (r >= nv) return -2;
                        const int sp = tokw + r;
                        const int d = udesc[(sp >> lbs) - sb0];
                        const int o = sp & (bs - 1);
                        return (o >= ((d >> 8) & 0xFF) && o < (d >> 16)) ? (d & 0xFF) - 1 : -2;
                    };
                    const int ga = row_seg(r0), gb = row_seg(r0 + 8);
                    vis = ((ga == -1 || ga == mem0) ? 1u : 0u) | ((ga == -1 || ga == mem1) ? 2u : 0u) |
                          ((gb == -1 || gb == mem0) ? 4u : 0u) | ((gb == -1 || gb == mem1) ? 8u : 0u);
                    zr = __ballot_sync(0xffffffffu, lane < 16 && row_seg(lane) == -2) & 0xFFFFu;
                } else if constexpr (MQ) {
                    const bool va = r0 < nv, vb = r0 + 8 < nv;
                    const int pa = tokw + r0, pb = pa + 8;
                    vis = ((va && pa < lim0) ? 1u : 0u) | ((va && pa < lim1) ? 2u : 0u) | ((vb && pb < lim0) ? 4u : 0u) |
                          ((vb && pb < lim1) ? 8u : 0u);
                    zr = dec::tail_rows(nv);
                } else {
                    vis = dec::tile_vis(r0 < nv, r0 + 8 < nv);
                    zr = dec::tail_rows(nv);
                }
                dec::consume_chunk<T, D, CW>(ws, smem_u32(kring + st * G::kStage), smem_u32(vring + st * G::kStage),
                                             zr, vis, MQ || grouped, warp, lane, a.scale_log2);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    if (!ok) {
        // give copies still in flight a bounded moment to land before the CTA exits
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 10000000ull) __nanosleep(100000);
        return;
    }

    // this CTA's main loop is done: the next kernel in the stream (an append,
    // which waits for this grid) may start launching as the grid drains
    if (threadIdx.x == 0) launch_dependents();

    // ================================================= epilogue
    // merge the warps' states through shared memory (the ring is free: every
    // chunk was consumed by every warp, so no copy is still landing)
    float* scratch = reinterpret_cast<float*>(kring);
    if (!epi_sync()) return;                      // every warp is done reading the ring
    if constexpr (KV8)
        dec::warp_state_to_smem_fp8<CW>(ws, scratch, warp, lane, __ldg(a.v_scale + kvh));
    else
        dec::warp_state_to_smem<D, CW>(ws, scratch, warp, lane);
    if (!epi_sync()) return;
    dec::combine_warps<T, D, CW, MQ>(a, scratch, rows, gc, part, nparts, threadIdx.x, MQ || grouped);
    if (nparts == 1) return;
    // The group barrier orders every thread's partial writes before thread 0's
    // gpu-scope fence, which releases them all before the ticket.
    if (!epi_sync()) return;
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned* ticket = a.tickets + static_cast<int64_t>(s) * a.num_kv_heads * a.head_groups + hh;
        const unsigned t = atomicAdd(ticket, 1u);
        __threadfence();
        *merge_flag = (t == static_cast<unsigned>(nparts - 1));
        if (t == static_cast<unsigned>(nparts - 1)) *ticket = 0u;   // every partition has taken it: reset for the next run
    }
    if (!epi_sync()) return;
    if (!*merge_flag) return;
    // last partition of this (sequence, head group) to finish: merge them all
    dec::merge_partitions<T, D, CW, MQ>(a, scratch, rows, gc, nparts, warp, lane, threadIdx.x, epi_sync);
}

template <typename T, int D, int CW, int STAGES, bool MQ = false, bool KV8 = false, bool UNITS = false>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    constexpr size_t smem = Smem<D, CW, STAGES, KV8 ? 1 : 2, UNITS && !MQ && !KV8>::kBytes;
    static_assert(smem <= 232448, "shared memory budget");
    auto kern = decode_kernel<T, D, CW, STAGES, MQ, KV8, UNITS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned nh = static_cast<unsigned>(a.num_kv_heads * a.head_groups);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = a.plan ? dim3(nh * static_cast<unsigned>(a.plan_capacity))
                         : dim3(nh, static_cast<unsigned>(a.direct_parts), static_cast<unsigned>(a.num_seqs));
    cfg.blockDim = dim3(Geo<D, CW>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];                    // may launch while the plan kernel runs (it waits for it)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, a);
}

// Pipeline shapes (one per pool type, measured best on the 8B-shaped, 70B
// mixed and 80-layer batches): 16-bit pools run 4 consumer warps over 64-position
// chunks with a 2-stage ring, three CTAs per SM at head_dim 128; E4M3 pools the
// same chunks with 4 stages (the same ring bytes); the multi-query form
// likewise.
constexpr int kCW = 4;             // consumer warps
constexpr int kStages16 = 2;       // ring depth over 16-bit pools
constexpr int kStages8 = 4;        // and over E4M3 pools

template <typename T, int D>
cudaError_t launch_cfg(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    if (a.kv8) {
        if constexpr (D == 128) {
            if (a.num_queries > 1) return launch_t<T, D, kCW, kStages8, true, true>(a, tmk, tmv, s);
            return launch_t<T, D, kCW, kStages8, false, true>(a, tmk, tmv, s);
        }
        return cudaErrorInvalidValue;
    }
    if (a.num_queries > 1) return launch_t<T, D, kCW, kStages16, true>(a, tmk, tmv, s);
    // the plan may serve forks of one prompt as shared-prefix units: the kernel that reads them
    if (a.units) return launch_t<T, D, kCW, kStages16, false, false, true>(a, tmk, tmv, s);
    return launch_t<T, D, kCW, kStages16>(a, tmk, tmv, s);
}

}  // namespace

DecodeWorkspace decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_parts) {
    auto pad = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int group = num_heads / num_kv_heads;
    const int64_t nh = static_cast<int64_t>(num_kv_heads) * ((group + 7) / 8);
    const int parts = max_parts > 1 ? max_parts : 1;
    DecodeWorkspace w;
    w.ticket_bytes = pad(sizeof(unsigned) * static_cast<size_t>(num_seqs) * nh);
    w.plan_bytes = pad(kPlanEntryInts * sizeof(int4) * static_cast<size_t>(num_seqs) * parts);
    const size_t sh = static_cast<size_t>(num_seqs) * num_heads * (max_parts > 1 ? max_parts : 0);
    w.o_bytes = pad(sh * head_dim * sizeof(float));
    w.ml_bytes = pad(sh * 2 * sizeof(float));
    return w;
}

namespace {
template <typename T, int D, int CW, int STAGES, bool KV8 = false>
int occupancy_of() {
    constexpr size_t smem = Smem<D, CW, STAGES, KV8 ? 1 : 2>::kBytes;
    auto kern = decode_kernel<T, D, CW, STAGES, false, KV8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Geo<D, CW>::kThreads, smem) != cudaSuccess) return 0;
    return n;
}

}  // namespace

int decode_ctas_per_sm(int head_dim, bool kv8) {
    // head_dim 64, 128, E4M3; the same on every GB300, so host threads that race
    // on a first call store the same value
    static std::atomic<int> cache[3] = {-1, -1, -1};
    const int i = kv8 ? 2 : head_dim == 64 ? 0 : 1;
    int n = cache[i].load(std::memory_order_relaxed);
    if (n < 0) {
        n = kv8 ? occupancy_of<__half, 128, kCW, kStages8, true>()
                : i == 0 ? occupancy_of<__half, 64, kCW, kStages16>() : occupancy_of<__half, 128, kCW, kStages16>();
        cache[i].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, cudaStream_t s, DecodeMode mode) {
    if (a.num_seqs <= 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (a.plan) {
        if (mode != DecodeMode::kRunOnly) e = launch_decode_plan(a, s);
        if (mode == DecodeMode::kPlanOnly) return e;
    } else if (mode == DecodeMode::kPlanOnly) {
        return cudaSuccess;                         // a full-grid batch plans nothing
    } else if (a.max_parts > 1) {
        const size_t n = sizeof(unsigned) * static_cast<size_t>(a.num_seqs) * a.num_kv_heads * a.head_groups;
        e = cudaMemsetAsync(a.tickets, 0, n, s);
    }
    if (e != cudaSuccess) return e;
    if (dtype == 0)
        return head_dim == 128 ? launch_cfg<__half, 128>(a, tmk, tmv, s) : launch_cfg<__half, 64>(a, tmk, tmv, s);
    return head_dim == 128 ? launch_cfg<__nv_bfloat16, 128>(a, tmk, tmv, s)
                           : launch_cfg<__nv_bfloat16, 64>(a, tmk, tmv, s);
}

}  // namespace pkv
