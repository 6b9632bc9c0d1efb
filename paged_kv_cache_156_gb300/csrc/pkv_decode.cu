// paged_attention_decode: one query token per sequence over its paged K/V.
//
// What is computed ("tbr8.org PagedAttention article" §2.2; "LLM 推理引擎内部原理"
// §2.4): for each sequence s and query head h, walk the logical blocks of s,
// look each one up in the block table, read K/V rows of KV head
// g = h / group up to seq_len, and return softmax(scale * q.K) V.
//
// How (sm_103a):
//  * One CTA per work item = (KV head, group of <= 8 query heads sharing it,
//    partition of part_tokens positions, sequence).  All query heads of a KV
//    head are served from the same K/V bytes, so every byte of the pool is
//    read from HBM once per step.  Two or three CTAs share an SM so one CTA's
//    start-up (table and q fetch, first loads in flight) hides behind the
//    others' streaming.
//  * The CTA's slice of the block table is staged in shared memory once; a
//    producer warp then streams the partition's K and V tiles with TMA
//    (cp.async.bulk.tensor; one box = one (physical block, KV head) tile of
//    block_size rows x 64 elements, 128B-swizzled) into a ring of STAGES
//    chunks of 64 positions, handing each chunk over with an mbarrier.
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
#include <float.h>
#include <stdlib.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kMaxTable = 512;       // staged table entries: part_tokens (<= 4096) / block_size (>= 8)
constexpr int kHeadsPerCta = 8;      // mma N
constexpr int kMaxParts = 512;       // partitions per sequence the in-kernel merge handles

// CW consumer warps each own 16 positions of a chunk of 16 * CW positions.
template <int D, int CW>
struct Geo {
    static constexpr int kChunk = 16 * CW;              // positions per pipeline stage
    static constexpr int kConsumers = 32 * CW;
    static constexpr int kThreads = kConsumers + 32;    // plus one producer warp
    static constexpr int kHalves = D / 64;              // 64-element (128-byte) column planes
    static constexpr int kPlane = kChunk * 128;         // bytes of one plane of a chunk
    static constexpr int kStage = kHalves * kPlane;     // bytes of K (or V) of one chunk
    static constexpr int kScratch = CW * kHeadsPerCta * (D + 2) * 4;                     // warp-merge scratch
    static constexpr int kMergeScratch = (kHeadsPerCta * kMaxParts + kHeadsPerCta) * 4;  // partition merge
};

template <int D, int CW, int STAGES>
struct Smem {
    using G = Geo<D, CW>;
    static constexpr size_t kRing = 2 * STAGES * G::kStage;
    static constexpr size_t kScratch = (G::kScratch > G::kMergeScratch ? G::kScratch : G::kMergeScratch);
    static constexpr size_t kArena = kRing > kScratch ? kRing : kScratch;   // the scratch aliases the ring
    static constexpr size_t kBars = kArena;
    static constexpr size_t kTable = kBars + (2 * STAGES + 1) * sizeof(uint64_t);
    static constexpr size_t kMisc = kTable + kMaxTable * sizeof(int);
    static constexpr size_t kBytes = kMisc + 16;
};

// Address of 16-byte column chunk `ch` (0..7) of row `row` in a 128B-swizzled
// plane whose base is 1024-byte aligned: the chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t swz(uint32_t plane, int row, int ch) {
    return plane + row * 128 + ((ch ^ (row & 7)) << 4);
}

// Bounded wait that also gives up as soon as the CTA's abort flag is raised.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, unsigned parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void raise_abort(const DecodeArgs& a, volatile int* abort_flag) {
    if (!*abort_flag) raise_error(a.err, kErrTimeout);
    *abort_flag = 1;
}

template <typename T, int D, int CW, int STAGES>
__global__ void __launch_bounds__(Geo<D, CW>::kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                     const __grid_constant__ CUtensorMap tmv,
                                                                     const DecodeArgs a) {
    using G = Geo<D, CW>;
    using S = Smem<D, CW, STAGES>;
    using M = Mma<T>;
    constexpr int kChunk = G::kChunk;
    constexpr int kConsumerWarps = CW;
    constexpr int kConsumers = G::kConsumers;
    constexpr int kThreads = G::kThreads;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* kring = smem;
    uint8_t* vring = smem + STAGES * G::kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
    uint64_t* empty = full + STAGES;
    uint64_t* epi = empty + STAGES;               // consumer-group barrier (all 128 consumer threads)
    int* tbl = reinterpret_cast<int*>(smem + S::kTable);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc);
    volatile int* merge_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hh = blockIdx.x;                    // KV head * head_groups + query-head group
    const int part = blockIdx.y;
    const int s = blockIdx.z;
    const int hg = hh % a.head_groups;
    const int kvh = hh / a.head_groups;
    const int h0 = kvh * a.group + hg * kHeadsPerCta;
    const int gc = min(kHeadsPerCta, a.group - hg * kHeadsPerCta);
    const int bs = a.block_size;
    const int start = part * a.part_tokens;
    T* out = reinterpret_cast<T*>(a.out);

    // Issue the loads that depend only on the work item before the sequence
    // length is known: this warp's slice of the block table (producer) or the
    // query fragments (consumers).
    constexpr int kTePerLane = (kMaxTable + 31) / 32;
    int te[kTePerLane];
    uint32_t qb[D / 16][2];
    const int first_blk = start / bs;
    const int tcount = min(a.part_tokens / bs, a.max_blocks_per_seq - first_blk);
    if (warp == kConsumerWarps) {
        const int32_t* row = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + first_blk;
#pragma unroll
        for (int k = 0; k < kTePerLane; ++k) {
            const int i = lane + 32 * k;
            te[k] = (32 * k < tcount && i < tcount) ? __ldg(row + i) : 0;
        }
    } else {
        // Q^T as the B operand (k = head_dim, n = query head): lane holds
        // q[n = lane/4][k = 16*ks + 2*(lane%4) + {0,1}] and the same at k + 8.
        const int n = lane >> 2;
        const int kq = (lane & 3) * 2;
        const int nq = min(n, gc - 1);      // lanes of absent heads read a present row, then drop it
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const T*>(a.q) + (static_cast<int64_t>(s) * a.num_heads + h0 + nq) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qb[ks][0] = n < gc ? __ldg(qrow + (ks * 16 + kq) / 2) : 0u;
            qb[ks][1] = n < gc ? __ldg(qrow + (ks * 16 + 8 + kq) / 2) : 0u;
        }
    }

    const int L = __ldg(a.seq_lens + s);
    if (L <= 0) {                                   // empty sequence: zeros
        if (part == 0)
            for (int i = threadIdx.x; i < gc * D; i += kThreads)
                out[(static_cast<int64_t>(s) * a.num_heads + h0) * D + i] = T(0.0f);
        return;
    }
    if (start >= L) return;                         // partition past the end of this sequence
    const int end = min(L, start + a.part_tokens);
    const int nparts = (L + a.part_tokens - 1) / a.part_tokens;
    const int nchunks = (end - start + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        mbar_init(epi, kConsumers);
        // the 128B swizzle assumes a 1 KB aligned ring; refuse to run otherwise
        const bool misaligned = (smem_u32(smem) & 1023u) != 0;
        if (misaligned) raise_error(a.err, kErrTimeout);
        *abort_flag = misaligned;
        *merge_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ================================================================ producer warp
    if (warp == kConsumerWarps) {
        const int nblk = (end - start + bs - 1) / bs;
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
        if (lane == 0 && !*abort_flag) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            const int per_chunk = kChunk / bs;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % STAGES;
                const unsigned ph = (c / STAGES) & 1;
                if (!wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                    raise_abort(a, abort_flag);
                    break;
                }
                const int tok0 = start + c * kChunk;
                const int nb = (min(end, tok0 + kChunk) - tok0 + bs - 1) / bs;
                mbar_arrive_expect_tx(&full[st], static_cast<unsigned>(nb * bs * D * 2 * 2));
                for (int j = 0; j < nb; ++j) {
                    const int pb = tbl[c * per_chunk + j];
#pragma unroll
                    for (int hf = 0; hf < G::kHalves; ++hf) {
                        const int off = st * G::kStage + hf * G::kPlane + j * bs * 128;
                        tma_load_4d(kring + off, &tmk, hf * 64, kvh, 0, pb, &full[st]);
                        tma_load_4d(vring + off, &tmv, hf * 64, kvh, 0, pb, &full[st]);
                    }
                }
            }
        }
        return;
    }

    // ================================================================ consumer warps
    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    float mrun0 = -INFINITY, mrun1 = -INFINITY, lrun0 = 0.0f, lrun1 = 0.0f;
    const float sl2 = a.scale_log2;
    const int krow = warp * 16 + (lane & 15);                     // ldmatrix row supplied by this lane (K)
    const int kcol = lane >> 4;                                    // +8 elements
    const int vrow = warp * 16 + (lane & 7) + ((lane >> 4) << 3);  // (V, transposed load)
    const int vcol = (lane >> 3) & 1;
    const int r0 = lane >> 2;                                      // accumulator row (position) of c0/c1
    bool ok = !*abort_flag;
    unsigned epi_uses = 0;
    auto epi_sync = [&]() -> bool {               // all 128 consumer threads, bounded
        mbar_arrive(epi);
        const bool r = wait_or_abort(epi, epi_uses & 1, abort_flag);
        ++epi_uses;
        return r;
    };

    for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c % STAGES;
        const unsigned ph = (c / STAGES) & 1;
        bool got = wait_or_abort(&full[st], ph, abort_flag);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
            if (lane == 0) raise_abort(a, abort_flag);
            ok = false;
            break;
        }
        const int tok0 = start + c * kChunk + warp * 16;
        const int nv = min(16, end - tok0);
        const uint32_t kst = smem_u32(kring + st * G::kStage);
        const uint32_t vst = smem_u32(vring + st * G::kStage);
        if (nv > 0) {
            if (nv < 16) {
                // rows past seq_len hold no token: zero their V so 0-weights stay 0
                const int nz = (16 - nv) * (D / 8);
                for (int i = lane; i < nz; i += 32) {
                    const int r = warp * 16 + nv + i / (D / 8);
                    const int cc = i % (D / 8);
                    const uint32_t addr = swz(vst + (cc >> 3) * G::kPlane, r, cc & 7);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- S^T = K Q^T
            float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t af[4];
                ldmatrix_x4(af, swz(kst + (ks >> 2) * G::kPlane, krow, (ks & 3) * 2 + kcol));
                M::run(sacc, af, qb[ks][0], qb[ks][1]);
            }
            // ---- online softmax (log2 domain); columns are heads 2*(lane%4) + {0,1}
            const bool va = r0 < nv, vb = r0 + 8 < nv;
            const float s0 = va ? sacc[0] * sl2 : -INFINITY;
            const float s1 = va ? sacc[1] * sl2 : -INFINITY;
            const float s2 = vb ? sacc[2] * sl2 : -INFINITY;
            const float s3 = vb ? sacc[3] * sl2 : -INFINITY;
            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
            const float al0 = fast_exp2(mrun0 - mn0), al1 = fast_exp2(mrun1 - mn1);
            mrun0 = mn0;
            mrun1 = mn1;
            const uint32_t p01 = M::pack(fast_exp2(s0 - mn0), fast_exp2(s1 - mn1));
            const uint32_t p23 = M::pack(fast_exp2(s2 - mn0), fast_exp2(s3 - mn1));
            const float2 f01 = M::unpack(p01), f23 = M::unpack(p23);   // the weights PV actually uses
            lrun0 = lrun0 * al0 + f01.x + f23.x;
            lrun1 = lrun1 * al1 + f01.y + f23.y;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            // ---- O^T += V^T P^T ; P^T fragment = transpose of the score fragment
            const uint32_t pb0 = movmatrix_trans(p01);
            const uint32_t pb1 = movmatrix_trans(p23);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                uint32_t vf[4];
                ldmatrix_x4_trans(vf, swz(vst + (mt >> 2) * G::kPlane, vrow, (mt & 3) * 2 + vcol));
                M::run(o[mt], vf, pb0, pb1);
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

    // ================================================= epilogue
    // merge the four warps' states through shared memory (the ring is free:
    // every chunk was consumed by every warp, so no copy is still landing)
    float l0 = lrun0, l1 = lrun1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* sm_m = reinterpret_cast<float*>(kring);
    float* sm_l = sm_m + kConsumerWarps * kHeadsPerCta;
    float* sm_o = sm_l + kConsumerWarps * kHeadsPerCta;
    if (!epi_sync()) return;                      // every warp is done reading the ring
    if (lane < 4) {
        sm_m[warp * kHeadsPerCta + 2 * lane] = mrun0;
        sm_m[warp * kHeadsPerCta + 2 * lane + 1] = mrun1;
        sm_l[warp * kHeadsPerCta + 2 * lane] = l0;
        sm_l[warp * kHeadsPerCta + 2 * lane + 1] = l1;
    }
    {
        const int hA = 2 * (lane & 3);
        float* oa = sm_o + (warp * kHeadsPerCta + hA) * D;
        float* ob = oa + D;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = mt * 16 + r0;
            oa[d0] = o[mt][0];
            ob[d0] = o[mt][1];
            oa[d0 + 8] = o[mt][2];
            ob[d0 + 8] = o[mt][3];
        }
    }
    if (!epi_sync()) return;
    const int64_t sh0 = static_cast<int64_t>(s) * a.num_heads + h0;
    for (int idx = threadIdx.x; idx < gc * D; idx += kConsumers) {
        const int hx = idx / D;
        const int d = idx - hx * D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, sm_m[w * kHeadsPerCta + hx]);
        float den = 0.0f, num = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = fast_exp2(sm_m[w * kHeadsPerCta + hx] - mx);
            den += wt * sm_l[w * kHeadsPerCta + hx];
            num += wt * sm_o[(w * kHeadsPerCta + hx) * D + d];
        }
        const int64_t sh = sh0 + hx;
        if (nparts == 1) {
            out[sh * D + d] = T(num / den);
        } else {
            a.ws_o[(sh * a.max_parts + part) * D + d] = num;
            if (d == 0) a.ws_ml[sh * a.max_parts + part] = make_float2(mx, den);
        }
    }
    if (nparts == 1) return;
    __threadfence();                              // partials visible device-wide before the ticket
    if (!epi_sync()) return;
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(a.tickets + static_cast<int64_t>(s) * a.num_kv_heads * a.head_groups + hh, 1u);
        *merge_flag = (t == static_cast<unsigned>(nparts - 1));
    }
    if (!epi_sync()) return;
    if (!*merge_flag) return;
    // Last partition of this (sequence, head group) to finish: merge them all.
    // Weights 2^(m_p - M) and the denominators first (one warp per head, lanes
    // over partitions), then every output element sums its partials with the
    // loads of all its heads in flight together.
    __threadfence();
    float* wsm = reinterpret_cast<float*>(kring);              // [8 heads][kMaxParts] weights
    float* dsm = wsm + kHeadsPerCta * kMaxParts;                // [8 heads] denominators
    for (int hx = warp; hx < gc; hx += kConsumerWarps) {
        const float2* ml = a.ws_ml + (sh0 + hx) * a.max_parts;
        float mx = -INFINITY;
        for (int p = lane; p < nparts; p += 32) mx = fmaxf(mx, __ldcg(ml + p).x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float den = 0.0f;
        for (int p = lane; p < nparts; p += 32) {
            const float2 e = __ldcg(ml + p);
            const float w = fast_exp2(e.x - mx);
            wsm[hx * kMaxParts + p] = w;
            den += w * e.y;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (lane == 0) dsm[hx] = den;
    }
    if (!epi_sync()) return;
    constexpr int kRows = kConsumers / D > 0 ? kConsumers / D : 1;   // heads covered per pass
    constexpr int kAcc = (kHeadsPerCta + kRows - 1) / kRows;
    for (int base = 0; base < D; base += kConsumers) {               // D > kConsumers: several passes over d
        const int d = base + (kConsumers >= D ? threadIdx.x % D : threadIdx.x);
        const int hb = kConsumers >= D ? threadIdx.x / D : 0;
        if (d >= D) continue;
        float num[kAcc];
#pragma unroll
        for (int k = 0; k < kAcc; ++k) num[k] = 0.0f;
        for (int p = 0; p < nparts; ++p) {
#pragma unroll
            for (int k = 0; k < kAcc; ++k) {
                const int hx = hb + k * kRows;
                if (hx < gc)
                    num[k] += wsm[hx * kMaxParts + p] * __ldcg(a.ws_o + ((sh0 + hx) * a.max_parts + p) * D + d);
            }
        }
#pragma unroll
        for (int k = 0; k < kAcc; ++k) {
            const int hx = hb + k * kRows;
            if (hx < gc) out[(sh0 + hx) * D + d] = T(num[k] / dsm[hx]);
        }
    }
}

template <typename T, int D, int CW, int STAGES>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    constexpr size_t smem = Smem<D, CW, STAGES>::kBytes;
    static_assert(smem <= 232448, "shared memory budget");
    auto kern = decode_kernel<T, D, CW, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(a.num_kv_heads * a.head_groups), static_cast<unsigned>(a.max_parts),
              static_cast<unsigned>(a.num_seqs));
    kern<<<grid, Geo<D, CW>::kThreads, smem, s>>>(tmk, tmv, a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_cfg(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int warps, int stages,
                       cudaStream_t s) {
    if (warps == 2) {
        switch (stages) {
            case 2: return launch_t<T, D, 2, 2>(a, tmk, tmv, s);
            case 4: return launch_t<T, D, 2, 4>(a, tmk, tmv, s);
            default: return launch_t<T, D, 2, 3>(a, tmk, tmv, s);
        }
    }
    switch (stages) {
        case 3: return launch_t<T, D, 4, 3>(a, tmk, tmv, s);
        case 4: return launch_t<T, D, 4, 4>(a, tmk, tmv, s);
        default: return launch_t<T, D, 4, 2>(a, tmk, tmv, s);
    }
}

// Pipeline shape: 4 consumer warps (64-position chunks) with a 2-stage ring,
// three CTAs per SM at head_dim 128.  PKV_DECODE_WARPS in {2, 4} and
// PKV_DECODE_STAGES in {2, 3, 4} override it (tuning knobs; read once).
int env_choice(const char* name, int dflt, int lo, int hi) {
    const char* e = getenv(name);
    const int x = e ? atoi(e) : dflt;
    return (x >= lo && x <= hi) ? x : dflt;
}
int ring_stages() {
    static const int v = env_choice("PKV_DECODE_STAGES", 2, 2, 4);
    return v;
}
int consumer_warps() {
    static const int v = env_choice("PKV_DECODE_WARPS", 4, 2, 4) == 2 ? 2 : 4;
    return v;
}

}  // namespace

DecodeWorkspace decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_parts) {
    auto pad = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int group = num_heads / num_kv_heads;
    const int64_t nh = static_cast<int64_t>(num_kv_heads) * ((group + 7) / 8);
    DecodeWorkspace w;
    w.ticket_bytes = pad(sizeof(unsigned) * (1 + static_cast<size_t>(num_seqs) * nh));
    const size_t sh = static_cast<size_t>(num_seqs) * num_heads * (max_parts > 1 ? max_parts : 0);
    w.o_bytes = pad(sh * head_dim * sizeof(float));
    w.ml_bytes = pad(sh * 2 * sizeof(float));
    return w;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, size_t zero_bytes, cudaStream_t s) {
    if (a.num_seqs <= 0) return cudaSuccess;
    if (a.max_parts > 1) {
        cudaError_t e = cudaMemsetAsync(a.tickets, 0, zero_bytes - sizeof(unsigned), s);
        if (e != cudaSuccess) return e;
    }
    const int st = ring_stages(), cw = consumer_warps();
    if (dtype == 0) {
        return head_dim == 128 ? launch_cfg<__half, 128>(a, tmk, tmv, cw, st, s)
                               : launch_cfg<__half, 64>(a, tmk, tmv, cw, st, s);
    }
    return head_dim == 128 ? launch_cfg<__nv_bfloat16, 128>(a, tmk, tmv, cw, st, s)
                           : launch_cfg<__nv_bfloat16, 64>(a, tmk, tmv, cw, st, s);
}

}  // namespace pkv
