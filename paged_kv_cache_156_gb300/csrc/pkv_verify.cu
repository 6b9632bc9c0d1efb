// paged_attention_verify for many query rows per KV head: the rows are the
// tensor-core M dimension.
//
// What is computed ("vLLM核心概念" §4.4.2 and "LLM 推理优化深度实战" §4.2: the
// target model scores all draft tokens in one pass over the prefix KV;
// "LLM 推理引擎内部原理" §5.2: their KV lives in the same blocks): query token
// i of sequence s (the last num_queries positions are the queries' own)
// attends over positions t < L - num_queries + i + 1 with softmax(scale q.K) V.
//
// How.  A KV head serves R = (num_heads / num_kv_heads) * num_queries query
// rows.  The decode kernel serves 8 rows per CTA (the mma's N), so a KV head
// with 32 rows would stream its K/V through 4 CTAs.  Here one CTA serves up
// to 64 rows: 4 consumer warps each own 16 rows (the mma's M) and run
// FlashAttention-style over the partition's chunks: S[16 x 64] = Q K^T with
// K fragments from the same TMA ring as decode (ldmatrix), an fp32 online
// softmax per row, and O[16 x d] += P V with P taken straight from the S
// accumulators (the accumulator layout of S is the A-operand layout of P)
// and V fragments by ldmatrix.trans.  With more than 32 rows a warp owns whole
// rows for the whole chunk.  With at most 32 (GQA 8 and four draft tokens,
// say) the two warps of a 16-row tile split each chunk's positions, 32 each,
// so all four warps work; each keeps its own online softmax and the pair
// merges lane by lane through shared memory after the last chunk.  Split
// partitions merge through the workspace with the same ticket protocol as
// decode (the last partition merges).
#include <atomic>

#include "pkv_decode_common.cuh"

namespace pkv {

namespace {

using dec::Geo;
using dec::kMaxTable;

constexpr int kVW = 4;                 // consumer warps
constexpr int kVRows = 16 * kVW;       // query rows per CTA
constexpr int kWholeStages = 2;        // K/V ring depth of the 64-row kernel (chunks)
constexpr int kSplitStages = 3;        // and of the 32-row kernel

template <int D, int STAGES>
struct VSmem {
    using G = Geo<D, kVW>;
    static constexpr size_t kRing = 2 * STAGES * G::kStage;
    static constexpr size_t kBars = kRing;
    static constexpr size_t kTable = kBars + (2 * STAGES + 1) * sizeof(uint64_t);
    static constexpr size_t kMisc = kTable + kMaxTable * sizeof(int);
    static constexpr size_t kBytes = kMisc + 16;
};

// Element offset / D of row r (0 <= r < R) of KV head kvh of sequence s in q / out.
__device__ __forceinline__ int64_t vrow_offset(const DecodeArgs& a, int s, int kvh, int r) {
    const int i = r / a.qgroup;
    const int hl = r - i * a.qgroup;
    return (static_cast<int64_t>(s) * a.num_queries + i) * a.num_heads + kvh * a.qgroup + hl;
}

// SPLIT: warps sharing one 16-row tile (1: 64 rows per CTA; 2: 32 rows, each
// warp takes half of every chunk's positions).  STAGES: depth of the K/V ring.
template <typename T, int D, int SPLIT, int STAGES>
__global__ void __launch_bounds__(Geo<D, kVW>::kThreads, 2) verify_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                          const __grid_constant__ CUtensorMap tmv,
                                                                          const DecodeArgs a) {
    constexpr int kVStages = STAGES;
    using G = Geo<D, kVW>;
    using S = VSmem<D, STAGES>;
    using M = Mma<T>;
    constexpr int kChunk = G::kChunk;               // 64 positions
    constexpr int kNT = kChunk / 8 / SPLIT;         // n-tiles of S per chunk and warp
    constexpr int kRows = kVRows / SPLIT;           // query rows per CTA
    constexpr int kDT = D / 8;                      // n-tiles of O
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* kring = smem;
    uint8_t* vring = smem + kVStages * G::kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
    uint64_t* empty = full + kVStages;
    uint64_t* epi = empty + kVStages;
    int* tbl = reinterpret_cast<int*>(smem + S::kTable);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc);
    volatile int* merge_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    grid_dependency_wait();

    // ---- work item (plan entry or full grid), as in decode
    const int nh = a.num_kv_heads * a.head_groups;
    int hh, part, s, P, L;
    if (a.plan) {
        const unsigned y = blockIdx.x / static_cast<unsigned>(nh);
        hh = static_cast<int>(blockIdx.x - y * static_cast<unsigned>(nh));
        const int4 it = __ldg(a.plan + kPlanEntryInts * y);   // (this kernel's plans have one-sequence units)
        s = it.x;
        part = it.y;
        L = it.z;
        P = it.w;
        if (s < 0) return;
        if (s >= a.num_seqs || part < 0 || L < 0 || L > a.max_seq_len || P < 64 || P > kMaxTable * a.block_size ||
            part * P >= max(L, 1) || (L + P - 1) / P > a.max_parts) {
            if (threadIdx.x == 0) raise_error(a.err, kErrBounds);
            return;
        }
    } else {
        hh = blockIdx.x;
        part = blockIdx.y;
        s = blockIdx.z;
        P = a.part_tokens;
        L = __ldg(a.seq_lens + s);
        if (L > a.max_seq_len) {
            if (threadIdx.x == 0 && part == 0 && hh == 0) raise_error(a.err, kErrBounds);
            L = a.max_seq_len;
        }
    }
    const int rg = hh % a.head_groups;              // group of kRows rows of this KV head
    const int kvh = hh / a.head_groups;
    const int R = a.group;                          // rows of the KV head
    const int half = SPLIT == 2 ? (warp & 1) : 0;   // which half of each chunk's positions (SPLIT 2)
    const int tile = warp / SPLIT;                  // 16-row tile of this warp
    const int pc0 = half * (kChunk / SPLIT);        // first chunk position of this warp
    int rw = rg * kRows + tile * 16;                // this warp's first row
    const int ra = rw + g, rb = rw + g + 8;         // this lane's rows
    T* out = reinterpret_cast<T*>(a.out);
    const int bs = a.block_size;
    const int start = part * P;

    if (L <= 0) {                                   // empty sequence: zeros
        if (part == 0 && warp < kVW && half == 0)
            for (int i = lane; i < 16 * D; i += 32) {
                const int r = rw + i / D;
                if (r < R) out[vrow_offset(a, s, kvh, r) * D + i % D] = T(0.0f);
            }
        return;
    }
    if (start >= L) return;
    const int end = min(L, start + P);
    const int nparts = (L + P - 1) / P;
    const int nchunks = (end - start + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kVW);
        }
        mbar_init(epi, 32 * kVW);
        const bool misaligned = (smem_u32(smem) & 1023u) != 0;
        if (misaligned) raise_error(a.err, kErrTimeout);
        *abort_flag = misaligned;
        *merge_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ================================================================ producer warp
    if (warp == kVW) {
        const int first_blk = start / bs;
        const int nblk = (end - start + bs - 1) / bs;
        const int32_t* row = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + first_blk;
        for (int i = lane; i < nblk; i += 32) {
            int b = __ldg(row + i);
            if (b < 0 || static_cast<int64_t>(b) >= a.num_blocks) {
                raise_error(a.err, kErrBounds);
                b = -1;                             // outside the tensor map: TMA fills zeros
            }
            tbl[i] = b;
        }
        __syncwarp();
        if (lane == 0 && !*abort_flag) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            // K/V read once: keep the reused data in L2.  With more than one
            // row group per KV head the sibling CTAs read the same tiles: no hint.
            const bool hint = a.head_groups == 1;
            const uint64_t pol = l2_policy_evict_first();
            const int per_chunk = kChunk / bs;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kVStages;
                const unsigned ph = (c / kVStages) & 1;
                if (!dec::wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                    dec::raise_abort(a.err, abort_flag);
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
                        if (hint) {
                            tma_load_4d_hint(kring + off, &tmk, hf * 64, kvh, 0, pb, &full[st], pol);
                            tma_load_4d_hint(vring + off, &tmv, hf * 64, kvh, 0, pb, &full[st], pol);
                        } else {
                            tma_load_4d(kring + off, &tmk, hf * 64, kvh, 0, pb, &full[st]);
                            tma_load_4d(vring + off, &tmv, hf * 64, kvh, 0, pb, &full[st]);
                        }
                    }
                }
            }
        }
        return;
    }

    // ================================================================ consumer warps
    // Q as the A operand (rows x head_dim), per 16-wide k-step: (row a, k 2t..2t+1),
    // (row b, same k), (row a, k 2t+8..2t+9), (row b, same k)
    bool va = ra < R, vb = rb < R;
    uint32_t qa[D / 16][4];
    {
        const uint32_t* qra = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(a.q) +
                                                                vrow_offset(a, s, kvh, va ? ra : 0) * D);
        const uint32_t* qrb = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(a.q) +
                                                                vrow_offset(a, s, kvh, vb ? rb : 0) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][0] = va ? __ldg(qra + ks * 8 + t) : 0u;
            qa[ks][1] = vb ? __ldg(qrb + ks * 8 + t) : 0u;
            qa[ks][2] = va ? __ldg(qra + ks * 8 + 4 + t) : 0u;
            qa[ks][3] = vb ? __ldg(qrb + ks * 8 + 4 + t) : 0u;
        }
    }
    // causal limits of the two rows: query token i sees positions < L - num_queries + i + 1
    const int lim_a = va ? L - a.num_queries + ra / a.qgroup + 1 : L;
    const int lim_b = vb ? L - a.num_queries + rb / a.qgroup + 1 : L;
    const float sl2 = a.scale_log2;

    float o[kDT][4];
#pragma unroll
    for (int dn = 0; dn < kDT; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.0f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;   // l: this lane's share of the row sum

    bool ok = !*abort_flag;
    unsigned epi_uses = 0;
    auto epi_sync = [&]() -> bool {               // all consumer threads, bounded
        mbar_arrive(epi);
        const bool r = dec::wait_or_abort(epi, epi_uses & 1, abort_flag);
        ++epi_uses;
        return r;
    };

    for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c % kVStages;
        const unsigned ph = (c / kVStages) & 1;
        bool got = dec::wait_or_abort(&full[st], ph, abort_flag);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
            if (lane == 0) dec::raise_abort(a.err, abort_flag);
            ok = false;
            break;
        }
        if (rw >= R) {                              // a warp with no rows keeps the ring's phases, computes nothing
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }
        const int tok0 = start + c * kChunk;
        const int nv = min(kChunk, end - tok0);     // positions of this chunk inside the partition
        const uint32_t kst = smem_u32(kring + st * G::kStage);
        const uint32_t vst = smem_u32(vring + st * G::kStage);

        // ---- S = Q K^T over the chunk's 64 positions (8 n-tiles)
        float sacc[kNT][4];
#pragma unroll
        for (int j = 0; j < kNT; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < kNT / 2; ++np) {
                uint32_t bf[4];
                const int pos = pc0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldmatrix_x4(bf, dec::swz(kst + (ks >> 2) * G::kPlane, pos, (ks & 3) * 2 + ((lane >> 3) & 1)));
                M::run(sacc[2 * np], qa[ks], bf[0], bf[1]);
                M::run(sacc[2 * np + 1], qa[ks], bf[2], bf[3]);
            }
        }
        // ---- online softmax per row (log2 domain); lane holds positions 8j + 2t + {0, 1}
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int j = 0; j < kNT; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int pc = pc0 + 8 * j + 2 * t + e;   // position within the chunk
                const int pos = tok0 + pc;
                sacc[j][e] = (pc < nv && pos < lim_a) ? sacc[j][e] * sl2 : -INFINITY;
                sacc[j][2 + e] = (pc < nv && pos < lim_b) ? sacc[j][2 + e] * sl2 : -INFINITY;
                mx_a = fmaxf(mx_a, sacc[j][e]);
                mx_b = fmaxf(mx_b, sacc[j][2 + e]);
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {      // the quad holding the row
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        // a row that has seen no position yet keeps max -inf: scale 1, weights 0
        const float al_a = mn_a == -INFINITY ? 1.0f : fast_exp2(m_a - mn_a);
        const float al_b = mn_b == -INFINITY ? 1.0f : fast_exp2(m_b - mn_b);
        const float b_a = mn_a == -INFINITY ? 0.0f : mn_a, b_b = mn_b == -INFINITY ? 0.0f : mn_b;
        m_a = mn_a;
        m_b = mn_b;
        // P (rounded to T) is the A operand of O += P V: per 16 positions kk,
        // (row a, pos 2t..), (row b, pos 2t..), (row a, pos 8+2t..), (row b, pos 8+2t..)
        uint32_t pa[kNT / 2][4];
        float sum_a = 0.0f, sum_b = 0.0f;
#pragma unroll
        for (int kk = 0; kk < kNT / 2; ++kk) {
            const int j0 = 2 * kk, j1 = 2 * kk + 1;
            pa[kk][0] = M::pack(fast_exp2(sacc[j0][0] - b_a), fast_exp2(sacc[j0][1] - b_a));
            pa[kk][1] = M::pack(fast_exp2(sacc[j0][2] - b_b), fast_exp2(sacc[j0][3] - b_b));
            pa[kk][2] = M::pack(fast_exp2(sacc[j1][0] - b_a), fast_exp2(sacc[j1][1] - b_a));
            pa[kk][3] = M::pack(fast_exp2(sacc[j1][2] - b_b), fast_exp2(sacc[j1][3] - b_b));
            const float2 f0 = M::unpack(pa[kk][0]), f1 = M::unpack(pa[kk][1]);
            const float2 f2 = M::unpack(pa[kk][2]), f3 = M::unpack(pa[kk][3]);
            sum_a += f0.x + f0.y + f2.x + f2.y;
            sum_b += f1.x + f1.y + f3.x + f3.y;
        }
        l_a = l_a * al_a + sum_a;
        l_b = l_b * al_b + sum_b;
        if (__any_sync(0xffffffffu, al_a != 1.0f || al_b != 1.0f)) {
#pragma unroll
            for (int dn = 0; dn < kDT; ++dn) {
                o[dn][0] *= al_a;
                o[dn][1] *= al_a;
                o[dn][2] *= al_b;
                o[dn][3] *= al_b;
            }
        }
        // ---- O += P V; V fragments by ldmatrix.trans, positions past the partition zeroed
        // in registers (a slot past the sequence may hold NaN, and 0 * NaN is NaN)
        const bool tail = nv < pc0 + kChunk / SPLIT;
#pragma unroll
        for (int kk = 0; kk < kNT / 2; ++kk) {
            uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;   // keep-masks of positions 16kk+2t(+1), +8
            if (tail) {
                const int p0 = pc0 + 16 * kk + 2 * t;
                mlo = (p0 < nv ? 0x0000FFFFu : 0u) | (p0 + 1 < nv ? 0xFFFF0000u : 0u);
                mhi = (p0 + 8 < nv ? 0x0000FFFFu : 0u) | (p0 + 9 < nv ? 0xFFFF0000u : 0u);
            }
#pragma unroll
            for (int dp = 0; dp < kDT / 2; ++dp) {
                uint32_t vf[4];
                const int pos = pc0 + 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int dch = 2 * dp + (lane >> 4);   // 8-element column chunk over head_dim
                ldmatrix_x4_trans(vf, dec::swz(vst + (dch >> 3) * G::kPlane, pos, dch & 7));
                vf[0] &= mlo;
                vf[1] &= mhi;
                vf[2] &= mlo;
                vf[3] &= mhi;
                M::run(o[2 * dp], pa[kk], vf[0], vf[1]);
                M::run(o[2 * dp + 1], pa[kk], vf[2], vf[3]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    if (!ok) {
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 10000000ull) __nanosleep(100000);
        return;
    }

    if (threadIdx.x == 0) launch_dependents();      // the main loop is done: the next kernel may launch

    // ---- SPLIT 2: the warp of the second half hands its state to the warp of
    // the first (the same lane holds the same rows and columns), which merges
    // it like two partitions; the ring is free once every warp is past its
    // last chunk
    if constexpr (SPLIT == 2) {
        constexpr int kSlot = kDT * 4 + 4;          // floats per lane: o, then (m_a, m_b, l_a, l_b)
        float* sc = reinterpret_cast<float*>(kring) + (tile * 32 + lane) * kSlot;
        if (!epi_sync()) return;
        if (half == 1) {
#pragma unroll
            for (int dn = 0; dn < kDT; ++dn)
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[4 * dn + i] = o[dn][i];
            sc[4 * kDT] = m_a;
            sc[4 * kDT + 1] = m_b;
            sc[4 * kDT + 2] = l_a;
            sc[4 * kDT + 3] = l_b;
        }
        if (!epi_sync()) return;
        if (half == 0) {
            const float m2a = sc[4 * kDT], m2b = sc[4 * kDT + 1];
            const float Ma = fmaxf(m_a, m2a), Mb = fmaxf(m_b, m2b);
            // a row neither half saw keeps max -inf and zero state
            const float w1a = Ma == -INFINITY ? 0.0f : fast_exp2(m_a - Ma);
            const float w2a = Ma == -INFINITY ? 0.0f : fast_exp2(m2a - Ma);
            const float w1b = Mb == -INFINITY ? 0.0f : fast_exp2(m_b - Mb);
            const float w2b = Mb == -INFINITY ? 0.0f : fast_exp2(m2b - Mb);
#pragma unroll
            for (int dn = 0; dn < kDT; ++dn) {
                o[dn][0] = o[dn][0] * w1a + sc[4 * dn] * w2a;
                o[dn][1] = o[dn][1] * w1a + sc[4 * dn + 1] * w2a;
                o[dn][2] = o[dn][2] * w1b + sc[4 * dn + 2] * w2b;
                o[dn][3] = o[dn][3] * w1b + sc[4 * dn + 3] * w2b;
            }
            l_a = l_a * w1a + sc[4 * kDT + 2] * w2a;
            l_b = l_b * w1b + sc[4 * kDT + 3] * w2b;
            m_a = Ma;
            m_b = Mb;
        } else {
            va = vb = false;                        // the first-half warp writes these rows
        }
    }

    // ================================================= epilogue: this warp's rows are complete
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
    }
    if (nparts == 1) {
        const float ia = l_a > 0.0f ? 1.0f / l_a : 0.0f, ib = l_b > 0.0f ? 1.0f / l_b : 0.0f;
        T* oa = va ? out + vrow_offset(a, s, kvh, ra) * D : nullptr;
        T* ob = vb ? out + vrow_offset(a, s, kvh, rb) * D : nullptr;
#pragma unroll
        for (int dn = 0; dn < kDT; ++dn) {
            const int d = 8 * dn + 2 * t;
            if (va) *reinterpret_cast<uint32_t*>(oa + d) = M::pack(o[dn][0] * ia, o[dn][1] * ia);
            if (vb) *reinterpret_cast<uint32_t*>(ob + d) = M::pack(o[dn][2] * ib, o[dn][3] * ib);
        }
        return;
    }
    // split: this partition's (max, sum, unnormalised output) of each row to the workspace
    const int64_t prow0 = static_cast<int64_t>(s) * a.num_heads * a.num_queries + static_cast<int64_t>(kvh) * R;
    if (va) {
        const int64_t pr = (prow0 + ra) * a.max_parts + part;
#pragma unroll
        for (int dn = 0; dn < kDT; ++dn)
            *reinterpret_cast<float2*>(a.ws_o + pr * D + 8 * dn + 2 * t) = make_float2(o[dn][0], o[dn][1]);
        if (t == 0) a.ws_ml[pr] = make_float2(m_a, l_a);
    }
    if (vb) {
        const int64_t pr = (prow0 + rb) * a.max_parts + part;
#pragma unroll
        for (int dn = 0; dn < kDT; ++dn)
            *reinterpret_cast<float2*>(a.ws_o + pr * D + 8 * dn + 2 * t) = make_float2(o[dn][2], o[dn][3]);
        if (t == 0) a.ws_ml[pr] = make_float2(m_b, l_b);
    }
    // the group barrier orders every thread's partial writes before thread 0's
    // gpu-scope fence, which releases them before the ticket
    if (!epi_sync()) return;
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned* ticket = a.tickets + static_cast<int64_t>(s) * nh + hh;
        const unsigned tk = atomicAdd(ticket, 1u);
        __threadfence();
        *merge_flag = (tk == static_cast<unsigned>(nparts - 1));
        if (tk == static_cast<unsigned>(nparts - 1)) *ticket = 0u;   // reset for the next run
    }
    if (!epi_sync()) return;
    if (!*merge_flag || half == 1) return;
    // last partition of this (sequence, row group): each warp merges its own rows;
    // lane covers head-dim elements [lane * D/32, +D/32)
    constexpr int kPer = D / 32;
    for (int rr = 0; rr < 16; ++rr) {
        const int r = rw + rr;
        if (r >= R) break;
        const float2* ml = a.ws_ml + (prow0 + r) * a.max_parts;
        float mx = -INFINITY;
        for (int p = lane; p < nparts; p += 32) mx = fmaxf(mx, __ldcg(ml + p).x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float num[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) num[k] = 0.0f;
        float den = 0.0f;
        if (mx != -INFINITY) {
            for (int p = 0; p < nparts; ++p) {
                const float2 e = __ldcg(ml + p);
                const float w = e.x == -INFINITY ? 0.0f : fast_exp2(e.x - mx);
                den += w * e.y;
                const float* op = a.ws_o + ((prow0 + r) * a.max_parts + p) * D + lane * kPer;
#pragma unroll
                for (int k = 0; k < kPer; ++k) num[k] += w * __ldcg(op + k);
            }
        }
        const float inv = den > 0.0f ? 1.0f / den : 0.0f;
        T* orow = out + vrow_offset(a, s, kvh, r) * D + lane * kPer;
#pragma unroll
        for (int k = 0; k < kPer; k += 2) *reinterpret_cast<uint32_t*>(orow + k) = M::pack(num[k] * inv, num[k + 1] * inv);
    }
}

template <typename T, int D, int SPLIT, int STAGES>
cudaError_t launch_verify_k(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    constexpr size_t smem = VSmem<D, STAGES>::kBytes;
    static_assert(2 * smem + 2048 <= 233472, "two CTAs per SM fit the shared memory");
    static_assert(2 * 32 * (D / 8 * 4 + 4) * sizeof(float) <= 2 * STAGES * Geo<D, kVW>::kStage,
                  "the half-merge scratch fits the ring");
    auto kern = verify_kernel<T, D, SPLIT, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned nh = static_cast<unsigned>(a.num_kv_heads * a.head_groups);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = a.plan ? dim3(nh * static_cast<unsigned>(a.plan_capacity))
                         : dim3(nh, static_cast<unsigned>(a.direct_parts), static_cast<unsigned>(a.num_seqs));
    cfg.blockDim = dim3(Geo<D, kVW>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, a);
}

template <typename T, int D>
cudaError_t launch_verify_t(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    // 32 rows per CTA: two warps per 16-row tile; 64: one warp per tile (head_groups matches)
    // (a 3-chunk ring for the 32-row kernel, whose warps each take half a chunk
    // and so wait on the ring sooner; 2 chunks for 64 rows, where the extra
    // stage measured no faster)
    const bool split = verify_rows_per_cta(a.group) == kVRows / 2;
    return split ? launch_verify_k<T, D, 2, kSplitStages>(a, tmk, tmv, s)
                 : launch_verify_k<T, D, 1, kWholeStages>(a, tmk, tmv, s);
}

}  // namespace

cudaError_t launch_verify(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, cudaStream_t s, DecodeMode mode) {
    if (a.num_seqs <= 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (a.plan) {
        if (mode != DecodeMode::kRunOnly) e = launch_decode_plan(a, s);
        if (mode == DecodeMode::kPlanOnly) return e;
    } else if (mode == DecodeMode::kPlanOnly) {
        return cudaSuccess;
    } else if (a.max_parts > 1) {
        const size_t n = sizeof(unsigned) * static_cast<size_t>(a.num_seqs) * a.num_kv_heads * a.head_groups;
        e = cudaMemsetAsync(a.tickets, 0, n, s);
    }
    if (e != cudaSuccess) return e;
    if (dtype == 0) return head_dim == 128 ? launch_verify_t<__half, 128>(a, tmk, tmv, s)
                                           : launch_verify_t<__half, 64>(a, tmk, tmv, s);
    return head_dim == 128 ? launch_verify_t<__nv_bfloat16, 128>(a, tmk, tmv, s)
                           : launch_verify_t<__nv_bfloat16, 64>(a, tmk, tmv, s);
}

}  // namespace pkv

namespace pkv {

int verify_rows_per_cta(int rows) {
    // up to 32 rows: two warps per 16-row tile; more: 64-row CTAs (two 32-row
    // CTAs per KV head measured slower: their K/V bytes leave HBM twice)
    return rows <= kVRows / 2 ? kVRows / 2 : kVRows;
}

int verify_ctas_per_sm(int head_dim, int rows) {
    // the same on every GB300; threads that race here store the same value
    static std::atomic<int> cache[4] = {-1, -1, -1, -1};
    const bool split = verify_rows_per_cta(rows) == kVRows / 2;
    const int i = (head_dim == 64 ? 0 : 1) + (split ? 2 : 0);
    int n_cached = cache[i].load(std::memory_order_relaxed);
    if (n_cached < 0) {
        int n = 0;
        auto set_and_query = [&](auto kern, size_t smem) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) ==
                    cudaSuccess &&
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Geo<128, kVW>::kThreads, smem) == cudaSuccess)
                return n;
            return 0;
        };
        switch (i) {
            case 0: n_cached = set_and_query(verify_kernel<__half, 64, 1, kWholeStages>, VSmem<64, kWholeStages>::kBytes); break;
            case 1: n_cached = set_and_query(verify_kernel<__half, 128, 1, kWholeStages>, VSmem<128, kWholeStages>::kBytes); break;
            case 2: n_cached = set_and_query(verify_kernel<__half, 64, 2, kSplitStages>, VSmem<64, kSplitStages>::kBytes); break;
            default: n_cached = set_and_query(verify_kernel<__half, 128, 2, kSplitStages>, VSmem<128, kSplitStages>::kBytes); break;
        }
        cache[i].store(n_cached, std::memory_order_relaxed);
    }
    return n_cached;
}

}  // namespace pkv
