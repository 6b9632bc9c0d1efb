// paged_attention_verify on the fifth-generation tensor cores (tcgen05): many
// query rows per KV head, the rows the MMA's M dimension.
//
// What is computed ("vLLM核心概念" §4.4.2 and "LLM 推理优化深度实战" §4.2: the
// target model scores all draft tokens in one pass over the prefix KV;
// "LLM 推理引擎内部原理" §5.2: their KV lives in the same blocks): query token
// i of sequence s (its last num_queries positions are the queries' own)
// attends over positions t < L - num_queries + i + 1 with softmax(scale q.K) V.
//
// How.  A KV head serves R = (num_heads / num_kv_heads) * num_queries query
// rows; one CTA serves M of them, M = 64 when R <= 64, else 128 (rows past R
// are zero), over one partition of one sequence from the same work list as
// decode.  An M = 64 product keeps its rows in the first 16 TMEM lanes of each
// warp's 32-lane quarter (rows 16 w .. 16 w + 15 in lanes 32 w ..).  The K/V
// tiles arrive by TMA, 128-byte swizzled, into a ring of 32-position stages
// laid out plane-major (plane, stage, position), so that the two stages of a
// 64-position step sit side by side in every plane, and per step:
//   S = Q K^T      tcgen05.mma, M rows x N = 64 positions: A = Q held in
//                  tensor memory (TMEM) as 16-bit pairs, B = the step's K rows
//                  (K-major, 128-byte swizzle), S in TMEM as fp32;
//   softmax        M = 64: the 16x256b TMEM load shape gives each thread two
//                  rows x 16 columns (all 32 lanes busy), the row maximum
//                  reduced over the quad; M = 128: one row a thread.  Positions
//                  past the partition and past the row's causal limit are
//                  masked; a running reference maximum moves only when a score
//                  exceeds it by more than 2^8 (then the rows' O and sums are
//                  rescaled in TMEM); P = 2^(s - ref) rounded to the input type
//                  goes to one of two 128-byte-swizzled P buffers;
//   O += P V       tcgen05.mma, A = that P buffer (K-major), B = the step's V
//                  read as an MN-major operand (its 64-element column blocks
//                  one plane apart), O in TMEM as fp32.
// The S products and the O products are issued by one thread each (warps 6 and
// 5), so the next step's S never waits behind this step's O product; a stage is
// refilled as soon as the O product that read it is done.  A producer warp
// streams the tiles (its lane 0 reads each stage's block ids one stage ahead).
// TMEM holds Q, S and O (256 columns), the shared memory the ring (96 KB at
// M = 64) and P, so two CTAs share an SM.
// Split partitions write (reference max, sum, unnormalised O) per row; the CTA
// that takes the last ticket merges them (split-K), from shared memory when the
// partitions' rows fit the idle ring, else from global memory.
// Every wait is bounded in wall time; a CTA that gives up raises the error
// word, waits (bounded) for its own MMAs and frees its TMEM.
#include <algorithm>
#include <atomic>

#include "pkv_decode_common.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {

namespace {

using dec::kMaxTable;

template <int D, int M>
struct TcGeo {
    static constexpr int kChunk = 32;                   // positions per ring stage
    static constexpr int kStep = 64;                    // positions per S product (two stages)
    static constexpr int kPlane = kChunk * 128;         // bytes of one 128-byte column plane of a stage
    static constexpr int kHalves = D * 2 / 128;         // planes per K (or V) tile
    static constexpr int kStage = kHalves * kPlane;     // bytes of K (or V) of one stage
    // ring depth (even: a step's two stages sit side by side in every plane): 96 KB of K/V
    // beside the 16 KB of P for M = 64, 64 KB beside 32 KB for M = 128
    static constexpr int kStages = (D == 128 ? 6 : 12) * (M == 128 ? 2 : 3) / 3;
    static constexpr int kPlaneRing = kStages * kPlane; // bytes of one plane across the ring
    static constexpr int kRows = M;                     // query rows per CTA (the MMAs' M)
    static constexpr int kThreads = 224;                // 4 softmax warps, producer, two MMA warps
    static constexpr int kSoftmaxThreads = 128;
    static constexpr int kProducerWarp = 4;
    static constexpr int kMmaWarp = 5;                  // issues O += P V; owns TMEM
    static constexpr int kSWarp = 6;                    // issues S = Q K^T
    static constexpr int kMaxBlocksPerChunk = kChunk / 8;   // block size 8 at least (and at most 32)
    // TMEM columns (32-bit) of the CTA's 256
    static constexpr uint32_t kColQ = 0;                // Q rows, two 16-bit elements a column (D / 2 columns)
    static constexpr uint32_t kColS = 64;               // S of one step, kStep fp32 columns
    static constexpr uint32_t kColO = 128;              // O, fp32, D columns
    static constexpr uint32_t kTmemCols = 256;
    // shared memory: the ring (plane-major: plane, stage, position), two P buffers
    // (M rows x kStep positions, 16-bit, 128-byte swizzled), barriers
    static constexpr size_t kRing = 2 * size_t(kStages) * kStage;
    static constexpr size_t kP = kRing;
    static constexpr int kPRowBytes = kStep * 2;        // a P row: one step's positions, 16-bit
    static constexpr size_t kPBuf = size_t(M) * kPRowBytes;
    static constexpr int kNumBars = 2 * kStages + 12;
    static constexpr size_t kBars = kP + 2 * kPBuf;
    static constexpr size_t kMisc = kBars + kNumBars * sizeof(uint64_t);
    static constexpr size_t kBytes = kMisc + 16;
};

// Element offset / D of row r (0 <= r < R) of KV head kvh of sequence s in q / out.
__device__ __forceinline__ int64_t tc_row_offset(const DecodeArgs& a, int s, int kvh, int r) {
    const int i = r / a.qgroup;
    const int hl = r - i * a.qgroup;
    return (static_cast<int64_t>(s) * a.num_queries + i) * a.num_heads + kvh * a.qgroup + hl;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return Mma<T>::pack(lo, hi); }

template <typename T, int D, int M>
__global__ void __launch_bounds__(TcGeo<D, M>::kThreads, 2) verify_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                             const __grid_constant__ CUtensorMap tmv,
                                                                             const DecodeArgs a) {
    using TG = TcGeo<D, M>;
    constexpr int ST = TG::kStages;
    constexpr int kChunk = TG::kChunk;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* kring = smem;
    uint8_t* vring = smem + ST * TG::kStage;
    uint8_t* ptile = smem + TG::kP;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TG::kBars);
    uint64_t* full = bars;                          // [ST] a chunk's K and V landed (TMA bytes)
    uint64_t* empty = bars + ST;                    // [ST] the chunk's O += P V done (MMA commit)
    uint64_t* s_full = bars + 2 * ST;               // a step's S in TMEM, earlier products done (MMA commit)
    uint64_t* s_free = s_full + 1;                  // the step's S read into registers (softmax threads)
    uint64_t* p_full = s_full + 2;                  // [2] a step's P written, V tail zeroed (softmax threads)
    uint64_t* o_done = s_full + 4;                  // [2] O += P V of a step using P buffer b done (MMA commit)
    uint64_t* q_ready = s_full + 6;                 // Q rows in TMEM (softmax threads)
    uint64_t* o_last = s_full + 7;                  // the item's last O += P V done (MMA commit)
    uint64_t* epi = s_full + 8;                     // softmax threads' epilogue barrier
    uint64_t* done = s_full + 9;                    // softmax threads finished with TMEM
    uint64_t* fin = s_full + 10;                    // every MMA this CTA issued is done (one commit per issuer)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + TG::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + TG::kMisc + 4);
    volatile int* merge_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    grid_dependency_wait();

    // ---- work item (plan entry or full grid), as in decode
    const int nh = a.num_kv_heads * a.head_groups;
    int hh, part, s, P, L;
    if (a.plan) {
        const unsigned y = blockIdx.x / static_cast<unsigned>(nh);
        hh = static_cast<int>(blockIdx.x - y * static_cast<unsigned>(nh));
        const int4 it = __ldg(a.plan + kPlanEntryInts * y);   // (verify plans hold one-sequence units)
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
    const int rg = hh % a.head_groups;              // group of 128 rows of this KV head
    const int kvh = hh / a.head_groups;
    const int R = a.group;                          // rows of the KV head
    // a softmax thread's row of the CTA (its TMEM lane is 32 w + its lane): M = 128, the
    // thread index; M = 64, 16 w + lane for lanes 0..15 (the other lanes hold none)
    const int lrow = M == 128 ? static_cast<int>(threadIdx.x) : (lane < 16 ? (warp << 4) + lane : -1);
    const int row = rg * TG::kRows + lrow;
    const bool has_row = threadIdx.x < TG::kSoftmaxThreads && lrow >= 0 && row < R;
    T* out = reinterpret_cast<T*>(a.out);
    const int bs = a.block_size;
    const int start = part * P;

    if (L <= 0) {                                   // empty sequence: zeros
        if (part == 0 && has_row) {
            uint4* o = reinterpret_cast<uint4*>(out + tc_row_offset(a, s, kvh, row) * D);
            for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        return;
    }
    if (start >= L) return;
    const int end = min(L, start + P);
    const int nparts = (L + P - 1) / P;
    const int nchunks = (end - start + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, TG::kSoftmaxThreads);
        for (int i = 0; i < 2; ++i) mbar_init(&p_full[i], TG::kSoftmaxThreads);
        mbar_init(&o_done[0], 1);
        mbar_init(&o_done[1], 1);
        mbar_init(q_ready, TG::kSoftmaxThreads);
        mbar_init(o_last, 1);
        mbar_init(epi, TG::kSoftmaxThreads);
        mbar_init(done, TG::kSoftmaxThreads);
        mbar_init(fin, 2);
        // the 128B swizzle and the MMA descriptors assume a 1 KB aligned ring
        const bool misaligned = (smem_u32(smem) & 1023u) != 0;
        if (misaligned) raise_error(a.err, kErrTimeout);
        *abort_flag = misaligned;
        *merge_flag = 0;
        fence_barrier_init();
    }
    if (warp == TG::kMmaWarp) tc::tmem_alloc(tmem_slot, TG::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // ================================================================ producer warp: the K/V ring
    if (warp == TG::kProducerWarp) {
        if (lane == 0 && !*abort_flag) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            // K/V read once; with several row groups per KV head the siblings read the same tiles
            const bool hint = a.head_groups == 1;
            const uint64_t pol = l2_policy_evict_first();
            const int per_chunk = kChunk / bs;
            const int first_blk = start / bs;
            const int nblk = (end - start + bs - 1) / bs;
            const int32_t* trow = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + first_blk;
            // each chunk's block ids, read one chunk ahead of their tile loads
            int nxt[TG::kMaxBlocksPerChunk];
#pragma unroll
            for (int j = 0; j < TG::kMaxBlocksPerChunk; ++j) nxt[j] = (j < per_chunk && j < nblk) ? __ldg(trow + j) : -1;
            for (int c = 0; c < nchunks; ++c) {
                int cur[TG::kMaxBlocksPerChunk];
#pragma unroll
                for (int j = 0; j < TG::kMaxBlocksPerChunk; ++j) {
                    cur[j] = nxt[j];
                    const int i = (c + 1) * per_chunk + j;
                    nxt[j] = (j < per_chunk && i < nblk) ? __ldg(trow + i) : -1;
                }
                const int st = c % ST;
                const unsigned ph = (c / ST) & 1;
                if (!dec::wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                    dec::raise_abort(a.err, abort_flag);
                    break;
                }
                const int tok0 = start + c * kChunk;
                const int nb = (min(end, tok0 + kChunk) - tok0 + bs - 1) / bs;
                mbar_arrive_expect_tx(&full[st], static_cast<unsigned>(nb * bs * D * 2 * 2));
#pragma unroll
                for (int j = 0; j < TG::kMaxBlocksPerChunk; ++j) {
                    if (j >= nb) break;
                    int pb = cur[j];
                    if (pb < 0 || static_cast<int64_t>(pb) >= a.num_blocks) {
                        raise_error(a.err, kErrBounds);
                        pb = -1;                    // outside the tensor map: TMA fills zeros
                    }
#pragma unroll
                    for (int hf = 0; hf < TG::kHalves; ++hf) {
                        const int off = hf * TG::kPlaneRing + st * TG::kPlane + j * bs * 128;
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

    // ================================================================ MMA warps: one thread each issues
    // The S products and the O products come from two threads, so that the next step's
    // S never queues behind this step's O += P V (which waits on the softmax).  Neither
    // needs the other's completions: a step's P is written only after its S was read, so
    // the O product that reads P (and frees the stage) follows the S that read K.
    if (warp == TG::kMmaWarp || warp == TG::kSWarp) {
        if (lane == 0) {
            const int n = end - start;                  // positions of the partition
            const int nsteps = (n + TG::kStep - 1) / TG::kStep;
            bool ok = !*abort_flag;
            if (warp == TG::kSWarp) {
                constexpr uint32_t kIdS = tc::idesc_f16(TG::kRows, TG::kStep, kBf16, false);   // S = Q K^T
                // step h's two stages: chunks 2h and 2h + 1 (the second absent past the end)
                auto wait_step = [&](int h) -> bool {
                    const int c = 2 * h;
                    if (!dec::wait_or_abort(&full[c % ST], (c / ST) & 1, abort_flag)) return false;
                    return c + 1 >= nchunks ||
                           dec::wait_or_abort(&full[(c + 1) % ST], ((c + 1) / ST) & 1, abort_flag);
                };
                ok = ok && dec::wait_or_abort(q_ready, 0, abort_flag);
                for (int h = 0; h < nsteps && ok; ++h) {
                    // S of step h (positions 64 h .. 64 h + 63) into the buffer the softmax
                    // threads have read: its K tile is 64 rows of 128 bytes per plane, the
                    // two stages side by side
                    ok = (h == 0 || dec::wait_or_abort(s_free, (h - 1) & 1, abort_flag)) && wait_step(h);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t kst = smem_u32(kring + ((2 * h) % ST) * TG::kPlane);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {   // 16 head-dim elements a step: 32 bytes of a row
                        const uint64_t bdesc =
                            tc::smem_desc_sw128(kst + (ks >> 2) * TG::kPlaneRing + (ks & 3) * 32, 16, 1024);
                        tc::mma_ts(tmem + TG::kColS, tmem + TG::kColQ + ks * 8, bdesc, kIdS, ks > 0);
                    }
                    tc::commit(s_full);
                }
            } else {
                constexpr uint32_t kIdO = tc::idesc_f16(TG::kRows, D, kBf16, true);   // O += P V
                const uint32_t pt = smem_u32(ptile);
                for (int h = 0; h < nsteps && ok; ++h) {
                    ok = dec::wait_or_abort(&p_full[h & 1], (h >> 1) & 1, abort_flag);   // its P written
                    if (!ok) break;
                    tc::fence_after_sync();
                    // O += P V over the step's positions, 16 a product (none wholly past the end)
                    const int nk = (min(TG::kStep, n - h * TG::kStep) + 15) / 16;
#pragma unroll
                    for (int kk = 0; kk < TG::kStep / 16; ++kk) {
                        if (kk >= nk) break;
                        const int c = 2 * h + (kk >> 1);
                        const uint32_t vst = smem_u32(vring + (c % ST) * TG::kPlane + (kk & 1) * 2048);
                        const uint64_t adesc = tc::smem_desc_sw128(pt + (h & 1) * TG::kPBuf + kk * 32, 16, 1024);
                        const uint64_t bdesc = tc::smem_desc_sw128(vst, TG::kPlaneRing, 1024);
                        tc::mma_ss(tmem + TG::kColO, adesc, bdesc, kIdO, (h > 0 || kk > 0) ? 1u : 0u);
                        if ((kk & 1) || kk + 1 == nk) tc::commit(&empty[c % ST]);   // the stage is read: refill
                    }
                    tc::commit(&o_done[h & 1]);
                    if (h == nsteps - 1) tc::commit(o_last);
                }
            }
            if (!ok) dec::raise_abort(a.err, abort_flag);
            tc::commit(fin);                        // every product this thread issued
            dec::wait_or_abort(fin, 0, abort_flag);
            if (!ok || *abort_flag) {               // (an abort may leave MMAs running: give them a moment)
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 10000000ull) __nanosleep(100000);
            }
        }
        if (warp == TG::kSWarp) return;
        __syncwarp();
        // the softmax threads read TMEM last; then free it
        dec::wait_or_abort(done, 0, abort_flag);
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TG::kTmemCols);
        return;
    }

    // ================================================================ softmax warps: one query row per thread
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);   // this warp's 32 TMEM lanes
    // Q row into TMEM (zeros past R), two elements a column
    {
        const uint4* qrow = has_row ? reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.q) +
                                                                     tc_row_offset(a, s, kvh, row) * D)
                                    : nullptr;
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t qv[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 x = has_row ? __ldg(qrow + c0 / 4 + j) : make_uint4(0u, 0u, 0u, 0u);
                qv[4 * j] = x.x;
                qv[4 * j + 1] = x.y;
                qv[4 * j + 2] = x.z;
                qv[4 * j + 3] = x.w;
            }
            tc::st32(tl + TG::kColQ + c0, qv);
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(q_ready);
    }
    // causal limit: query token i sees positions < L - num_queries + i + 1 (rows past R: none)
    const int lim = has_row ? L - a.num_queries + row / a.qgroup + 1 : 0;
    const float sl2 = a.scale_log2;
    const int prow = lrow;                          // this thread's row of the P tile (-1: none)
    const uint32_t pbase = smem_u32(ptile) + max(prow, 0) * TG::kPRowBytes;
    float m_ref = -INFINITY;                        // the row's reference maximum (log2 units)
    float l = 0.0f;                                 // the row's sum of rounded weights, relative to m_ref
    bool ok = !*abort_flag;
    bool gave_up = false;                           // a rescale's wait timed out (the CTA is aborting)
    const int nsteps = (end - start + TG::kStep - 1) / TG::kStep;
    if constexpr (M == 64) {
        // Two rows a thread, all 32 lanes busy: the 16x256b TMEM shape gives thread t rows
        // ra = 16 w + t / 4 and ra + 8, columns 8 i + 2 (t % 4) + {0, 1} of each 8-column
        // group i.  A row's maximum is reduced over its quad; its sum stays split over the
        // quad until the end (every part is relative to the same reference).
        const int q4 = lane & 3;
        const int ra = (warp << 4) + (lane >> 2);
        const int row_a = rg * TG::kRows + ra, row_b = row_a + 8;
        const int lim_a = row_a < R ? L - a.num_queries + row_a / a.qgroup + 1 : 0;
        const int lim_b = row_b < R ? L - a.num_queries + row_b / a.qgroup + 1 : 0;
        const uint32_t pa = smem_u32(ptile) + ra * TG::kPRowBytes + 4 * q4;
        const uint32_t pb = pa + 8 * TG::kPRowBytes;
        const int sw = ra & 7;                      // (row ra + 8 has the same swizzle phase)
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
        for (int h = 0; h < nsteps && ok; ++h) {
            const int b = h & 1;
            ok = !gave_up && dec::wait_or_abort(s_full, h & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::fence_after_sync();
            uint32_t r[32];
            tc::ld16x256_x8(r, tl + TG::kColS);
            tc::wait_ld();
            tc::fence_before_sync();
            mbar_arrive(s_free);                    // the MMA may write the next S
            const int tok0 = start + h * TG::kStep;
            const int nv = min(TG::kStep, end - tok0);
            const int vis_a = min(nv, lim_a - tok0), vis_b = min(nv, lim_b - tok0);
            float sa[16], sb[16];
            float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = 8 * i + 2 * q4 + e;
                    sa[2 * i + e] = col < vis_a ? __uint_as_float(r[4 * i + e]) * sl2 : -INFINITY;
                    sb[2 * i + e] = col < vis_b ? __uint_as_float(r[4 * i + 2 + e]) * sl2 : -INFINITY;
                    mxa = fmaxf(mxa, sa[2 * i + e]);
                    mxb = fmaxf(mxb, sb[2 * i + e]);
                }
            }
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            // a new reference when a score exceeds the old one by more than 2^8 (the same
            // in the row's four threads): rescale what O and the sums hold
            float alpha_a = 1.0f, alpha_b = 1.0f;
            if (mxa > m_a + 8.0f) {
                if (m_a != -INFINITY) alpha_a = fast_exp2(m_a - mxa);
                m_a = mxa;
            }
            if (mxb > m_b + 8.0f) {
                if (m_b != -INFINITY) alpha_b = fast_exp2(m_b - mxb);
                m_b = mxb;
            }
            if (__any_sync(0xffffffffu, alpha_a != 1.0f || alpha_b != 1.0f)) {
                // the previous step's product (and so every earlier one) must be done
                if (h >= 1 && !gave_up && !dec::wait_or_abort(&o_done[b ^ 1], ((h - 1) >> 1) & 1, abort_flag)) {
                    gave_up = true;
                    dec::raise_abort(a.err, abort_flag);
                }
                gave_up = __any_sync(0xffffffffu, gave_up);
                tc::fence_after_sync();
                l_a *= alpha_a;
                l_b *= alpha_b;
                if (!gave_up) {
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[16];
                        tc::ld16x256_x4(o, tl + TG::kColO + c0);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            o[4 * i] = __float_as_uint(__uint_as_float(o[4 * i]) * alpha_a);
                            o[4 * i + 1] = __float_as_uint(__uint_as_float(o[4 * i + 1]) * alpha_a);
                            o[4 * i + 2] = __float_as_uint(__uint_as_float(o[4 * i + 2]) * alpha_b);
                            o[4 * i + 3] = __float_as_uint(__uint_as_float(o[4 * i + 3]) * alpha_b);
                        }
                        tc::st16x256_x4(tl + TG::kColO + c0, o);
                    }
                    tc::wait_st();
                }
            }
            // P buffer b is free once the product two steps back is done (waited every step)
            if (h >= 2 && !gave_up && !dec::wait_or_abort(&o_done[b], ((h >> 1) - 1) & 1, abort_flag)) {
                gave_up = true;
                dec::raise_abort(a.err, abort_flag);
            }
            gave_up = __any_sync(0xffffffffu, gave_up);
            if (!gave_up) {
                // P = 2^(s - m) rounded to T: thread q4's pair of group i sits at byte 4 q4 of
                // the row's 16-byte chunk i, chunk i at i ^ (row % 8) (128-byte swizzle)
                const bool any_a = m_a != -INFINITY, any_b = m_b != -INFINITY;
                const uint32_t boff = b * static_cast<uint32_t>(TG::kPBuf);
                float sum_a = 0.0f, sum_b = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t wa = pack2<T>(any_a ? fast_exp2(sa[2 * i] - m_a) : 0.0f,
                                                 any_a ? fast_exp2(sa[2 * i + 1] - m_a) : 0.0f);
                    const uint32_t wb = pack2<T>(any_b ? fast_exp2(sb[2 * i] - m_b) : 0.0f,
                                                 any_b ? fast_exp2(sb[2 * i + 1] - m_b) : 0.0f);
                    const float2 fa = Mma<T>::unpack(wa), fb = Mma<T>::unpack(wb);
                    sum_a += fa.x + fa.y;
                    sum_b += fb.x + fb.y;
                    const uint32_t off = boff + (static_cast<uint32_t>(i ^ sw) << 4);
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(pa + off), "r"(wa) : "memory");
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(pb + off), "r"(wb) : "memory");
                }
                l_a += sum_a;
                l_b += sum_b;
            }
            // V rows past the partition's end, up to the end of the last 16-position product,
            // may hold NaN (0 * NaN is NaN in the product)
            if (nv < TG::kStep && (nv & 15)) {
                constexpr int kCh = D * 2 / 16;         // 16-byte chunks of a V row
                const int z1 = (nv + 15) & ~15;
                for (int i = threadIdx.x; i < (z1 - nv) * kCh; i += TG::kSoftmaxThreads) {
                    const int pos = nv + i / kCh, cc = i % kCh;
                    uint8_t* vst = vring + ((2 * h + (pos >> 5)) % ST) * TG::kPlane;
                    const uint32_t addr = dec::swz(smem_u32(vst + (cc >> 3) * TG::kPlaneRing), pos & 31, cc & 7);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                }
            }
            fence_proxy_async_smem();               // P (and zeroed V) before the MMA reads them
            tc::fence_before_sync();
            mbar_arrive(&p_full[b]);
        }
        // the rows' sums over their quads; lane r < 16 then takes row 16 w + r (the epilogue's
        // 32x32b shape) from the quad that holds it
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        const int src = (lane & 7) << 2;
        const float la = __shfl_sync(0xffffffffu, l_a, src), lb = __shfl_sync(0xffffffffu, l_b, src);
        const float ma = __shfl_sync(0xffffffffu, m_a, src), mb = __shfl_sync(0xffffffffu, m_b, src);
        l = lane < 8 ? la : lb;
        m_ref = lane < 8 ? ma : mb;
    } else {
        for (int h = 0; h < nsteps && ok; ++h) {
            const int b = h & 1;
            // S of step h (every product before the one two steps back is done)
            ok = !gave_up && dec::wait_or_abort(s_full, h & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::fence_after_sync();
            float sv[TG::kStep];
    #pragma unroll
            for (int c0 = 0; c0 < TG::kStep; c0 += 32) {
                uint32_t r[32];
                tc::ld32(r, tl + TG::kColS + c0);
                tc::wait_ld();
    #pragma unroll
                for (int j = 0; j < 32; ++j) sv[c0 + j] = __uint_as_float(r[j]);
            }
            tc::fence_before_sync();
            mbar_arrive(s_free);                        // the MMA may write the next S
            const int tok0 = start + h * TG::kStep;
            const int nv = min(TG::kStep, end - tok0);  // positions of this step inside the partition (>= 1)
            const int vis = min(nv, lim - tok0);        // this row sees positions j < vis of the step
            float mx = -INFINITY;
    #pragma unroll
            for (int j = 0; j < TG::kStep; ++j) {
                sv[j] = j < vis ? sv[j] * sl2 : -INFINITY;
                mx = fmaxf(mx, sv[j]);
            }
            // a new reference when a score exceeds the old one by more than 2^8: rescale what O
            // and l hold (TMEM loads and stores are warp-wide: the warp rescales when any of its
            // rows needs it, by 1 for the others)
            float alpha = 1.0f;
            if (mx > m_ref + 8.0f) {
                if (m_ref != -INFINITY) alpha = fast_exp2(m_ref - mx);
                m_ref = mx;
            }
            if (__any_sync(0xffffffffu, alpha != 1.0f)) {
                // the previous step's product (and so every earlier one) must be done before O is read
                if (h >= 1 && !gave_up && !dec::wait_or_abort(&o_done[b ^ 1], ((h - 1) >> 1) & 1, abort_flag)) {
                    gave_up = true;                     // (the warp leaves the loop together at the next step)
                    dec::raise_abort(a.err, abort_flag);
                }
                gave_up = __any_sync(0xffffffffu, gave_up);
                tc::fence_after_sync();
                l *= alpha;
                if (!gave_up) {
    #pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        uint32_t o[16];
                        tc::ld16(o, tl + TG::kColO + c0);
                        tc::wait_ld();
    #pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tc::st16(tl + TG::kColO + c0, o);
                    }
                    tc::wait_st();
                }
            }
            // P = 2^(s - m_ref) rounded to T into this row of P buffer b (128-byte swizzle:
            // 16-byte chunk k of row r at chunk k ^ (r % 8)), once the product two steps back,
            // which read this buffer, is done (waited every step, so each wait is on the phase
            // after the last one seen)
            if (h >= 2 && !gave_up && !dec::wait_or_abort(&o_done[b], ((h >> 1) - 1) & 1, abort_flag)) {
                gave_up = true;
                dec::raise_abort(a.err, abort_flag);
            }
            gave_up = __any_sync(0xffffffffu, gave_up);
            if (!gave_up) {
                const bool any = m_ref != -INFINITY;
                const uint32_t prow_addr = pbase + b * static_cast<uint32_t>(TG::kPBuf);
                float sum = 0.0f;
    #pragma unroll
                for (int k = 0; k < TG::kStep / 8; ++k) {
                    uint32_t w[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 8 * k + 2 * e;
                        const float p0 = any ? fast_exp2(sv[j] - m_ref) : 0.0f;
                        const float p1 = any ? fast_exp2(sv[j + 1] - m_ref) : 0.0f;
                        w[e] = pack2<T>(p0, p1);
                        const float2 f = Mma<T>::unpack(w[e]);
                        sum += f.x + f.y;
                    }
                    const uint32_t addr = prow_addr + ((k ^ (prow & 7)) << 4);
                    if (prow >= 0)
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                                     "r"(w[2]), "r"(w[3])
                                     : "memory");
                }
                l += sum;
            }
            // V rows past the partition's end, up to the end of the last 16-position product,
            // may hold NaN (0 * NaN is NaN in the product)
            if (nv < TG::kStep && (nv & 15)) {
                constexpr int kCh = D * 2 / 16;         // 16-byte chunks of a V row
                const int z1 = (nv + 15) & ~15;
                for (int i = threadIdx.x; i < (z1 - nv) * kCh; i += TG::kSoftmaxThreads) {
                    const int pos = nv + i / kCh, cc = i % kCh;
                    uint8_t* vst = vring + ((2 * h + (pos >> 5)) % ST) * TG::kPlane;
                    const uint32_t addr = dec::swz(smem_u32(vst + (cc >> 3) * TG::kPlaneRing), pos & 31, cc & 7);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                }
            }
            fence_proxy_async_smem();                   // P (and zeroed V) before the MMA reads them
            tc::fence_before_sync();
            mbar_arrive(&p_full[b]);
        }
    }
    if (ok) ok = !gave_up && dec::wait_or_abort(o_last, 0, abort_flag);   // the item's last product
    ok = __all_sync(0xffffffffu, ok);

    // ---- epilogue: this thread's row of O
    const int64_t prow0 = static_cast<int64_t>(s) * a.num_heads * a.num_queries + static_cast<int64_t>(kvh) * R;
    if (ok) {
        tc::fence_after_sync();
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        T* orow = has_row ? out + tc_row_offset(a, s, kvh, row) * D : nullptr;
        float* wrow = (has_row && nparts > 1) ? a.ws_o + ((prow0 + row) * a.max_parts + part) * D : nullptr;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc::ld32(o, tl + TG::kColO + c0);
            tc::wait_ld();
            if (has_row) {
                if (nparts == 1) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        w[j] = pack2<T>(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                } else {
                    float4* dst = reinterpret_cast<float4*>(wrow + c0);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                             __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
                }
            }
        }
        if (has_row && nparts > 1) a.ws_ml[(prow0 + row) * a.max_parts + part] = make_float2(m_ref, l);
    }
    tc::fence_before_sync();
    mbar_arrive(done);                              // TMEM is no longer read by this thread
    if (!ok) {
        if (lane == 0) dec::raise_abort(a.err, abort_flag);
        return;
    }
    if (threadIdx.x == 0) launch_dependents();
    if (nparts == 1) return;

    // ---- split-K: the last partition of this (sequence, row group) merges every partition's rows
    unsigned epi_uses = 0;
    auto epi_sync = [&]() -> bool {
        mbar_arrive(epi);
        const bool r = dec::wait_or_abort(epi, epi_uses & 1, abort_flag);
        ++epi_uses;
        return r;
    };
    if (!epi_sync()) return;                        // every row's partial is written
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned* ticket = a.tickets + static_cast<int64_t>(s) * nh + hh;
        const unsigned tk = atomicAdd(ticket, 1u);
        __threadfence();
        *merge_flag = (tk == static_cast<unsigned>(nparts - 1));
        if (tk == static_cast<unsigned>(nparts - 1)) *ticket = 0u;   // reset for the next run
    }
    if (!epi_sync()) return;
    if (!*merge_flag) return;
    // every softmax thread merges: 128 / M threads a row, D * M / 128 columns each
    constexpr int kTpr = TG::kSoftmaxThreads / M;   // threads per row
    constexpr int kCols = D / kTpr;                 // columns per thread
    const int mr = static_cast<int>(threadIdx.x) / kTpr;
    const int mrow = rg * TG::kRows + mr;
    const int cb = (static_cast<int>(threadIdx.x) % kTpr) * kCols;
    // Partitions that fit the (now idle) K/V ring: all of them copied in at once (every
    // thread's 16-byte copies in flight together), then summed from shared memory; more
    // partitions than fit: straight from global memory, four partitions' loads at a time.
    constexpr int kPartBytes = M * D * 4;
    constexpr int kFit = static_cast<int>(TG::kRing / kPartBytes);
    static_assert(kFit >= 1, "one partition's rows fit the ring");
    const float2* ml = a.ws_ml + (prow0 + mrow) * a.max_parts;
    const float* wo = a.ws_o + (prow0 + mrow) * a.max_parts * D;
    float* part_sm = reinterpret_cast<float*>(smem);
    const bool staged = nparts <= kFit;
    if (staged) {
        constexpr int kVec = D / 4;                 // 16-byte pieces of a row
        const int pieces = nparts * M * kVec;
        for (int i = threadIdx.x; i < pieces; i += TG::kSoftmaxThreads) {
            const int j = i / (M * kVec), rem = i - j * (M * kVec);
            const int r = rem / kVec, c4 = rem - r * kVec;
            const int grow = rg * TG::kRows + r;
            if (grow >= R) continue;
            const float* src = a.ws_o + ((prow0 + grow) * a.max_parts + j) * D + 4 * c4;
            const uint32_t dst = smem_u32(part_sm + (static_cast<size_t>(j) * M + r) * D + 4 * c4);
            cp_async_16(dst, src);
        }
        cp_async_commit();
    }
    // the rows' (maximum, sum) pairs, up to 8 at once
    constexpr int kMl = 8;
    static_assert(kFit <= kMl, "staged partitions have their weights in registers");
    float2 e[kMl];
#pragma unroll
    for (int p = 0; p < kMl; ++p)
        e[p] = (p < nparts && mrow < R) ? __ldcg(ml + p) : make_float2(-INFINITY, 0.0f);
    float mmax = -INFINITY;
#pragma unroll
    for (int p = 0; p < kMl; ++p) mmax = fmaxf(mmax, e[p].x);
    for (int p = kMl; p < nparts && mrow < R; ++p) mmax = fmaxf(mmax, __ldcg(ml + p).x);
    float den = 0.0f;
#pragma unroll
    for (int p = 0; p < kMl; ++p) den += e[p].x == -INFINITY ? 0.0f : fast_exp2(e[p].x - mmax) * e[p].y;
    for (int p = kMl; p < nparts && mrow < R; ++p) {
        const float2 x = __ldcg(ml + p);
        den += x.x == -INFINITY ? 0.0f : fast_exp2(x.x - mmax) * x.y;
    }
    const float inv = den > 0.0f ? 1.0f / den : 0.0f;
    if (staged) {
        cp_async_wait_all();
        if (!epi_sync()) return;                    // every thread's pieces landed
    }
    if (mrow >= R) return;
    T* orow = out + tc_row_offset(a, s, kvh, mrow) * D;
#pragma unroll 1
    for (int c0 = cb; c0 < cb + kCols; c0 += 16) {
        float num[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) num[jj] = 0.0f;
        if (staged) {
            for (int p = 0; p < nparts; ++p) {
                const float w = p < kMl ? (e[p].x == -INFINITY ? 0.0f : fast_exp2(e[p].x - mmax)) : 0.0f;
                const float4* src = reinterpret_cast<const float4*>(part_sm + (static_cast<size_t>(p) * M + mr) * D + c0);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float4 v = src[jj];
                    num[4 * jj] += w * v.x;
                    num[4 * jj + 1] += w * v.y;
                    num[4 * jj + 2] += w * v.z;
                    num[4 * jj + 3] += w * v.w;
                }
            }
        } else {
#pragma unroll 1
            for (int p0 = 0; p0 < nparts; p0 += 4) {
                float w[4];
                float4 v[4][4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int p = p0 + q;
                    w[q] = 0.0f;
                    if (p < nparts) {
                        const float2 x = __ldcg(ml + p);
                        w[q] = x.x == -INFINITY ? 0.0f : fast_exp2(x.x - mmax);
                        const float4* src = reinterpret_cast<const float4*>(wo + static_cast<int64_t>(p) * D + c0);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) v[q][jj] = __ldcg(src + jj);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) v[q][jj] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        num[4 * jj] += w[q] * v[q][jj].x;
                        num[4 * jj + 1] += w[q] * v[q][jj].y;
                        num[4 * jj + 2] += w[q] * v[q][jj].z;
                        num[4 * jj + 3] += w[q] * v[q][jj].w;
                    }
                }
            }
        }
        uint32_t wv[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) wv[jj] = pack2<T>(num[2 * jj] * inv, num[2 * jj + 1] * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
        dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    }
}

template <typename T, int D, int M>
cudaError_t launch_tc(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    using TG = TcGeo<D, M>;
    constexpr size_t smem = TG::kBytes;
    static_assert(2 * (smem + 1024) <= 233472, "two CTAs per SM fit the shared memory");
    static_assert(TG::kP % 1024 == 0, "the P tile starts on a swizzle atom");
    static_assert(TG::kStages % 2 == 0 && TG::kStages >= 4, "a step's stages are adjacent; two steps in flight");
    auto kern = verify_tc_kernel<T, D, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned nh = static_cast<unsigned>(a.num_kv_heads * a.head_groups);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = a.plan ? dim3(nh * static_cast<unsigned>(a.plan_capacity))
                         : dim3(nh, static_cast<unsigned>(a.direct_parts), static_cast<unsigned>(a.num_seqs));
    cfg.blockDim = dim3(TG::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, a);
}

}  // namespace

cudaError_t launch_verify_tc(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
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
    const bool m64 = verify_tc_rows_per_cta(a.group) == 64;
    if (dtype == 0) {
        if (head_dim == 128) return m64 ? launch_tc<__half, 128, 64>(a, tmk, tmv, s) : launch_tc<__half, 128, 128>(a, tmk, tmv, s);
        return m64 ? launch_tc<__half, 64, 64>(a, tmk, tmv, s) : launch_tc<__half, 64, 128>(a, tmk, tmv, s);
    }
    if (head_dim == 128)
        return m64 ? launch_tc<__nv_bfloat16, 128, 64>(a, tmk, tmv, s) : launch_tc<__nv_bfloat16, 128, 128>(a, tmk, tmv, s);
    return m64 ? launch_tc<__nv_bfloat16, 64, 64>(a, tmk, tmv, s) : launch_tc<__nv_bfloat16, 64, 128>(a, tmk, tmv, s);
}

int verify_tc_rows_per_cta(int rows) { return rows <= 64 ? 64 : kVerifyTcRows; }

// CTAs of the verify kernel an SM holds at once, from its resources: tensor memory (each CTA
// allocates kTmemCols of the SM's 512 columns), shared memory, and registers, where an SM's
// four sub-partitions each hold a quarter of the register file and take the resident warps in
// turn.  (cudaOccupancyMaxActiveBlocksPerMultiprocessor answers 1 for this kernel, while the
// hardware runs 2 at a time on every SM; the partition rule needs the real count.)
int verify_tc_ctas_per_sm(int head_dim) {
    static std::atomic<int> cache[2] = {-1, -1};   // head_dim 64, 128; the same on every GB300
    const int i = head_dim == 64 ? 0 : 1;
    int n = cache[i].load(std::memory_order_relaxed);
    if (n < 0) {
        auto fit = [](auto kern, size_t smem, int tmem_cols) -> int {
            cudaFuncAttributes fa{};
            int dev = 0, smem_sm = 0, reserved = 0, regs_sm = 0;
            if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess)
                return 1;
            const int warps = (TcGeo<128, 64>::kThreads + 31) / 32;
            const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;
            int k = 512 / tmem_cols;
            while (k > 1 && (static_cast<size_t>(k) * (smem + reserved) > static_cast<size_t>(smem_sm) ||
                             (k * warps + 3) / 4 * regs_warp > regs_sm / 4))
                --k;
            return k;
        };
        n = i == 0 ? std::min(fit(verify_tc_kernel<__half, 64, 128>, TcGeo<64, 128>::kBytes, TcGeo<64, 128>::kTmemCols),
                              fit(verify_tc_kernel<__half, 64, 64>, TcGeo<64, 64>::kBytes, TcGeo<64, 64>::kTmemCols))
                   : std::min(fit(verify_tc_kernel<__half, 128, 128>, TcGeo<128, 128>::kBytes, TcGeo<128, 128>::kTmemCols),
                              fit(verify_tc_kernel<__half, 128, 64>, TcGeo<128, 64>::kBytes, TcGeo<128, 64>::kTmemCols));
        cache[i].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace pkv
