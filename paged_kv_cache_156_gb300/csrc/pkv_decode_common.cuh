// Pieces of the decode kernel: the shared memory geometry of a chunk, the
// per-chunk consumer arithmetic and the epilogue that merges warps and
// partitions; MQ instantiates the multi-query (verify) form.
#pragma once

#include <cuda_fp8.h>
#include <float.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace dec {

constexpr int kMaxTable = kPlanTableEntries;   // staged table entries: part_tokens (<= 4096) / block_size (>= 8)
constexpr int kHeadsPerCta = dec_heads_per_cta();   // mma N: query rows served by one CTA

// CW consumer warps each own 16 positions of a chunk of 16 * CW positions;
// EB is the pool's element size (2: fp16 / bf16; 1: E4M3 codes).
template <int D, int CW, int EB = 2>
struct Geo {
    static constexpr int kChunk = 16 * CW;              // positions per pipeline stage
    static constexpr int kConsumers = 32 * CW;
    static constexpr int kThreads = kConsumers + 32;    // plus one producer warp
    static constexpr int kHalves = D * EB / 128;        // 128-byte column planes
    static constexpr int kPlane = kChunk * 128;         // bytes of one plane of a chunk
    static constexpr int kStage = kHalves * kPlane;     // bytes of K (or V) of one chunk
    static constexpr int kScratch = (CW * kHeadsPerCta * (D + 2) + 2 * kHeadsPerCta) * 4;  // merge scratch
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

__device__ __forceinline__ void raise_abort(unsigned* err, volatile int* abort_flag) {
    if (!*abort_flag) raise_error(err, kErrTimeout);
    *abort_flag = 1;
}

// MQ (template flag) selects the multi-query (verify) form of the helpers
// below; the decode kernels compile with MQ = false and carry none of it.
//
// Query rows.  A KV head serves `group` query rows: for query token i of the
// sequence (0 <= i < num_queries) and query head hl of the KV head's
// `qgroup`, row vh = i * qgroup + hl.  q and out are [B][num_queries][Hq][D].
// An item (sequence s, KV head kvh, rows vh0 .. vh0 + 7) is addressed by
// sh0, the row of vh0 in the split-K partials ([B][Hq * nq][parts]); with one
// query token that is also the row of vh0 in q and out, and row vh0 + hx is
// sh0 + hx in all three.
template <bool MQ>
__device__ __forceinline__ int64_t item_row0(const DecodeArgs& a, int s, int kvh, int vh0) {
    if constexpr (MQ)
        return static_cast<int64_t>(s) * a.num_heads * a.num_queries + static_cast<int64_t>(kvh) * a.group + vh0;
    else
        return static_cast<int64_t>(s) * a.num_heads + kvh * a.group + vh0;
}

// Row of q / out (element offset / D) of the item's row vh0 + hx.
template <bool MQ>
__device__ __forceinline__ int64_t qo_row(const DecodeArgs& a, int64_t sh0, int s, int kvh, int vh0, int hx) {
    if constexpr (MQ) {
        const int vh = vh0 + hx;
        const int i = vh / a.qgroup;
        const int hl = vh - i * a.qgroup;
        return (static_cast<int64_t>(s) * a.num_queries + i) * a.num_heads + kvh * a.qgroup + hl;
    } else {
        return sh0 + hx;
    }
}

// Exclusive causal limit of query row vh: query token i of a sequence of L
// positions (its last num_queries being the queries' own) sees positions
// < L - num_queries + i + 1; for decode (one query) that is all L positions.
template <bool MQ>
__device__ __forceinline__ int causal_limit(const DecodeArgs& a, int L, int vh) {
    return MQ ? L - a.num_queries + vh / a.qgroup + 1 : L;
}

// One consumer warp's running state for one work item: O^T accumulators
// (d x 8 heads, fp32), running max and sum of its two head columns, and the
// Q^T operand fragments.
template <int D>
struct WarpState {
    float o[D / 16][4];
    float m0, m1, l0, l1;
    uint32_t qb[D / 16][2];
};

template <int D>
__device__ __forceinline__ void reset_state(WarpState<D>& w) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) w.o[mt][0] = w.o[mt][1] = w.o[mt][2] = w.o[mt][3] = 0.0f;
    w.m0 = w.m1 = -INFINITY;
    w.l0 = w.l1 = 0.0f;
}

// Score masks of one lane for one 16-position tile: bit 0 (row r0, column
// 2t), bit 1 (row r0, column 2t + 1), bit 2 (row r0 + 8, column 2t), bit 3
// (row r0 + 8, column 2t + 1), with r0 = lane / 4 and t = lane % 4.  A tile's
// zero-row mask has bit r set for each of its 16 rows that holds no token
// (past the stream, or a slot outside every column's range).
__device__ __forceinline__ unsigned tile_vis(bool va, bool vb) { return (va ? 3u : 0u) | (vb ? 12u : 0u); }
__device__ __forceinline__ unsigned tail_rows(int nv) { return nv < 16 ? (0xFFFFu << max(nv, 0)) & 0xFFFFu : 0u; }

// One warp's 16 positions of a chunk: S^T = K Q^T on the tensor cores, online
// softmax over those scores (log2 domain, masked by `vis`), then O^T += V^T
// P^T.  `warp` selects the 16 rows of the chunk; kst / vst are the stage's K
// and V ring addresses; rows in `zrows` have their V zeroed first (their
// slots may hold NaN).  `guard`: a column may have seen no position yet (its
// maximum is still -inf), so its rescale is 1 and its weights 0.
template <typename T, int D, int CW>
__device__ __forceinline__ void consume_chunk(WarpState<D>& w, uint32_t kst, uint32_t vst, unsigned zrows,
                                              unsigned vis, bool guard, int warp, int lane, float sl2) {
    using G = Geo<D, CW>;
    using M = Mma<T>;
    const int krow = warp * 16 + (lane & 15);                     // ldmatrix row supplied by this lane (K)
    const int kcol = lane >> 4;                                    // +8 elements
    const int vrow = warp * 16 + (lane & 7) + ((lane >> 4) << 3);  // (V, transposed load)
    const int vcol = (lane >> 3) & 1;
    if (zrows) {
        // rows that hold no token: zero their V so 0-weights stay 0
        unsigned zr = zrows;
        while (zr) {
            const int r = warp * 16 + __ffs(zr) - 1;
            zr &= zr - 1;
            for (int cc = lane; cc < D / 8; cc += 32) {
                const uint32_t addr = swz(vst + (cc >> 3) * G::kPlane, r, cc & 7);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
            }
        }
        fence_proxy_async_smem();                 // before the async proxy refills this stage
        __syncwarp();
    }
    // ---- S^T = K Q^T
    float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4];
        ldmatrix_x4(af, swz(kst + (ks >> 2) * G::kPlane, krow, (ks & 3) * 2 + kcol));
        M::run(sacc, af, w.qb[ks][0], w.qb[ks][1]);
    }
    // ---- online softmax (log2 domain); columns are heads 2*(lane%4) + {0,1}
    const float s0 = (vis & 1u) ? sacc[0] * sl2 : -INFINITY;
    const float s1 = (vis & 2u) ? sacc[1] * sl2 : -INFINITY;
    const float s2 = (vis & 4u) ? sacc[2] * sl2 : -INFINITY;
    const float s3 = (vis & 8u) ? sacc[3] * sl2 : -INFINITY;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(w.m0, mx0), mn1 = fmaxf(w.m1, mx1);
    // a column with no visible position yet keeps max -inf: scale 1, weights 0
    // (a one-sequence decode item never has one: row 0 of the warp is always visible)
    const float al0 = (guard && mn0 == -INFINITY) ? 1.0f : fast_exp2(w.m0 - mn0);
    const float al1 = (guard && mn1 == -INFINITY) ? 1.0f : fast_exp2(w.m1 - mn1);
    w.m0 = mn0;
    w.m1 = mn1;
    const float b0 = (guard && mn0 == -INFINITY) ? 0.0f : mn0, b1 = (guard && mn1 == -INFINITY) ? 0.0f : mn1;
    const uint32_t p01 = M::pack(fast_exp2(s0 - b0), fast_exp2(s1 - b1));
    const uint32_t p23 = M::pack(fast_exp2(s2 - b0), fast_exp2(s3 - b1));
    const float2 f01 = M::unpack(p01), f23 = M::unpack(p23);   // the weights PV actually uses
    w.l0 = w.l0 * al0 + f01.x + f23.x;
    w.l1 = w.l1 * al1 + f01.y + f23.y;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        w.o[mt][0] *= al0;
        w.o[mt][1] *= al1;
        w.o[mt][2] *= al0;
        w.o[mt][3] *= al1;
    }
    // ---- O^T += V^T P^T ; P^T fragment = transpose of the score fragment
    const uint32_t pb0 = movmatrix_trans(p01);
    const uint32_t pb1 = movmatrix_trans(p23);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t vf[4];
        ldmatrix_x4_trans(vf, swz(vst + (mt >> 2) * G::kPlane, vrow, (mt & 3) * 2 + vcol));
        M::run(w.o[mt], vf, pb0, pb1);
    }
}

// ---------------------------------------------------------------- 8-bit (E4M3) pools
// Four E4M3 codes (a 32-bit word, byte 0 first) to two f16 pairs: lo =
// (byte 0, byte 1), hi = (byte 2, byte 3), the first of each in the low half.
// Every E4M3 value is exact in f16.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// One warp's 16 positions of a chunk of an E4M3 pool (head_dim 128, one
// 128-byte swizzled plane per stage).  The tensor cores run in f16: each
// lane reads its K and V bytes from shared memory and converts them in
// registers.  The contraction index of S^T = K Q^T is permuted so that a
// lane's K bytes are contiguous: logical k = 16*ks + 2*t + j (t = lane % 4,
// j in {0, 1, 8, 9}) is head-dim element 32*t + 4*ks + {0, 1, 2, 3}[j]; Q is
// loaded in the same order, so the dot products are unchanged.  For O^T =
// V^T P^T the rows of tile mt are head-dim elements 16*g + 2*mt (row g) and
// 16*g + 2*mt + 1 (row g + 8), g = lane / 4, so a lane reads 16 contiguous
// bytes of each of its four positions; warp_state_to_smem_fp8 undoes it.
template <int CW, bool MQ = false>
__device__ __forceinline__ void consume_chunk_fp8(WarpState<128>& w, uint32_t kst, uint32_t vst, int nv, int warp,
                                                  int lane, float sl2, int tokw = 0, int lim0 = 0, int lim1 = 0) {
    using M = Mma<__half>;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = warp * 16 + g;
    // ---- S^T = K Q^T: this lane's 32 bytes of K rows g and g + 8
    const uint4 ka0 = ld_shared_v4(swz(kst, row0, 2 * t)), ka1 = ld_shared_v4(swz(kst, row0, 2 * t + 1));
    const uint4 kb0 = ld_shared_v4(swz(kst, row0 + 8, 2 * t)), kb1 = ld_shared_v4(swz(kst, row0 + 8, 2 * t + 1));
    const uint32_t kra[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
    const uint32_t krb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
    float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4];                            // rows g, g+8 at logical k (2t, 2t+1), then (2t+8, 2t+9)
        e4m3x4_to_f16x2x2(kra[ks], af[0], af[2]);
        e4m3x4_to_f16x2x2(krb[ks], af[1], af[3]);
        M::run(sacc, af, w.qb[ks][0], w.qb[ks][1]);
    }
    // ---- online softmax, as consume_chunk (verify: each column's causal limit)
    const bool va = g < nv, vb = g + 8 < nv;
    const int pa = tokw + g, pb = pa + 8;
    const float s0 = (va && (!MQ || pa < lim0)) ? sacc[0] * sl2 : -INFINITY;
    const float s1 = (va && (!MQ || pa < lim1)) ? sacc[1] * sl2 : -INFINITY;
    const float s2 = (vb && (!MQ || pb < lim0)) ? sacc[2] * sl2 : -INFINITY;
    const float s3 = (vb && (!MQ || pb < lim1)) ? sacc[3] * sl2 : -INFINITY;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(w.m0, mx0), mn1 = fmaxf(w.m1, mx1);
    // verify: a column with no visible position yet keeps max -inf: scale 1, weights 0
    const float al0 = (MQ && mn0 == -INFINITY) ? 1.0f : fast_exp2(w.m0 - mn0);
    const float al1 = (MQ && mn1 == -INFINITY) ? 1.0f : fast_exp2(w.m1 - mn1);
    w.m0 = mn0;
    w.m1 = mn1;
    const float b0 = (MQ && mn0 == -INFINITY) ? 0.0f : mn0, b1 = (MQ && mn1 == -INFINITY) ? 0.0f : mn1;
    const uint32_t p01 = M::pack(fast_exp2(s0 - b0), fast_exp2(s1 - b1));
    const uint32_t p23 = M::pack(fast_exp2(s2 - b0), fast_exp2(s3 - b1));
    const float2 f01 = M::unpack(p01), f23 = M::unpack(p23);
    w.l0 = w.l0 * al0 + f01.x + f23.x;
    w.l1 = w.l1 * al1 + f01.y + f23.y;
    // the accumulators need rescaling only when some column's maximum moved
    if (__any_sync(0xffffffffu, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            w.o[mt][0] *= al0;
            w.o[mt][1] *= al1;
            w.o[mt][2] *= al0;
            w.o[mt][3] *= al1;
        }
    }
    // ---- O^T += V^T P^T: bytes 16g .. 16g+15 of positions 2t, 2t+1, 2t+8, 2t+9;
    // positions past seq_len may hold NaN codes and are zeroed
    const uint32_t pb0 = movmatrix_trans(p01);
    const uint32_t pb1 = movmatrix_trans(p23);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 v0 = 2 * t < nv ? ld_shared_v4(swz(vst, warp * 16 + 2 * t, g)) : z;
    const uint4 v1 = 2 * t + 1 < nv ? ld_shared_v4(swz(vst, warp * 16 + 2 * t + 1, g)) : z;
    const uint4 v2 = 2 * t + 8 < nv ? ld_shared_v4(swz(vst, warp * 16 + 2 * t + 8, g)) : z;
    const uint4 v3 = 2 * t + 9 < nv ? ld_shared_v4(swz(vst, warp * 16 + 2 * t + 9, g)) : z;
    const uint32_t V0[4] = {v0.x, v0.y, v0.z, v0.w}, V1[4] = {v1.x, v1.y, v1.z, v1.w};
    const uint32_t V2[4] = {v2.x, v2.y, v2.z, v2.w}, V3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int r = mt >> 1, b = (mt & 1) * 2;           // bytes 2mt, 2mt + 1 of the 16
        const unsigned sel = b | ((4 + b) << 4) | ((b + 1) << 8) | ((5 + b) << 12);
        const uint32_t x01 = __byte_perm(V0[r], V1[r], sel);   // (pos 2t, 2t+1) at d, then at d + 1
        const uint32_t x89 = __byte_perm(V2[r], V3[r], sel);   // (pos 2t+8, 2t+9)
        uint32_t vf[4];
        e4m3x4_to_f16x2x2(x01, vf[0], vf[1]);
        e4m3x4_to_f16x2x2(x89, vf[2], vf[3]);
        M::run(w.o[mt], vf, pb0, pb1);
    }
}

// As warp_state_to_smem for the E4M3 path: undoes the head-dim permutation of
// consume_chunk_fp8 and applies the V scale to the partial output.
template <int CW>
__device__ __forceinline__ void warp_state_to_smem_fp8(const WarpState<128>& w, float* scratch, int warp, int lane,
                                                       float vscale) {
    float l0 = w.l0, l1 = w.l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* sm_m = scratch;
    float* sm_l = sm_m + CW * kHeadsPerCta;
    float* sm_o = sm_l + CW * kHeadsPerCta;
    if (lane < 4) {
        sm_m[warp * kHeadsPerCta + 2 * lane] = w.m0;
        sm_m[warp * kHeadsPerCta + 2 * lane + 1] = w.m1;
        sm_l[warp * kHeadsPerCta + 2 * lane] = l0;
        sm_l[warp * kHeadsPerCta + 2 * lane + 1] = l1;
    }
    const int hA = 2 * (lane & 3);
    float* oa = sm_o + (warp * kHeadsPerCta + hA) * 128;
    float* ob = oa + 128;
    const int g = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int d0 = 16 * g + 2 * mt;
        oa[d0] = w.o[mt][0] * vscale;
        ob[d0] = w.o[mt][1] * vscale;
        oa[d0 + 1] = w.o[mt][2] * vscale;
        ob[d0 + 1] = w.o[mt][3] * vscale;
    }
}

// This warp's (max, sum, O) into the merge scratch: m[CW][8], l[CW][8], o[CW][8][D].
template <int D, int CW>
__device__ __forceinline__ void warp_state_to_smem(const WarpState<D>& w, float* scratch, int warp, int lane) {
    float l0 = w.l0, l1 = w.l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* sm_m = scratch;
    float* sm_l = sm_m + CW * kHeadsPerCta;
    float* sm_o = sm_l + CW * kHeadsPerCta;
    if (lane < 4) {
        sm_m[warp * kHeadsPerCta + 2 * lane] = w.m0;
        sm_m[warp * kHeadsPerCta + 2 * lane + 1] = w.m1;
        sm_l[warp * kHeadsPerCta + 2 * lane] = l0;
        sm_l[warp * kHeadsPerCta + 2 * lane + 1] = l1;
    }
    const int hA = 2 * (lane & 3);
    float* oa = sm_o + (warp * kHeadsPerCta + hA) * D;
    float* ob = oa + D;
    const int r0 = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int d0 = mt * 16 + r0;
        oa[d0] = w.o[mt][0];
        ob[d0] = w.o[mt][1];
        oa[d0 + 8] = w.o[mt][2];
        ob[d0 + 8] = w.o[mt][3];
    }
}

// Where column hx of an item goes: its row of the split-K partials and its
// row of the output (element offset / D).
struct ItemRows {
    int64_t sh0;          // partial (and decode output) row of column 0 of a one-sequence item
    int s, kvh, vh0;
    int unit;             // members of a shared-prefix unit (> 1), else 1
    __device__ __forceinline__ int64_t unit_row(const DecodeArgs& a, int hx) const {
        return static_cast<int64_t>(s + hx / a.group) * a.num_heads + kvh * a.group + hx % a.group;
    }
    template <bool MQ>
    __device__ __forceinline__ int64_t ws(const DecodeArgs& a, int hx) const {
        return unit > 1 ? unit_row(a, hx) : sh0 + hx;
    }
    template <bool MQ>
    __device__ __forceinline__ int64_t out(const DecodeArgs& a, int hx) const {
        return unit > 1 ? unit_row(a, hx) : qo_row<MQ>(a, sh0, s, kvh, vh0, hx);
    }
};

// Combine the warps' states of one item (scratch written and synchronised):
// a sequence of one partition gets its output; otherwise the partition's
// (max, sum, unnormalised output) go to the workspace.  `guard`: a column may
// have seen nothing in this item (its warps' maxima are all -inf).
template <typename T, int D, int CW, bool MQ>
__device__ __forceinline__ void combine_warps(const DecodeArgs& a, const float* scratch, const ItemRows& rows, int gc,
                                              int part, int nparts, int tid, bool guard) {
    const float* sm_m = scratch;
    const float* sm_l = sm_m + CW * kHeadsPerCta;
    const float* sm_o = sm_l + CW * kHeadsPerCta;
    T* out = reinterpret_cast<T*>(a.out);
    for (int idx = tid; idx < gc * D; idx += 32 * CW) {
        const int hx = idx / D;
        const int d = idx - hx * D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < CW; ++w) mx = fmaxf(mx, sm_m[w * kHeadsPerCta + hx]);
        float den = 0.0f, num = 0.0f;
#pragma unroll
        for (int w = 0; w < CW; ++w) {
            const float mw = sm_m[w * kHeadsPerCta + hx];
            // a warp that saw nothing adds nothing (without the guard mx is finite and the weight 0 anyway)
            const float wt = (guard && mw == -INFINITY) ? 0.0f : fast_exp2(mw - mx);
            den += wt * sm_l[w * kHeadsPerCta + hx];
            num += wt * sm_o[(w * kHeadsPerCta + hx) * D + d];
        }
        if (nparts == 1) {
            out[rows.out<MQ>(a, hx) * D + d] = T(guard ? (den > 0.0f ? num / den : 0.0f) : num / den);
        } else {
            const int64_t sh = rows.ws<MQ>(a, hx);
            a.ws_o[(sh * a.max_parts + part) * D + d] = num;
            if (d == 0) a.ws_ml[sh * a.max_parts + part] = make_float2(mx, den);
        }
    }
}

// Merge every partition of (sequence, head group) into the output; run by the
// CTA that took the last ticket.  Up to four partitions: each thread first loads
// every partition's value of its output elements (they do not depend on the
// maxima), then one warp per head turns the partitions' (maximum, sum) pairs
// into normalised weights in shared memory; one round trip in all.  More
// partitions: phase A (one warp per head) puts the maximum and the denominator
// into msm[8] / dsm[8]; `sync` separates the phases; phase B: each output
// element sums its partials with four partitions' loads in flight.  Partitions
// are summed in partition order either way.
template <typename T, int D, int CW, bool MQ, typename Sync>
__device__ __forceinline__ bool merge_partitions(const DecodeArgs& a, float* scratch, const ItemRows& rows, int gc,
                                                 int nparts, int warp, int lane, int tid, Sync&& sync) {
    if (nparts <= 4) {
        constexpr int kConsumers = 32 * CW;
        static_assert(kConsumers >= D, "one pass over d");
        constexpr int kRows = kConsumers / D;       // heads covered per pass
        constexpr int kAcc = (kHeadsPerCta + kRows - 1) / kRows;
        const int d = tid % D;
        const int hb = tid / D;
        float v[kAcc][4];
#pragma unroll
        for (int k = 0; k < kAcc; ++k) {
            const int hx = hb + k * kRows;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[k][j] = (j < nparts && hx < gc) ? __ldcg(a.ws_o + (rows.ws<MQ>(a, hx) * a.max_parts + j) * D + d)
                                                  : 0.0f;
        }
        float* wsm = scratch;                       // [kHeadsPerCta][4] normalised weights
        for (int hx = warp; hx < gc; hx += CW) {
            const float2 e = lane < nparts ? __ldcg(a.ws_ml + rows.ws<MQ>(a, hx) * a.max_parts + lane)
                                           : make_float2(-INFINITY, 0.0f);
            float mx = e.x;
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float w = e.x == -INFINITY ? 0.0f : fast_exp2(e.x - mx);
            float den = w * e.y;
            den += __shfl_xor_sync(0xffffffffu, den, 1);
            den += __shfl_xor_sync(0xffffffffu, den, 2);
            if (lane < 4) wsm[hx * 4 + lane] = den > 0.0f ? w / den : 0.0f;
        }
        if (!sync()) return false;
        T* out = reinterpret_cast<T*>(a.out);
#pragma unroll
        for (int k = 0; k < kAcc; ++k) {
            const int hx = hb + k * kRows;
            if (hx >= gc) continue;
            float num = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) num += wsm[hx * 4 + j] * v[k][j];
            out[rows.out<MQ>(a, hx) * D + d] = T(num);
        }
        return true;
    }
    float* msm = scratch;
    float* dsm = scratch + kHeadsPerCta;
    for (int hx = warp; hx < gc; hx += CW) {
        const float2* ml = a.ws_ml + rows.ws<MQ>(a, hx) * a.max_parts;
        float mx = -INFINITY;
        for (int p = lane; p < nparts; p += 32) mx = fmaxf(mx, __ldcg(ml + p).x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float den = 0.0f;
        for (int p = lane; p < nparts; p += 32) {
            const float2 e = __ldcg(ml + p);
            den += fast_exp2(e.x - mx) * e.y;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (lane == 0) {
            msm[hx] = mx;
            dsm[hx] = den;
        }
    }
    if (!sync()) return false;
    constexpr int kConsumers = 32 * CW;
    constexpr int kRows = kConsumers / D > 0 ? kConsumers / D : 1;   // heads covered per pass
    constexpr int kAcc = (kHeadsPerCta + kRows - 1) / kRows;
    T* out = reinterpret_cast<T*>(a.out);
    for (int base = 0; base < D; base += kConsumers) {               // D > kConsumers: several passes over d
        const int d = base + (kConsumers >= D ? tid % D : tid);
        const int hb = kConsumers >= D ? tid / D : 0;
        float num[kAcc];
        float mk[kAcc];
#pragma unroll
        for (int k = 0; k < kAcc; ++k) {
            num[k] = 0.0f;
            const int hx = hb + k * kRows;
            mk[k] = hx < gc ? msm[hx] : 0.0f;
        }
        // partitions in groups of 4 so that 4 * kAcc independent load pairs are in flight
        int p = 0;
        for (; p + 4 <= nparts; p += 4) {
            float e[4][kAcc], v[4][kAcc];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int k = 0; k < kAcc; ++k) {
                    const int hx = hb + k * kRows;
                    const int64_t row = rows.ws<MQ>(a, hx < gc ? hx : 0) * a.max_parts + p + j;
                    e[j][k] = __ldcg(reinterpret_cast<const float*>(a.ws_ml + row));
                    v[j][k] = __ldcg(a.ws_o + row * D + d);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int k = 0; k < kAcc; ++k) num[k] += fast_exp2(e[j][k] - mk[k]) * v[j][k];
            }
        }
        for (; p < nparts; ++p) {
#pragma unroll
            for (int k = 0; k < kAcc; ++k) {
                const int hx = hb + k * kRows;
                if (hx < gc) {
                    const int64_t row = rows.ws<MQ>(a, hx) * a.max_parts + p;
                    num[k] += fast_exp2(__ldcg(a.ws_ml + row).x - mk[k]) * __ldcg(a.ws_o + row * D + d);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kAcc; ++k) {
            const int hx = hb + k * kRows;
            if (hx < gc)
                out[rows.out<MQ>(a, hx) * D + d] =
                    T(MQ ? (dsm[hx] > 0.0f ? num[k] / dsm[hx] : 0.0f) : num[k] / dsm[hx]);
        }
    }
    return true;
}

}  // namespace dec
}  // namespace pkv
