// paged_attention_decode: one query token per sequence over its paged K/V.
//
// What is computed ("tbr8.org PagedAttention article" §2.2; "LLM 推理引擎内部原理"
// §2.4): for each sequence s and query head h, walk the logical blocks of s,
// look each one up in the block table, read K/V rows of KV head
// g = h / group up to seq_len, and return softmax(scale * q.K) V.
//
// How (sm_103a):
//  * One CTA per (KV head, group of <= 8 query heads, partition of
//    part_tokens positions, sequence).  All query heads that share a KV head
//    are served from the same K/V bytes, so each byte of the pool is read from
//    HBM once per step.
//  * The CTA's slice of the block table is staged in shared memory once; a
//    producer warp then streams the partition's K and V tiles with TMA
//    (cp.async.bulk.tensor, one box = one (physical block, KV head) tile of
//    block_size rows x 64 elements, 128B-swizzled) into a ring of STAGES
//    chunks of 64 positions, synchronised with mbarriers.
//  * Four consumer warps each own 16 positions of every chunk.  Scores are a
//    small dense contraction over the query-head group, done on the tensor
//    cores with keys as the M dimension: S^T[16 pos x 8 heads] = K Q^T
//    (mma.m16n8k16, fp32 accumulate).  Each warp keeps an fp32 online softmax
//    (running max and sum per head, log2 domain), rounds the weights to the
//    input type, transposes them in registers (movmatrix) and accumulates
//    O^T[d x 8 heads] += V^T P^T, again on the tensor cores.
//  * Positions past seq_len are masked: their scores are replaced by -inf and
//    their V rows in shared memory are zeroed (the slots hold no token and may
//    be NaN), so nothing beyond seq_len contributes.
//  * At the end the four warps' states are merged through shared memory.  A
//    sequence that fits one partition writes its output directly; otherwise
//    each partition writes (max, sum, unnormalised output) and the merge
//    kernel combines them (split-K over the sequence):
//        M = max_p m_p,  out = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p.
#include <float.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kChunk = 64;           // positions per pipeline stage
constexpr int kConsumerWarps = 4;    // each owns 16 positions of a chunk
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxTable = 512;       // staged table entries: part_tokens (<= 4096) / block_size (>= 8)
constexpr int kHeadsPerCta = 8;      // mma N

template <int D>
struct Geo {
    static constexpr int kHalves = D / 64;              // 64-element (128-byte) column planes
    static constexpr int kPlane = kChunk * 128;         // bytes of one plane of a chunk
    static constexpr int kStage = kHalves * kPlane;     // bytes of K (or V) of one chunk
    static constexpr int kPitch = D + 4;                // fp32 pitch of the merge scratch
};

template <int D, int STAGES>
constexpr size_t smem_bytes() {
    return 1024 /* alignment slack */ + 2 * STAGES * Geo<D>::kStage + 2 * STAGES * sizeof(uint64_t) +
           kMaxTable * sizeof(int) + 16;
}

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

template <typename T, int D, int STAGES>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv,
                                                         const DecodeArgs a) {
    using G = Geo<D>;
    using M = Mma<T>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* kring = smem;
    uint8_t* vring = smem + STAGES * G::kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(vring + STAGES * G::kStage);
    uint64_t* empty = full + STAGES;
    int* tbl = reinterpret_cast<int*>(empty + STAGES);
    volatile int* abort_flag = tbl + kMaxTable;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hgi = blockIdx.x % a.head_groups;
    const int kvh = blockIdx.x / a.head_groups;
    const int part = blockIdx.y;
    const int s = blockIdx.z;
    const int h0 = kvh * a.group + hgi * kHeadsPerCta;
    const int gc = min(kHeadsPerCta, a.group - hgi * kHeadsPerCta);
    const int L = a.seq_lens[s];
    const int start = part * a.part_tokens;
    T* out = reinterpret_cast<T*>(a.out);

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
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer warp
    if (warp == kConsumerWarps) {
        const int bs = a.block_size;
        const int nblk = (end - start + bs - 1) / bs;
        const int32_t* row = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + start / bs;
        for (int i = lane; i < nblk; i += 32) {
            int b = row[i];
            if (b < 0 || static_cast<int64_t>(b) >= a.num_blocks) {
                raise_error(a.err, kErrBounds);
                b = -1;                             // out of the tensor map: TMA fills zeros, reads nothing
            }
            tbl[i] = b;
        }
        __syncwarp();
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            const int per_chunk = kChunk / bs;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % STAGES;
                const unsigned ph = (c / STAGES) & 1;
                if (!wait_or_abort(&empty[st], ph ^ 1, abort_flag)) {
                    if (!*abort_flag) raise_error(a.err, kErrTimeout);
                    *abort_flag = 1;
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

    // ------------------------------------------------------------ consumer warps
    // Q^T as the B operand (k = head_dim, n = query head): lane holds
    // q[n = lane/4][k = 16*ks + 2*(lane%4) + {0,1}] and the same at k + 8.
    uint32_t qb[D / 16][2];
    {
        const int n = lane >> 2;
        const int kq = (lane & 3) * 2;
        const int nq = min(n, gc - 1);              // lanes of absent heads read a present row, then drop it
        const uint32_t* qrow =
            reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(a.q) +
                                              (static_cast<int64_t>(s) * a.num_heads + h0 + nq) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qb[ks][0] = n < gc ? __ldg(qrow + (ks * 16 + kq) / 2) : 0u;
            qb[ks][1] = n < gc ? __ldg(qrow + (ks * 16 + 8 + kq) / 2) : 0u;
        }
    }
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
    bool ok = true;

    for (int c = 0; c < nchunks; ++c) {
        const int st = c % STAGES;
        const unsigned ph = (c / STAGES) & 1;
        if (ok) {
            bool got = wait_or_abort(&full[st], ph, abort_flag);
            got = __all_sync(0xffffffffu, got);
            if (!got) {
                if (lane == 0) {
                    if (!*abort_flag) raise_error(a.err, kErrTimeout);
                    *abort_flag = 1;
                }
                ok = false;
            }
        }
        const int tok0 = start + c * kChunk + warp * 16;
        const int nv = min(16, end - tok0);
        const uint32_t kst = smem_u32(kring + st * G::kStage);
        const uint32_t vst = smem_u32(vring + st * G::kStage);
        if (ok && nv > 0) {
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
    }

    // ---- merge the four warps' states (the ring is free: every chunk was consumed)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        lrun0 += __shfl_xor_sync(0xffffffffu, lrun0, off);
        lrun1 += __shfl_xor_sync(0xffffffffu, lrun1, off);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    float* sm_m = reinterpret_cast<float*>(kring);
    float* sm_l = sm_m + kConsumerWarps * kHeadsPerCta;
    float* sm_o = sm_l + kConsumerWarps * kHeadsPerCta;
    if (lane < 4) {
        sm_m[warp * kHeadsPerCta + 2 * lane] = mrun0;
        sm_m[warp * kHeadsPerCta + 2 * lane + 1] = mrun1;
        sm_l[warp * kHeadsPerCta + 2 * lane] = lrun0;
        sm_l[warp * kHeadsPerCta + 2 * lane + 1] = lrun1;
    }
    {
        const int hA = 2 * (lane & 3);
        float* oa = sm_o + (warp * kHeadsPerCta + hA) * G::kPitch;
        float* ob = oa + G::kPitch;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = mt * 16 + r0;
            oa[d0] = o[mt][0];
            ob[d0] = o[mt][1];
            oa[d0 + 8] = o[mt][2];
            ob[d0 + 8] = o[mt][3];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    for (int idx = threadIdx.x; idx < gc * D; idx += kConsumerWarps * 32) {
        const int hh = idx / D;
        const int d = idx - hh * D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, sm_m[w * kHeadsPerCta + hh]);
        float den = 0.0f, num = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = fast_exp2(sm_m[w * kHeadsPerCta + hh] - mx);
            den += wt * sm_l[w * kHeadsPerCta + hh];
            num += wt * sm_o[(w * kHeadsPerCta + hh) * G::kPitch + d];
        }
        const int64_t sh = static_cast<int64_t>(s) * a.num_heads + h0 + hh;
        if (nparts == 1) {
            out[sh * D + d] = T(num / den);
        } else {
            a.ws_o[(sh * a.max_parts + part) * D + d] = num;
            if (d == 0) a.ws_ml[sh * a.max_parts + part] = make_float2(mx, den);
        }
    }
}

// Combine the partitions of every (sequence, query head) whose sequence spans
// more than one partition.  One warp per (sequence, head).
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeArgs a) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t sh = static_cast<int64_t>(blockIdx.x) * 4 + warp;
    if (sh >= static_cast<int64_t>(a.num_seqs) * a.num_heads) return;
    const int s = static_cast<int>(sh / a.num_heads);
    const int L = a.seq_lens[s];
    const int np = (L + a.part_tokens - 1) / a.part_tokens;
    if (np <= 1) return;                            // written directly by the partition kernel
    const float2* ml = a.ws_ml + sh * a.max_parts;
    float mx = -INFINITY;
    for (int p = lane; p < np; p += 32) mx = fmaxf(mx, ml[p].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    constexpr int V = D / 32;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    float den = 0.0f;
    const float* o = a.ws_o + sh * a.max_parts * D + lane * V;
    for (int p = 0; p < np; ++p) {
        const float2 e = ml[p];
        const float w = fast_exp2(e.x - mx);
        den += w * e.y;
        if constexpr (V == 4) {
            const float4 x = *reinterpret_cast<const float4*>(o + p * D);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
            acc[2] += w * x.z;
            acc[3] += w * x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(o + p * D);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
        }
    }
    const float inv = 1.0f / den;
    T* out = reinterpret_cast<T*>(a.out) + sh * D + lane * V;
#pragma unroll
    for (int i = 0; i < V; i += 2) {
        const uint32_t packed = Mma<T>::pack(acc[i] * inv, acc[i + 1] * inv);
        *reinterpret_cast<uint32_t*>(out + i) = packed;
    }
}

template <typename T, int D, int STAGES>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t s) {
    constexpr size_t smem = smem_bytes<D, STAGES>();
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(a.num_kv_heads * a.head_groups), static_cast<unsigned>(a.max_parts),
              static_cast<unsigned>(a.num_seqs));
    decode_kernel<T, D, STAGES><<<grid, kThreads, smem, s>>>(tmk, tmv, a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.max_parts <= 1) return e;
    const int64_t pairs = static_cast<int64_t>(a.num_seqs) * a.num_heads;
    merge_kernel<T, D><<<static_cast<unsigned>((pairs + 3) / 4), 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, cudaStream_t s) {
    constexpr int kStages = 3;
    if (a.num_seqs <= 0) return cudaSuccess;
    if (dtype == 0) {
        return head_dim == 128 ? launch_t<__half, 128, kStages>(a, tmk, tmv, s)
                               : launch_t<__half, 64, kStages>(a, tmk, tmv, s);
    }
    return head_dim == 128 ? launch_t<__nv_bfloat16, 128, kStages>(a, tmk, tmv, s)
                           : launch_t<__nv_bfloat16, 64, kStages>(a, tmk, tmv, s);
}

}  // namespace pkv
