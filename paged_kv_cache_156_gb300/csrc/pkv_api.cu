// The C ABI (include/pkv.h): host-side validation, TMA descriptors, the
// split-K partition choice and dispatch to the kernels.  No torch types, no
// allocation, no state carried between calls beyond per-device caches of
// immutable facts (SM count, the error word's address, configured kernels).
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pkv.h"
#include "pkv_internal.h"

// Device error word (bit meanings in include/pkv.h, pkv_device_error).
__device__ unsigned int g_pkv_error_word;

static_assert(PKV_PLAN_MAX_SEQS == pkv::kPlanMaxSeqs, "plan batch limit: header and kernels agree");

namespace {

thread_local char g_msg[512] = "";

pkv_status fail(pkv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

pkv_status ok() {
    g_msg[0] = '\0';
    return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An NVTX range around each launching call when PKV_NVTX is set in the
// environment: a profiler's timeline then shows which call issued which kernels.
bool nvtx_enabled() {
    static const bool v = getenv("PKV_NVTX") != nullptr;
    return v;
}
struct CallRange {
    bool on;
    explicit CallRange(const char* name) : on(nvtx_enabled()) {
        if (on) nvtxRangePushA(name);
    }
    ~CallRange() {
        if (on) nvtxRangePop();
    }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices];
unsigned* g_err_ptr[kMaxDevices];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int sm_count_of(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

// Address of the error word on the current device (looked up once per device).
unsigned* error_word(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_error_word) == cudaSuccess) g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_err_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

// TMA descriptor of one pool [num_blocks][block_size][num_kv_heads][head_dim]
// of `e`-byte elements (2: fp16 / bf16; 1: E4M3 codes).  One box is one
// (physical block, KV head) tile: block_size rows of 128 bytes (64 or 128
// elements), 128-byte swizzled in shared memory.
pkv_status encode_pool(CUtensorMap* map, const void* base, int64_t num_blocks, int bs, int hkv, int d, int e = 2) {
    auto enc = encode_fn();
    if (!enc) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(bs),
                          static_cast<cuuint64_t>(num_blocks)};
    cuuint64_t strides[3] = {d * e, static_cast<cuuint64_t>(hkv) * d * e,
                             static_cast<cuuint64_t>(bs) * hkv * d * e};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / e), 1, static_cast<cuuint32_t>(bs), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, e == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return PKV_OK;
}

bool valid_dtype(pkv_dtype dt) { return dt == PKV_F16 || dt == PKV_BF16; }
bool valid_block_size(int bs) { return bs == 8 || bs == 16 || bs == 32; }

constexpr int kChunk = 64;
constexpr int kMaxPartition = 4096;
constexpr int kMaxPartsPerSeq = 512;               // partitions of one sequence a decode call accepts

// Partition size for a decode batch.  1024 positions (measured best on the
// 8B- and 70B-shaped batches), grown while a sequence would need more than 512
// partitions.  When the batch, taken as max_seq_len long everywhere, would
// fill fewer than three waves of CTAs, the size in [512, 1024] (multiple of
// 64) whose last wave is fullest is taken instead (a uniform 16 x 4096 batch
// at three CTAs per SM: 640).  Below one wave, halved down to 128 while the
// batch gives fewer than two CTAs per SM.  No step takes a sequence past 512
// partitions unless even 4096 positions do (a max_seq_len above 2M).
int choose_partition(int num_seqs, int num_kv_heads, int head_groups, int max_seq_len, int sms, int ctas_per_sm) {
    auto parts = [&](int q) { return (static_cast<int64_t>(max_seq_len) + q - 1) / q; };
    int p = 1024;
    while (p < kMaxPartition && parts(p) > kMaxPartsPerSeq) p <<= 1;
    const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads * head_groups;
    const int64_t slots = static_cast<int64_t>(sms > 0 ? sms : 152) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    auto waves = [&](int q) { return static_cast<double>(pairs * parts(q)) / slots; };
    if (p == 1024 && waves(1024) >= 1.0 && waves(1024) < 3.0) {
        double best = -1.0;
        int best_p = 1024;
        for (int q = 1024; q >= 512 && parts(q) <= kMaxPartsPerSeq; q -= 64) {
            const double w = waves(q);
            const double fill = w / static_cast<double>(static_cast<int64_t>(w + 0.999999));
            if (fill > best + 1e-9) {
                best = fill;
                best_p = q;
            }
        }
        return best_p;
    }
    while (p > 128 && pairs * parts(p) < 2LL * (sms > 0 ? sms : 152) && parts(p >> 1) <= kMaxPartsPerSeq) p >>= 1;
    return p;
}

pkv_status check_decode_shape(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_seq_len) {
    if (num_seqs < 0 || num_seqs > 65535) return fail(PKV_ERR_INVALID, "num_seqs %d outside [0, 65535]", num_seqs);
    if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PKV_ERR_INVALID, "num_heads %d must be a positive multiple of num_kv_heads %d", num_heads,
                    num_kv_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not built (64 or 128)", head_dim);
    if (max_seq_len < 0) return fail(PKV_ERR_INVALID, "max_seq_len %d < 0", max_seq_len);
    return PKV_OK;
}

int resolve_partition(int num_seqs, int num_heads, int num_kv_heads, int max_seq_len, int partition_tokens,
                      int head_dim) {
    const int group = num_heads / num_kv_heads;
    const int hg = (group + 7) / 8;
    if (partition_tokens > 0) return partition_tokens;
    return choose_partition(num_seqs, num_kv_heads, hg, max_seq_len, sm_count_of(current_device()),
                            pkv::decode_ctas_per_sm(head_dim));
}

// Partials per query row the workspace holds: the longest sequence's
// partitions at the smallest partition size, plus one when the plan may form
// shared-prefix units (at most 4 query rows per KV head): a unit's stream runs
// past the longest member by the other members' own segments.
int64_t partial_slots(int max_seq_len, int part, int rows_per_kv_head) {
    const int64_t base = max_seq_len > 0 ? (static_cast<int64_t>(max_seq_len) + part - 1) / part : 1;
    return base + (rows_per_kv_head <= pkv::dec_heads_per_cta() / 2 ? 1 : 0);
}

size_t workspace_for(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_seq_len, int part) {
    const int64_t max_parts = partial_slots(max_seq_len, part, num_heads / num_kv_heads);
    return pkv::decode_workspace_layout(num_seqs, num_heads, num_kv_heads, head_dim, static_cast<int>(max_parts))
        .total();
}

}  // namespace

namespace pkv {
int set_error_message(int st, const char* msg) {
    snprintf(g_msg, sizeof(g_msg), "%s", msg);
    return st;
}
}  // namespace pkv

extern "C" {

int pkv_version(void) { return 100; }

const char* pkv_last_error(void) { return g_msg; }

pkv_status pkv_paged_kv_append(const void* k, const void* v, void* key_cache, void* value_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                               int block_size, int num_kv_heads, int head_dim, pkv_dtype dt, void* stream) {
    CallRange range_("pkv_paged_kv_append");
    if (num_tokens < 0) return fail(PKV_ERR_INVALID, "num_tokens %lld < 0", static_cast<long long>(num_tokens));
    if (!valid_dtype(dt)) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", static_cast<int>(dt));
    if (num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0)
        return fail(PKV_ERR_INVALID, "num_kv_heads %d / head_dim %d (head_dim must be a positive multiple of 8)",
                    num_kv_heads, head_dim);
    if (block_size <= 0 || num_blocks <= 0)
        return fail(PKV_ERR_INVALID, "block_size %d / num_blocks %lld", block_size, static_cast<long long>(num_blocks));
    if (num_tokens == 0) return ok();
    if (!k || !v || !key_cache || !value_cache || !slot_mapping) return fail(PKV_ERR_INVALID, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return fail(PKV_ERR_INVALID, "tensors must be 16-byte aligned (slot_mapping 8-byte)");
    const int dev = current_device();
    pkv::AppendArgs a;
    a.k = static_cast<const uint4*>(k);
    a.v = static_cast<const uint4*>(v);
    a.key_cache = static_cast<uint4*>(key_cache);
    a.value_cache = static_cast<uint4*>(value_cache);
    a.slots = slot_mapping;
    a.num_tokens = num_tokens;
    a.num_slots = num_blocks * block_size;
    a.row_vecs = num_kv_heads * head_dim * 2 / 16;
    a.err = error_word(dev);
    cudaError_t e = pkv::launch_append(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    return ok();
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_seq_len,
                                  int partition_tokens) {
    if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len) != PKV_OK) return (size_t)-1;
    if (partition_tokens < 0 || partition_tokens > kMaxPartition || partition_tokens % kChunk != 0)
        return (size_t)-1;
    const int part = resolve_partition(num_seqs, num_heads, num_kv_heads, max_seq_len, partition_tokens, head_dim);
    return workspace_for(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, part);
}

int pkv_decode_plan_partition_tokens(const void* workspace, int num_seqs, int num_heads, int num_kv_heads,
                                     void* stream) {
    if (!workspace || num_seqs <= 0 || num_seqs > pkv::kPlanMaxSeqs || num_kv_heads <= 0 || num_heads <= 0 ||
        num_heads % num_kv_heads != 0)
        return -1;
    const pkv::DecodeWorkspace lay = pkv::decode_workspace_layout(num_seqs, num_heads, num_kv_heads, 64, 1);
    int4 first;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&first, static_cast<const char*>(workspace) + lay.ticket_bytes, sizeof(first),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return -1;
    return first.w;
}

int pkv_decode_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_seq_len) {
    if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len) != PKV_OK) return -1;
    return resolve_partition(num_seqs, num_heads, num_kv_heads, max_seq_len, 0, head_dim);
}

}  // extern "C"

namespace {

// The new tokens of a fused slot write + decode call (one per sequence).
struct NewTokens {
    const void* k;
    const void* v;
    const int64_t* slot_mapping;
    bool inputs_ready;              // PKV_INPUTS_READY: pools, tables, lengths and plan final before the launch
};

// Decode (num_queries == 1) and multi-query verify share one path: a KV head
// serves (num_heads / num_kv_heads) * num_queries query rows.  `mode`: plan
// and run (one call), plan only (pkv_decode_plan; q, out and the pools are
// not used), or run only over the plan already in the workspace.
pkv_status attention_call(void* out, const void* q, const void* key_cache, const void* value_cache,
                          const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                          int max_seq_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                          int64_t num_blocks, float scale, pkv_dtype dt, int num_queries, void* workspace,
                          size_t workspace_bytes, int partition_tokens, void* stream, const float* k_scale = nullptr,
                          const float* v_scale = nullptr, pkv::DecodeMode mode = pkv::DecodeMode::kPlanAndRun,
                          bool kv8_plan = false, int64_t sum_seq_lens = 0, const NewTokens* fused = nullptr) {
    const bool runs = mode != pkv::DecodeMode::kPlanOnly;
    pkv_status st = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len);
    if (st != PKV_OK) return st;
    const bool kv8 = runs ? (k_scale || v_scale) : kv8_plan;    // an E4M3 pool (the _fp8 entry points)
    if (kv8 && head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "E4M3 pools: head_dim 128 only");
    if (num_queries < 1 || num_queries > 64) return fail(PKV_ERR_INVALID, "num_queries %d outside [1, 64]", num_queries);
    const int rows = num_heads * num_queries;            // query rows per sequence
    if (!valid_dtype(dt)) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", static_cast<int>(dt));
    if (!valid_block_size(block_size)) return fail(PKV_ERR_UNSUPPORTED, "block_size %d not built (8, 16, 32)", block_size);
    if (num_blocks <= 0 || num_blocks > (int64_t(1) << 31))
        return fail(PKV_ERR_INVALID, "num_blocks %lld outside [1, 2^31]", static_cast<long long>(num_blocks));
    if (max_blocks_per_seq < 0 || static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return fail(PKV_ERR_INVALID, "max_seq_len %d exceeds max_blocks_per_seq %d * block_size %d", max_seq_len,
                    max_blocks_per_seq, block_size);
    if (runs && !isfinite(scale)) return fail(PKV_ERR_INVALID, "scale is not finite");
    if (partition_tokens < 0 || partition_tokens > kMaxPartition || partition_tokens % kChunk != 0)
        return fail(PKV_ERR_INVALID, "partition_tokens %d: 0 or a multiple of 64 up to 4096", partition_tokens);
    if (num_seqs == 0) return ok();
    if (!block_tables || !seq_lens) return fail(PKV_ERR_INVALID, "null pointer");
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return fail(PKV_ERR_INVALID, "tables and lengths must be 4-byte aligned");
    if (runs) {
        if (!out || !q || !key_cache || !value_cache || (kv8 && (!k_scale || !v_scale)))
            return fail(PKV_ERR_INVALID, "null pointer");
        if (kv8 && ((reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u)))
            return fail(PKV_ERR_INVALID, "k_scale / v_scale must be 4-byte aligned");
        if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
            return fail(PKV_ERR_INVALID, "out, q and caches must be 16-byte aligned");
        if (fused) {
            if (num_queries != 1) return fail(PKV_ERR_INVALID, "a fused slot write decodes one query token");
            if (!fused->k || !fused->v || !fused->slot_mapping) return fail(PKV_ERR_INVALID, "null pointer");
            if (!aligned16(fused->k) || !aligned16(fused->v) ||
                (reinterpret_cast<uintptr_t>(fused->slot_mapping) & 7u))
                return fail(PKV_ERR_INVALID, "k and v must be 16-byte aligned (slot_mapping 8-byte)");
        }
    }

    const int dev = current_device();
    const int part = resolve_partition(num_seqs, rows, num_kv_heads, max_seq_len, partition_tokens, head_dim);
    const int64_t base_parts = max_seq_len > 0 ? (static_cast<int64_t>(max_seq_len) + part - 1) / part : 1;
    if (base_parts > kMaxPartsPerSeq)
        return fail(PKV_ERR_UNSUPPORTED, "%lld partitions per sequence (at most %d; use a larger partition_tokens)",
                    static_cast<long long>(base_parts), kMaxPartsPerSeq);
    const int64_t max_parts = partial_slots(max_seq_len, part, rows / num_kv_heads);
    const pkv::DecodeWorkspace lay =
        pkv::decode_workspace_layout(num_seqs, rows, num_kv_heads, head_dim, static_cast<int>(max_parts));
    const size_t need = lay.total();
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(PKV_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu", need,
                    workspace ? workspace_bytes : size_t(0));
    const int group = rows / num_kv_heads;
    if (static_cast<int64_t>(num_kv_heads) * ((group + 7) / 8) * max_parts * num_seqs >= (int64_t(1) << 31))
        return fail(PKV_ERR_UNSUPPORTED, "too many work items");

    CUtensorMap tmk{}, tmv{};
    const int eb = kv8 ? 1 : 2;
    if (runs) {
        if ((st = encode_pool(&tmk, key_cache, num_blocks, block_size, num_kv_heads, head_dim, eb)) != PKV_OK) return st;
        if ((st = encode_pool(&tmv, value_cache, num_blocks, block_size, num_kv_heads, head_dim, eb)) != PKV_OK)
            return st;
    }

    pkv::DecodeArgs a;
    a.out = out;
    a.q = q;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    char* ws = static_cast<char*>(workspace);
    a.tickets = reinterpret_cast<unsigned*>(ws);
    a.plan = num_seqs <= pkv::kPlanMaxSeqs ? reinterpret_cast<int4*>(ws + lay.ticket_bytes) : nullptr;
    a.ws_o = max_parts > 1 ? reinterpret_cast<float*>(ws + lay.ticket_bytes + lay.plan_bytes) : nullptr;
    a.ws_ml = max_parts > 1 ? reinterpret_cast<float2*>(ws + lay.ticket_bytes + lay.plan_bytes + lay.o_bytes)
                            : nullptr;
    a.err = error_word(dev);
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.qgroup = num_heads / num_kv_heads;
    a.num_queries = num_queries;
    a.group = a.qgroup * num_queries;
    // more than kVerifyMinRows query rows per KV head: the tensor-core verify kernel, 64 or 128 rows per CTA
    // (E4M3 pools: the decode kernel's multi-query form, 8 rows per CTA, for any row count)
    const bool verify_kernel = num_queries > 1 && a.group > pkv::kVerifyMinRows && !kv8;
    a.head_groups = verify_kernel ? (a.group + pkv::kVerifyTcRows - 1) / pkv::kVerifyTcRows : (a.group + 7) / 8;
    a.block_size = block_size;
    a.part_tokens = part;
    a.part_auto = partition_tokens == 0;
    a.slots = sm_count_of(dev) * (verify_kernel ? pkv::verify_tc_ctas_per_sm(head_dim)
                                                : pkv::decode_ctas_per_sm(head_dim, kv8));
    a.rule_weight = verify_kernel ? pkv::kRuleVerifyTc : kv8 ? pkv::kRuleDecode8 : pkv::kRuleDecode;
    a.max_seq_len = max_seq_len;
    a.max_parts = static_cast<int>(max_parts);
    a.direct_parts = static_cast<int>(base_parts);
    // work-list entries the grid covers: every (sequence, partition) the longest sequence
    // could need, or, with the lengths' sum known, at most B + sum / P entries (a sequence
    // of length l has max(1, ceil(l / P)) <= 1 + l / P partitions)
    int64_t capacity = static_cast<int64_t>(num_seqs) * max_parts;
    if (sum_seq_lens > 0) {
        capacity = std::min(capacity, static_cast<int64_t>(num_seqs) + sum_seq_lens / part);
        if (partition_tokens == 0) {
            // The plan's automatic size is never below pb = min(max(rule size, part), table
            // span) unless every sequence fits one partition; later adjustments only lower the
            // item count.  So at most B + sum / pb items, and B when no length exceeds pb.
            const int64_t nh = static_cast<int64_t>(a.num_kv_heads) * a.head_groups;
            const int64_t rule = pkv::plan_rule_tokens(sum_seq_lens, nh, a.rule_weight, a.slots > 0 ? a.slots : 1);
            const int64_t pb = std::min<int64_t>(std::max<int64_t>(rule, part),
                                                 static_cast<int64_t>(pkv::kPlanTableEntries) * block_size);
            const int64_t bound = static_cast<int64_t>(num_seqs) + (max_seq_len > pb ? sum_seq_lens / pb : 0);
            capacity = std::min(capacity, bound);
        }
    }
    a.plan_capacity = static_cast<int>(capacity);
    a.sum_seq_lens = sum_seq_lens;
    // shared-prefix units: one query token over 16-bit pools, the members' query heads in one
    // CTA's columns.  (A unit's stream is never longer than its members' lengths' sum, since it
    // shares at least kUnitMinShare positions, so the grid bound above still holds.)
    a.units = num_queries == 1 && !kv8 && a.qgroup <= pkv::dec_heads_per_cta() / 2;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.kv8 = kv8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    if (runs && fused) {
        a.k_new = static_cast<const uint4*>(fused->k);
        a.v_new = static_cast<const uint4*>(fused->v);
        a.slot_mapping = fused->slot_mapping;
        a.key_cache = const_cast<void*>(key_cache);
        a.value_cache = const_cast<void*>(value_cache);
        a.early = fused->inputs_ready && mode == pkv::DecodeMode::kRunOnly && a.plan != nullptr && !kv8 ? 1 : 0;
    }
    cudaError_t e = verify_kernel ? pkv::launch_verify_tc(a, tmk, tmv, dt == PKV_F16 ? 0 : 1, head_dim,
                                                          static_cast<cudaStream_t>(stream), mode)
                                  : pkv::launch_decode(a, tmk, tmv, dt == PKV_F16 ? 0 : 1, head_dim,
                                                       static_cast<cudaStream_t>(stream), mode);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* key_cache, const void* value_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                      int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale, pkv_dtype dt, void* workspace,
                                      size_t workspace_bytes, int partition_tokens, void* stream) {
    CallRange range_("pkv_paged_attention_decode");
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt, 1,
                          workspace, workspace_bytes, partition_tokens, stream);
}

pkv_status pkv_paged_attention_verify(void* out, const void* q, const void* key_cache, const void* value_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                      int num_seqs, int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
                                      pkv_dtype dt, int num_queries, void* workspace, size_t workspace_bytes,
                                      int partition_tokens, void* stream) {
    CallRange range_("pkv_paged_attention_verify");
    if (sum_seq_lens < 0) return fail(PKV_ERR_INVALID, "sum_seq_lens < 0");
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt,
                          num_queries, workspace, workspace_bytes, partition_tokens, stream, nullptr, nullptr,
                          pkv::DecodeMode::kPlanAndRun, false, sum_seq_lens);
}

pkv_status pkv_paged_attention_verify_fp8(void* out, const void* q, const void* key_cache, const void* value_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                          int num_seqs, int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                          float scale, pkv_dtype dt, const float* k_scale, const float* v_scale,
                                          int num_queries, void* workspace, size_t workspace_bytes,
                                          int partition_tokens, void* stream) {
    CallRange range_("pkv_paged_attention_verify_fp8");
    if (sum_seq_lens < 0) return fail(PKV_ERR_INVALID, "sum_seq_lens < 0");
    if (!k_scale || !v_scale) return fail(PKV_ERR_INVALID, "E4M3 pools need k_scale and v_scale");
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt,
                          num_queries, workspace, workspace_bytes, partition_tokens, stream, k_scale, v_scale,
                          pkv::DecodeMode::kPlanAndRun, false, sum_seq_lens);
}

pkv_status pkv_decode_plan(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                           int max_seq_len, int64_t sum_seq_lens, int num_heads, int num_kv_heads, int head_dim,
                           int block_size, pkv_dtype kv_dt, void* workspace, size_t workspace_bytes,
                           int partition_tokens, void* stream) {
    CallRange range_("pkv_decode_plan");
    if (!valid_dtype(kv_dt) && kv_dt != PKV_E4M3) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", static_cast<int>(kv_dt));
    if (sum_seq_lens < 0) return fail(PKV_ERR_INVALID, "sum_seq_lens < 0");
    return attention_call(nullptr, nullptr, nullptr, nullptr, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, 1, 1.0f,
                          kv_dt == PKV_E4M3 ? PKV_F16 : kv_dt, 1, workspace, workspace_bytes, partition_tokens,
                          stream, nullptr, nullptr, pkv::DecodeMode::kPlanOnly, kv_dt == PKV_E4M3, sum_seq_lens);
}

pkv_status pkv_paged_attention_decode_planned(void* out, const void* q, const void* key_cache,
                                              const void* value_cache, const int32_t* block_tables,
                                              int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                              int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                              float scale, pkv_dtype dt, void* workspace, size_t workspace_bytes,
                                              int partition_tokens, void* stream) {
    CallRange range_("pkv_paged_attention_decode_planned");
    if (sum_seq_lens < 0) return fail(PKV_ERR_INVALID, "sum_seq_lens < 0");
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt, 1,
                          workspace, workspace_bytes, partition_tokens, stream, nullptr, nullptr,
                          pkv::DecodeMode::kRunOnly, false, sum_seq_lens);
}

pkv_status pkv_paged_attention_decode_fp8_planned(void* out, const void* q, const void* key_cache,
                                                  const void* value_cache, const int32_t* block_tables,
                                                  int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                                  int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int64_t num_blocks, float scale, pkv_dtype dt,
                                                  const float* k_scale, const float* v_scale, void* workspace,
                                                  size_t workspace_bytes, int partition_tokens, void* stream) {
    CallRange range_("pkv_paged_attention_decode_fp8_planned");
    if (!k_scale || !v_scale) return fail(PKV_ERR_INVALID, "k_scale / v_scale are required");
    if (sum_seq_lens < 0) return fail(PKV_ERR_INVALID, "sum_seq_lens < 0");
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt, 1,
                          workspace, workspace_bytes, partition_tokens, stream, k_scale, v_scale,
                          pkv::DecodeMode::kRunOnly, false, sum_seq_lens);
}

pkv_status pkv_paged_attention_decode_fp8(void* out, const void* q, const void* key_cache, const void* value_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                          int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int64_t num_blocks, float scale, pkv_dtype dt,
                                          const float* k_scale, const float* v_scale, void* workspace,
                                          size_t workspace_bytes, int partition_tokens, void* stream) {
    CallRange range_("pkv_paged_attention_decode_fp8");
    if (!k_scale || !v_scale) return fail(PKV_ERR_INVALID, "k_scale / v_scale are required");
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt, 1,
                          workspace, workspace_bytes, partition_tokens, stream, k_scale, v_scale);
}

pkv_status pkv_paged_kv_append_decode(void* out, const void* q, const void* k, const void* v, void* key_cache,
                                      void* value_cache, const int64_t* slot_mapping, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                      int64_t sum_seq_lens, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale, pkv_dtype dt, pkv_dtype kv_dt,
                                      const float* k_scale, const float* v_scale, void* workspace,
                                      size_t workspace_bytes, int partition_tokens, int planned, void* stream) {
    CallRange range_("pkv_paged_kv_append_decode");
    if (sum_seq_lens < 0) return fail(PKV_ERR_INVALID, "sum_seq_lens < 0");
    if ((planned & ~(PKV_PLANNED | PKV_INPUTS_READY)) != 0 || planned == PKV_INPUTS_READY)
        return fail(PKV_ERR_INVALID, "planned %d: 0, PKV_PLANNED or PKV_PLANNED | PKV_INPUTS_READY", planned);
    if (kv_dt == PKV_E4M3) {
        if (!k_scale || !v_scale) return fail(PKV_ERR_INVALID, "E4M3 pools need k_scale and v_scale");
    } else if (kv_dt != dt) {
        return fail(PKV_ERR_INVALID, "kv_dt must be dt or PKV_E4M3");
    } else {
        k_scale = v_scale = nullptr;
    }
    const NewTokens nt{k, v, slot_mapping, (planned & PKV_INPUTS_READY) != 0};
    return attention_call(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dt, 1,
                          workspace, workspace_bytes, partition_tokens, stream, k_scale, v_scale,
                          (planned & PKV_PLANNED) ? pkv::DecodeMode::kRunOnly : pkv::DecodeMode::kPlanAndRun, false,
                          sum_seq_lens, &nt);
}

pkv_status pkv_paged_kv_append_fp8(const void* k, const void* v, void* key_cache, void* value_cache,
                                   const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks, int block_size,
                                   int num_kv_heads, int head_dim, pkv_dtype dt, const float* k_scale,
                                   const float* v_scale, void* stream) {
    CallRange range_("pkv_paged_kv_append_fp8");
    if (num_tokens < 0) return fail(PKV_ERR_INVALID, "num_tokens %lld < 0", static_cast<long long>(num_tokens));
    if (!valid_dtype(dt)) return fail(PKV_ERR_UNSUPPORTED, "dtype %d (fp16 or bf16 inputs)", static_cast<int>(dt));
    if (num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0)
        return fail(PKV_ERR_INVALID, "num_kv_heads %d / head_dim %d (head_dim must be a positive multiple of 8)",
                    num_kv_heads, head_dim);
    if (block_size <= 0 || num_blocks <= 0)
        return fail(PKV_ERR_INVALID, "block_size %d / num_blocks %lld", block_size, static_cast<long long>(num_blocks));
    if (num_tokens == 0) return ok();
    if (!k || !v || !key_cache || !value_cache || !slot_mapping || !k_scale || !v_scale)
        return fail(PKV_ERR_INVALID, "null pointer");
    if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(key_cache) & 7u) ||
        (reinterpret_cast<uintptr_t>(value_cache) & 7u) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return fail(PKV_ERR_INVALID, "k, v 16-byte aligned; caches and slot_mapping 8-byte; scales 4-byte");
    pkv::AppendFp8Args a;
    a.k = static_cast<const uint4*>(k);
    a.v = static_cast<const uint4*>(v);
    a.key_cache = static_cast<uint2*>(key_cache);
    a.value_cache = static_cast<uint2*>(value_cache);
    a.slots = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.num_tokens = num_tokens;
    a.num_slots = num_blocks * block_size;
    a.row_vecs = num_kv_heads * head_dim / 8;
    a.head_vecs = head_dim / 8;
    a.bf16 = dt == PKV_BF16;
    a.err = error_word(current_device());
    cudaError_t e = pkv::launch_append_fp8(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"

namespace {

// Shared by copy_blocks (one pool) and swap_blocks (two pools).
pkv_status block_copies(void* const* src_key, void* const* src_value, void* const* dst_key, void* const* dst_value,
                        int num_layers, const int64_t* src_dst_pairs, int64_t num_pairs, int64_t src_num_blocks,
                        int64_t dst_num_blocks, int block_size, int num_kv_heads, int head_dim, pkv_dtype dt,
                        void* stream, const char* what) {
    if (num_layers < 0 || num_pairs < 0) return fail(PKV_ERR_INVALID, "%s: num_layers / num_pairs < 0", what);
    if (!valid_dtype(dt) && dt != PKV_E4M3) return fail(PKV_ERR_UNSUPPORTED, "%s: dtype %d", what, static_cast<int>(dt));
    if (block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return fail(PKV_ERR_INVALID, "%s: bad pool shape", what);
    const int64_t block_bytes = static_cast<int64_t>(block_size) * num_kv_heads * head_dim * (dt == PKV_E4M3 ? 1 : 2);
    if (block_bytes % 16 != 0)
        return fail(PKV_ERR_INVALID, "%s: block bytes %lld not a multiple of 16", what,
                    static_cast<long long>(block_bytes));
    if (num_layers == 0 || num_pairs == 0) return ok();
    if (!src_key || !src_value || !dst_key || !dst_value || !src_dst_pairs)
        return fail(PKV_ERR_INVALID, "%s: null pointer", what);
    if (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) return fail(PKV_ERR_INVALID, "%s: pairs must be 8-byte aligned", what);
    for (int l = 0; l < num_layers; ++l) {
        const void* p[4] = {src_key[l], src_value[l], dst_key[l], dst_value[l]};
        for (const void* x : p)
            if (!x || !aligned16(x))
                return fail(PKV_ERR_INVALID, "%s: layer %d pool pointer null or not 16-byte aligned", what, l);
    }
    const int dev = current_device();
    for (int l0 = 0; l0 < num_layers; l0 += pkv::kMaxCopyLayers) {
        pkv::CopyArgs a;
        const int n = num_layers - l0 < pkv::kMaxCopyLayers ? num_layers - l0 : pkv::kMaxCopyLayers;
        for (int i = 0; i < pkv::kMaxCopyLayers; ++i) {
            a.src_key[i] = i < n ? static_cast<const uint4*>(src_key[l0 + i]) : nullptr;
            a.src_value[i] = i < n ? static_cast<const uint4*>(src_value[l0 + i]) : nullptr;
            a.dst_key[i] = i < n ? static_cast<uint4*>(dst_key[l0 + i]) : nullptr;
            a.dst_value[i] = i < n ? static_cast<uint4*>(dst_value[l0 + i]) : nullptr;
        }
        a.pairs = src_dst_pairs;
        a.num_pairs = num_pairs;
        a.src_num_blocks = src_num_blocks;
        a.dst_num_blocks = dst_num_blocks;
        a.num_layers = n;
        a.block_vecs = static_cast<int>(block_bytes / 16);
        a.err = error_word(dev);
        cudaError_t e = pkv::launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    }
    return ok();
}

}  // namespace

extern "C" {

pkv_status pkv_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                           const int64_t* src_dst_pairs, int64_t num_pairs, int64_t num_blocks, int block_size,
                           int num_kv_heads, int head_dim, pkv_dtype dt, void* stream) {
    CallRange range_("pkv_copy_blocks");
    return block_copies(key_caches, value_caches, key_caches, value_caches, num_layers, src_dst_pairs, num_pairs,
                        num_blocks, num_blocks, block_size, num_kv_heads, head_dim, dt, stream, "copy_blocks");
}

pkv_status pkv_swap_blocks(void* const* src_key_caches, void* const* src_value_caches, void* const* dst_key_caches,
                           void* const* dst_value_caches, int num_layers, const int64_t* src_dst_pairs,
                           int64_t num_pairs, int64_t src_num_blocks, int64_t dst_num_blocks, int block_size,
                           int num_kv_heads, int head_dim, pkv_dtype dt, void* stream) {
    CallRange range_("pkv_swap_blocks");
    return block_copies(src_key_caches, src_value_caches, dst_key_caches, dst_value_caches, num_layers, src_dst_pairs,
                        num_pairs, src_num_blocks, dst_num_blocks, block_size, num_kv_heads, head_dim, dt, stream,
                        "swap_blocks");
}

pkv_status pkv_device_error(unsigned int* value, int reset) {
    if (!value) return fail(PKV_ERR_INVALID, "null pointer");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "synchronize: %s", cudaGetErrorString(e));
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_pkv_error_word, sizeof(v));
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
    if (reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_pkv_error_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "reset error word: %s", cudaGetErrorString(e));
    }
    *value = v;
    return ok();
}

}  // extern "C"
