// Launchers shared between the C-ABI translation unit and the kernel units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

constexpr int kMaxCopyLayers = 64;   // layer pointers carried per copy_blocks launch

struct AppendArgs {
    const uint4* k;          // [T][row_vecs]
    const uint4* v;
    uint4* key_cache;        // [num_blocks * block_size][row_vecs]
    uint4* value_cache;
    const int64_t* slots;
    int64_t num_tokens;
    int64_t num_slots;       // num_blocks * block_size
    int row_vecs;            // num_kv_heads * head_dim * 2 / 16
    unsigned* err;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

// Append into an E4M3 pool: each element is quantized as
// e4m3(float32(x) / float32(scale[head])), round to nearest even, saturating.
struct AppendFp8Args {
    const uint4* k;          // [T][row_vecs] 8 fp16 / bf16 elements per vector
    const uint4* v;
    uint2* key_cache;        // [num_blocks * block_size][row_vecs] 8 codes per vector
    uint2* value_cache;
    const int64_t* slots;
    const float* k_scale;    // [num_kv_heads]
    const float* v_scale;
    int64_t num_tokens;
    int64_t num_slots;
    int row_vecs;            // num_kv_heads * head_dim / 8
    int head_vecs;           // head_dim / 8
    int bf16;                // input elements: 0 = fp16, 1 = bf16
    unsigned* err;
};
cudaError_t launch_append_fp8(const AppendFp8Args& a, cudaStream_t s);

// Block copies between two pools of the same block shape (the same pool for
// copy-on-write, a device pool and a pinned host pool for swapping).
struct CopyArgs {
    const uint4* src_key[kMaxCopyLayers];
    const uint4* src_value[kMaxCopyLayers];
    uint4* dst_key[kMaxCopyLayers];
    uint4* dst_value[kMaxCopyLayers];
    const int64_t* pairs;    // [num_pairs][2] (source block, destination block)
    int64_t num_pairs;
    int64_t src_num_blocks;
    int64_t dst_num_blocks;
    int num_layers;
    int block_vecs;          // block_size * num_kv_heads * head_dim * 2 / 16
    unsigned* err;
};
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t s);

struct DecodeArgs {
    void* out;                       // [B][nq][Hq][D]
    const void* q;                   // [B][nq][Hq][D]
    const int32_t* block_tables;     // [B][max_blocks_per_seq]
    const int32_t* seq_lens;         // [B]
    int4* plan;                      // [plan_capacity][2] work list, written per call by the plan kernel
                                     // (nullptr: direct grid): (first sequence, partition, stream length,
                                     // partition tokens), then (unit members, shared prefix length, lengths of
                                     // the unit's first two sequences)
    unsigned* tickets;               // [B][num_kv_heads * head_groups] finished partitions (zeroed per call)
    float* ws_o;                     // [B][Hq*nq][max_parts][D] unnormalised partial outputs
    float2* ws_ml;                   // [B][Hq*nq][max_parts] (running max in log2 units, sum)
    unsigned* err;
    int64_t num_blocks;
    int max_blocks_per_seq;
    int num_seqs;
    int max_seq_len;
    int num_heads;
    int num_kv_heads;
    int group;                       // query rows per KV head: (num_heads / num_kv_heads) * num_queries
    int qgroup;                      // query heads per KV head: num_heads / num_kv_heads
    int num_queries;                 // query tokens per sequence (1 = decode; > 1 = verify, causal)
    int head_groups;                 // ceil(group / 8): groups of query rows per KV head
    int block_size;
    int part_tokens;                 // tokens per partition (multiple of 64); with a plan, the smallest the
                                     // plan kernel may use
    int part_auto;                   // with a plan: 1 = the plan kernel picks the partition size (>= part_tokens)
    int slots;                       // SMs x resident decode CTAs per SM (for the plan kernel's choice)
    int rule_weight;                 // the automatic partition rule's weight (twentieths; plan_rule_tokens)
    int max_parts;                   // partials per query row: ceil(max_seq_len / part_tokens), plus one when
                                     // shared-prefix units are possible (the partials' stride)
    int direct_parts;                // ceil(max_seq_len / part_tokens): the direct grid's partition extent
    int plan_capacity;               // entries of `plan` the grid covers (<= num_seqs * max_parts)
    int64_t sum_seq_lens;            // the caller's sum of seq_lens (0: not given); the plan checks it
    int units;                       // 1: the plan may serve adjacent sequences that share leading blocks
                                     // (forks of one prompt) as one unit (16-bit decode, <= 4 query heads
                                     // per KV head: the members' heads fill one CTA's 8 columns)
    float scale_log2;                // scale * log2(e)
    int kv8;                         // 1: the pools hold E4M3 codes (head_dim 128), scaled per KV head
    const float* k_scale;            // [num_kv_heads] (E4M3 pools only)
    const float* v_scale;
    // Fused slot write (decode only; nullptr k_new: none).  Before attending,
    // the CTA whose partition holds position seq_len - 1 of sequence s writes
    // that sequence's new token (k_new / v_new row s, quantized for an E4M3
    // pool) into slot_mapping[s], which must be that position's slot.
    const uint4* k_new = nullptr;    // [B][num_kv_heads][D] in the query dtype
    const uint4* v_new = nullptr;
    const int64_t* slot_mapping = nullptr;   // [B]
    void* key_cache = nullptr;       // the pools written by the fused slot write
    void* value_cache = nullptr;
    // 1: nothing still running before this launch writes the pools, block tables,
    // lengths or plan (the caller's PKV_INPUTS_READY): a CTA reads its work item,
    // stages its table and starts its first tile loads before waiting for the
    // preceding kernel, then waits before it reads q, the new rows or the slots
    // (and never loads early the chunk that receives the new token)
    int early = 0;
};

// Sequences a call plans (sorts and compacts) at most; larger batches run the
// direct grid (one CTA per (KV head group, partition, sequence)).
constexpr int kPlanMaxSeqs = 1024;

// Shared-prefix units.  Adjacent sequences whose block tables agree on a
// leading run of blocks (forks of one prompt, copy-on-write after the fork)
// hold the same K/V there.  The plan serves up to 8 / (query heads per KV
// head) of them as one unit: the unit's stream is the shared prefix once,
// then each member's own blocks from the end of the prefix, block-aligned;
// a member's query heads attend to the prefix and to its own segment only.
// A unit shares at least this many positions (shorter runs stay separate).
constexpr int kUnitMinShare = 256;
// Work-list entries are two int4 each.
constexpr int kPlanEntryInts = 2;

// Block-table entries a decode CTA stages (a partition spans at most this many blocks).
constexpr int kPlanTableEntries = 512;
// Automatic partition sizes are multiples of this many positions.
constexpr int kPlanGranule = 512;

// The plan kernel's automatic partition size from the lengths' sum alone:
// about w / 20 of the positions per resident CTA slot (sum * nh / slots),
// rounded to the nearest multiple of kPlanGranule, at least one granule.  The
// weight w (twentieths) is the kernel's: kRuleDecode for the 16-bit decode
// kernel (0.85), kRuleDecode8 for E4M3 pools (an E4M3 position is half the
// bytes of a 16-bit one, with the same arithmetic and per-CTA costs; measured
// best on the 8B-shaped batch: 3072 positions against 4096 at twice), and
// kRuleVerifyTc for the tensor-core verify kernel, whose items carry a longer
// start-up and epilogue.  The host uses the same rule to bound the work list
// the grid must cover.
constexpr int kRuleDecode = 17;
constexpr int kRuleDecode8 = 24;
constexpr int kRuleVerifyTc = 22;
__host__ __device__ inline long long plan_rule_tokens(long long sum_lens, long long nh, int weight, long long slots) {
    const long long target = (sum_lens * nh * weight) / (slots * 20);
    const long long p = ((target + kPlanGranule / 2) / kPlanGranule) * kPlanGranule;
    return p > kPlanGranule ? p : kPlanGranule;
}

// Query rows (mma columns) one decode CTA serves.
constexpr int dec_heads_per_cta() { return 8; }

// Workspace layout of one decode call:
//   [tickets | work list | partial outputs | (max, sum) pairs]
// each region 256-byte aligned.  Every call re-initialises what it uses.
struct DecodeWorkspace {
    size_t ticket_bytes;   // tickets, padded
    size_t plan_bytes;     // work list (16 bytes per entry), padded
    size_t o_bytes;        // partial outputs, padded (0 when max_parts == 1)
    size_t ml_bytes;       // (max, sum) pairs (0 when max_parts == 1)
    size_t total() const { return ticket_bytes + plan_bytes + o_bytes + ml_bytes; }
};
DecodeWorkspace decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_parts);

// What one decode call launches: the plan kernel then the decode kernel; the
// plan alone; or the decode kernel alone over the plan already in the
// workspace (the merging CTA zeroes its ticket, so a plan serves any number
// of runs).
enum class DecodeMode { kPlanAndRun, kPlanOnly, kRunOnly };

// dtype: 0 = f16, 1 = bf16.  Runs one decode call on stream `s`: the plan
// kernel (work list + tickets) or, for a batch above kPlanMaxSeqs, a ticket
// memset; then the decode kernel, which merges split partitions in-kernel.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, cudaStream_t s, DecodeMode mode = DecodeMode::kPlanAndRun);
cudaError_t launch_decode_plan(const DecodeArgs& a, cudaStream_t s);

// More than kVerifyMinRows query rows per KV head (num_queries > 1, 16-bit pools):
// the verify kernel on the tensor cores; fewer, and E4M3 pools: the decode
// kernel's multi-query form, 8 rows per CTA.
constexpr int kVerifyMinRows = 16;

// The verify kernel on the fifth-generation tensor cores (tcgen05): up to
// kVerifyTcRows query rows per CTA (head_groups = ceil(rows / kVerifyTcRows));
// a KV head with at most 64 rows runs the M = 64 form.
constexpr int kVerifyTcRows = 128;
int verify_tc_rows_per_cta(int rows);
cudaError_t launch_verify_tc(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                             int head_dim, cudaStream_t s, DecodeMode mode = DecodeMode::kPlanAndRun);
int verify_tc_ctas_per_sm(int head_dim);

// CTAs of the decode kernel resident per SM on the current device (current
// configuration; kv8: the E4M3-pool kernel), or 0 if it cannot be queried.
int decode_ctas_per_sm(int head_dim, bool kv8 = false);

// Record `msg` as the calling thread's pkv_last_error() message and return `st`.
int set_error_message(int st, const char* msg);

}  // namespace pkv
