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
    void* out;                       // [B][Hq][D]
    const void* q;                   // [B][Hq][D]
    const int32_t* block_tables;     // [B][max_blocks_per_seq]
    const int32_t* seq_lens;         // [B]
    unsigned* work_counter;          // next work unit of the persistent variant (zeroed per call)
    unsigned* n_items;               // items in `items` (written per call by the plan kernel)
    unsigned* tickets;               // [B][num_kv_heads * head_groups] finished partitions (zeroed per call)
    unsigned* items;                 // [B * max_parts] (sequence << 9 | partition), largest first
    float* ws_o;                     // [B][Hq][max_parts][D] unnormalised partial outputs
    float2* ws_ml;                   // [B][Hq][max_parts] (running max in log2 units, sum)
    unsigned* err;
    int64_t num_blocks;
    int max_blocks_per_seq;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int group;                       // query rows per KV head: (num_heads / num_kv_heads) * num_queries
    int qgroup;                      // query heads per KV head: num_heads / num_kv_heads
    int num_queries;                 // query tokens per sequence (1 = decode; > 1 = verify, causal)
    int head_groups;                 // ceil(group / 8): groups of query rows per KV head
    int block_size;
    int part_tokens;                 // tokens per partition (multiple of 64)
    int max_parts;                   // ceil(max_seq_len / part_tokens)
    float scale_log2;                // scale * log2(e)
};

// Workspace layout of one decode call:
//   [work counter, item count, tickets | item list | partial outputs | (max, sum) pairs]
// each region 256-byte aligned.  Every call re-initialises what it uses.
struct DecodeWorkspace {
    size_t ticket_bytes;   // work counter + item count + tickets, padded
    size_t item_bytes;     // item list, padded
    size_t o_bytes;        // partial outputs, padded (0 when max_parts == 1)
    size_t ml_bytes;       // (max, sum) pairs (0 when max_parts == 1)
    size_t total() const { return ticket_bytes + item_bytes + o_bytes + ml_bytes; }
};
DecodeWorkspace decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_parts);

// dtype: 0 = f16, 1 = bf16.  Runs one decode call on stream `s`: either the
// grid variant (one CTA per work item; a memset zeroes the tickets) or the
// persistent variant (a plan kernel builds the item list, then CTAs resident
// on every SM pull items).  Both merge split partitions in-kernel.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, cudaStream_t s);
cudaError_t launch_decode_grid(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                               int head_dim, cudaStream_t s);
cudaError_t launch_decode_persistent(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                                     int head_dim, cudaStream_t s);

// CTAs of the decode kernel resident per SM on the current device (grid
// variant, current configuration), or 0 if it cannot be queried.
int decode_ctas_per_sm(int head_dim);

// Record `msg` as the calling thread's pkv_last_error() message and return `st`.
int set_error_message(int st, const char* msg);

}  // namespace pkv
