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

struct CopyArgs {
    uint4* key[kMaxCopyLayers];
    uint4* value[kMaxCopyLayers];
    const int64_t* pairs;    // [num_pairs][2]
    int64_t num_pairs;
    int64_t num_blocks;
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
    unsigned* work_counter;          // next work item (zeroed before each launch)
    unsigned* tickets;               // [B][num_kv_heads * head_groups] finished partitions (zeroed)
    float* ws_o;                     // [B][Hq][max_parts][D] unnormalised partial outputs
    float2* ws_ml;                   // [B][Hq][max_parts] (running max in log2 units, sum)
    unsigned* err;
    int64_t num_blocks;
    int max_blocks_per_seq;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int group;                       // num_heads / num_kv_heads
    int head_groups;                 // ceil(group / 8): query-head groups per KV head
    int block_size;
    int part_tokens;                 // tokens per partition (multiple of 64)
    int max_parts;                   // ceil(max_seq_len / part_tokens)
    float scale_log2;                // scale * log2(e)
};

// Workspace layout of one decode call: [counter + tickets | partial outputs | (max, sum) pairs],
// each region 256-byte aligned.  Only the first region needs zeroing per call.
struct DecodeWorkspace {
    size_t ticket_bytes;   // counter + tickets, padded
    size_t o_bytes;        // partial outputs, padded (0 when max_parts == 1)
    size_t ml_bytes;       // (max, sum) pairs (0 when max_parts == 1)
    size_t total() const { return ticket_bytes + o_bytes + ml_bytes; }
};
DecodeWorkspace decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_parts);

// dtype: 0 = f16, 1 = bf16.  Zeroes the counters (one memset) and launches
// the persistent decode kernel, which also merges split partitions.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int dtype,
                          int head_dim, size_t zero_bytes, cudaStream_t s);

// Record `msg` as the calling thread's pkv_last_error() message and return `st`.
int set_error_message(int st, const char* msg);

}  // namespace pkv
