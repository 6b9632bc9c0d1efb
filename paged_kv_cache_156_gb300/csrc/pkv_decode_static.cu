// pkv_paged_attention_decode_static: the decode call for callers that cannot
// allocate device memory (a plugin given only its input and output buffers,
// a serving loop that must not allocate after start-up).  Its split-K scratch
// is the file-scope device array below instead of a caller-provided
// workspace; everything else is pkv_paged_attention_decode, called as is.
#include <stdio.h>

#include <mutex>

#include "../../include/pkv.h"
#include "pkv_internal.h"

// The scratch: PKV_STATIC_DECODE_SCRATCH_BYTES on every device that loads the
// library, alive until the process exits, shared by every call.
static __device__ __align__(256) unsigned char g_static_decode_scratch[PKV_STATIC_DECODE_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch on the current device.  Host code must not
// pass the array's name to a kernel (on the host it is only a stand-in), so
// the address is looked up once per device, with that device current, and
// cached.  Returns a message on failure, nullptr on success.
const char* scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return "no current CUDA device";
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_decode_scratch);
        if (e != cudaSuccess || !p) return "cudaGetSymbolAddress of the static decode scratch failed";
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return nullptr;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_static(
    void* out, const void* q, const void* key_cache, const void* value_cache, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int max_seq_len, int num_heads,
    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale, pkv_dtype dt,
    int partition_tokens, void* stream) {
    const size_t need =
        pkv_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, partition_tokens);
    if (need != (size_t)-1 && need > PKV_STATIC_DECODE_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "batch needs %zu bytes of decode scratch; the built-in scratch holds %zu "
                 "(use pkv_paged_attention_decode with a workspace, or a larger partition_tokens)",
                 need, (size_t)PKV_STATIC_DECODE_SCRATCH_BYTES);
        return static_cast<pkv_status>(pkv::set_error_message(PKV_ERR_WORKSPACE, msg));
    }
    void* scratch = nullptr;
    if (need != (size_t)-1 && num_seqs > 0) {
        if (const char* why = scratch_for_current_device(&scratch))
            return static_cast<pkv_status>(pkv::set_error_message(PKV_ERR_CUDA, why));
    }
    // Invalid shapes fall through to the full validation of the regular call.
    return pkv_paged_attention_decode(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                                      num_seqs, max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                                      num_blocks, scale, dt, scratch, scratch ? PKV_STATIC_DECODE_SCRATCH_BYTES : 0,
                                      partition_tokens, stream);
}
