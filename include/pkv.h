/*
 * pkv.h -- C ABI of the paged KV-cache decode library (sm_103a, one GPU).
 *
 * The library implements the decode-step hot path of PagedAttention as the
 * following pages describe it (cited by title and section):
 *
 *   P1 "vLLM核心概念：PagedAttention原理、KV Cache分页管理、连续批处理、投机解码概览"
 *   P2 "LLM 推理引擎内部原理：PagedAttention、Continuous Batching 与现代推理架构剖析"
 *   P3 "LLM 推理优化深度实战：从 PagedAttention 到 Speculative Decoding 的工程架构"
 *   P4 the tbr8.org PagedAttention article (title not in the extract)
 *
 * Memory layout shared by every call (P4 §2.2, the kernel signature's cache
 * shape): one K pool and one V pool per layer, each a contiguous array
 *
 *     cache[num_blocks][block_size][num_kv_heads][head_dim]      (fp16 or bf16)
 *
 * Token position t of sequence s lives in physical block
 * block_tables[s][t / block_size] at offset t % block_size (P4 §2.1).  Its
 * flat slot is physical_block * block_size + offset (P2 §2.3, append_slot).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates and frees nothing and keeps no per-call state.  Tensors are
 *     dense, row-major, in the shapes stated, and 16-byte aligned.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  A return of PKV_OK means the launch was
 *     accepted, not that the kernels finished.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and returns PKV_ERR_INVALID /
 *     PKV_ERR_UNSUPPORTED / PKV_ERR_WORKSPACE.  A failed launch returns
 *     PKV_ERR_CUDA.  pkv_last_error() then holds a message (thread-local).
 *   - Device-side bounds: a block id outside [0, num_blocks) or a slot
 *     outside [0, num_blocks * block_size) is never dereferenced; the kernel
 *     skips that access and raises the device error word (pkv_device_error).
 *     Such inputs give unspecified output values but never a fault.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,      /* bad pointer, size, shape or alignment               */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, block_size, dtype    */
    PKV_ERR_WORKSPACE = 3,    /* decode workspace missing or too small               */
    PKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed                */
    PKV_ERR_OOM = 5           /* block manager: not enough free blocks (nothing changed) */
} pkv_status;

/* Element types.  PKV_E4M3 (8-bit OCP FP8 E4M3 codes) is a pool type only:
 * accepted by pkv_copy_blocks / pkv_swap_blocks and as the pool of the
 * *_fp8 calls, never for q, out or new K/V. */
typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_E4M3 = 2 } pkv_dtype;

/* Library ABI version (major * 100 + minor). */
PKV_API int pkv_version(void);

/* Message for the last non-OK status returned on this thread ("" if none). */
PKV_API const char* pkv_last_error(void);

/*
 * paged_kv_append -- write each new token's K and V into its slot.
 *
 * P2 §2.3 (BlockEngine.append_slot gives the slot of the token a sequence
 * generates next) and P1 §4.2.2 ("增长": each new token goes into the current
 * block, a new block when it is full).  For every t < num_tokens with
 * slot_mapping[t] >= 0:
 *     key_cache  [slot / block_size][slot % block_size][:][:] = k[t][:][:]
 *     value_cache[slot / block_size][slot % block_size][:][:] = v[t][:][:]
 * bit for bit.  A negative slot is a padding entry and writes nothing.
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim], dtype `dt`
 *   key_cache,
 *   value_cache   [num_blocks][block_size][num_kv_heads][head_dim], updated in place
 *   slot_mapping  int64 [num_tokens]
 * Slots must be distinct (two tokens writing one slot race).  num_tokens == 0
 * is a no-op.  head_dim must be a multiple of 8.
 */
PKV_API pkv_status pkv_paged_kv_append(const void* k, const void* v, void* key_cache, void* value_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                               int block_size, int num_kv_heads, int head_dim, pkv_dtype dt,
                               void* stream);

/*
 * Workspace for pkv_paged_attention_decode: bytes needed for its
 * per-(sequence, head group) merge tickets, its work list and the split-K
 * partials (never 0).  partition_tokens: 0 sizes it for the smallest
 * partition the decode call may use for the same arguments on the current
 * device; otherwise for the caller's partition size.  Returns (size_t)-1 for
 * invalid arguments.
 */
PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int max_seq_len, int partition_tokens);

/*
 * Smallest partition size (tokens) pkv_paged_attention_decode uses when
 * passed 0 (its device-side plan may take a larger one from the actual
 * lengths, see below), or -1 on bad arguments.
 */
PKV_API int pkv_decode_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int max_seq_len);

/* Batches of up to this many sequences run through the plan kernel (below). */
#define PKV_PLAN_MAX_SEQS 1024

/*
 * Partition size (tokens) the last pkv_paged_attention_decode call with this
 * workspace and batch shape used, read back from its work list (synchronises
 * `stream`); -1 for a batch above PKV_PLAN_MAX_SEQS (no work list), bad
 * arguments or a failed read.  For pkv_paged_attention_verify pass
 * num_heads * num_queries.
 */
PKV_API int pkv_decode_plan_partition_tokens(const void* workspace, int num_seqs, int num_heads, int num_kv_heads,
                                     void* stream);

/*
 * paged_attention_decode -- one query token per sequence attends over its
 * paged K/V (GQA).
 *
 * P4 §2.2 (paged_attention_kernel: walk the logical blocks, look up each
 * physical block in the block table, read its K/V rows, stop at seq_len,
 * score = q.k / sqrt(head_dim), weight V by the softmax of the scores) and
 * P2 §2.4 (indirect addressing through the block table; softmax and V
 * weighting follow the scores).  For sequence s and query head h, with
 * g = h / (num_heads / num_kv_heads) and positions t < seq_lens[s]:
 *     z_t = scale * <q[s][h], K_t>,   out[s][h] = sum_t softmax(z)_t * V_t
 * where K_t, V_t are KV head g's rows at position t.  seq_lens[s] == 0 gives
 * zeros.  Accumulation is fp32; `out` is rounded to nearest even.
 *
 *   out           [num_seqs][num_heads][head_dim], dtype `dt`
 *   q             [num_seqs][num_heads][head_dim], dtype `dt`
 *   key_cache,
 *   value_cache   [num_blocks][block_size][num_kv_heads][head_dim]
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]; only the first
 *                 ceil(seq_lens[s] / block_size) entries of row s are read
 *   seq_lens      int32 [num_seqs], each in [0, max_seq_len] (a length above
 *                 it is treated as max_seq_len and raises the device error
 *                 word)
 *   max_seq_len   host-known upper bound of seq_lens (sizes the launch; it
 *                 must not exceed max_blocks_per_seq * block_size)
 *   workspace     device scratch of at least pkv_decode_workspace_bytes(...)
 *                 bytes, 16-byte aligned; its contents on entry are ignored
 *                 (the call zeroes the counters it needs on `stream`).  Calls
 *                 that share a workspace must be ordered on one stream.
 *   partition_tokens  0 = automatic; else a multiple of 64 in [64, 4096].
 *                 Sequences longer than one partition are split into
 *                 partitions whose partial softmax states are merged in the
 *                 same launch by the last partition to finish (split-K over
 *                 the sequence).  For up to 1024 sequences a plan kernel
 *                 first lists the (sequence, partition) items that exist,
 *                 longest sequences first, and with 0 picks the partition
 *                 size from the lengths themselves (about 0.85 x the
 *                 positions per resident CTA, an E4M3 position counting
 *                 1.4 times, multiples of 512, at least
 *                 pkv_decode_partition_tokens); the output does not depend
 *                 on that order.  A sequence may span at most 512
 *                 partitions at the host's size: a longer max_seq_len with
 *                 a small explicit size returns PKV_ERR_UNSUPPORTED (raise
 *                 partition_tokens); 0 always picks a size that fits.
 *   Shared prefixes: the plan compares the block-table rows of adjacent
 *   sequences whose first entries agree (forks of one prompt, P2 §3.3) and,
 *   with at most 4 query heads per KV head and 16-bit pools, serves up to
 *   8 / (num_heads / num_kv_heads) sequences that share at least 256 leading
 *   positions in one CTA per KV head: the shared blocks are streamed once for
 *   all of them, then each sequence's own blocks, each sequence's heads
 *   seeing the shared positions and its own.  The result is that of the
 *   sequences attended one by one, up to the summation order.
 * head_dim in {64, 128}; block_size in {8, 16, 32}; num_heads a multiple of
 * num_kv_heads.
 */
PKV_API pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                      int max_seq_len, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale, pkv_dtype dt,
                                      void* workspace, size_t workspace_bytes, int partition_tokens,
                                      void* stream);

/*
 * Plan once, run per layer.  Every layer of a decode step attends over the
 * same batch (the same lengths and block tables), so the work list the plan
 * kernel builds (above) is the same for all of them.  pkv_decode_plan writes
 * it into `workspace` (and zeroes the merge tickets) on `stream`;
 * pkv_paged_attention_decode_planned and pkv_paged_attention_decode_fp8_planned
 * then run the decode alone, each exactly as pkv_paged_attention_decode /
 * _fp8 would, leaving the tickets zeroed again for the next run.
 *
 * sum_seq_lens: the sum of seq_lens when the caller knows it (a scheduler
 * does), else 0.  It only sizes the decode grid: the work list then needs at
 * most num_seqs + sum_seq_lens / P entries (P the smallest partition size the
 * plan can pick, which with the automatic size the host derives from the
 * same sum) instead of num_seqs * ceil(max_seq_len / P), and a mixed-length
 * batch launches far fewer CTAs that find no work.  The plan kernel checks it
 * against the real sum; a wrong value raises the error word's bounds bit
 * (entries past the grid are then dropped and their outputs are undefined,
 * never out of range).
 *
 * Preconditions (not checked on the host): the runs pass the same
 * block_tables contents, seq_lens contents, num_seqs, max_seq_len,
 * sum_seq_lens, num_heads, num_kv_heads, head_dim, block_size and
 * partition_tokens as the plan; kv_dt
 * is the pools' element type (PKV_E4M3 for the _fp8 runs); calls are ordered
 * on one stream; the plan is made again after any call that raised the
 * device error word.  A run whose work list does not fit its arguments skips
 * the offending entries and raises the error word's bounds bit; it never
 * reads or writes outside its buffers.  A batch above PKV_PLAN_MAX_SEQS has
 * no work list: pkv_decode_plan does nothing and each run launches its full
 * grid.
 */
PKV_API pkv_status pkv_decode_plan(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                           int num_seqs, int max_seq_len, int64_t sum_seq_lens, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, pkv_dtype kv_dt, void* workspace,
                           size_t workspace_bytes, int partition_tokens, void* stream);

PKV_API pkv_status pkv_paged_attention_decode_planned(void* out, const void* q, const void* key_cache,
                                              const void* value_cache, const int32_t* block_tables,
                                              int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                              int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int64_t num_blocks, float scale, pkv_dtype dt, void* workspace,
                                              size_t workspace_bytes, int partition_tokens, void* stream);

PKV_API pkv_status pkv_paged_attention_decode_fp8_planned(void* out, const void* q, const void* key_cache,
                                                  const void* value_cache, const int32_t* block_tables,
                                                  int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                                  int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int64_t num_blocks, float scale, pkv_dtype dt,
                                                  const float* k_scale, const float* v_scale, void* workspace,
                                                  size_t workspace_bytes, int partition_tokens, void* stream);

/*
 * paged_kv_append + paged_attention_decode in one launch.
 *
 * P2 §2.3 and P1 §4.2.2 (each step's new token goes into the slot the block
 * manager gave it, and the step then attends over the sequence including that
 * token).  Same results as pkv_paged_kv_append (pkv_paged_kv_append_fp8 for
 * kv_dt == PKV_E4M3) of token s = 0 .. num_seqs - 1 followed by
 * pkv_paged_attention_decode (_fp8; _planned when `planned` is non-zero, over
 * the plan pkv_decode_plan wrote), bit for bit in the caches, without the
 * separate slot-write launch: the decode CTA that reads position
 * seq_lens[s] - 1 writes the token there itself before its tile loads.
 *
 *   k, v          [num_seqs][num_kv_heads][head_dim] in dtype `dt` (q's)
 *   slot_mapping  int64 [num_seqs]: the slot of position seq_lens[s] - 1 of
 *                 sequence s (block_tables[s][(seq_lens[s]-1) / block_size] *
 *                 block_size + (seq_lens[s]-1) % block_size), or negative for
 *                 a sequence with no new token (nothing is written)
 *   kv_dt         dt for 16-bit pools, PKV_E4M3 for 8-bit pools (then
 *                 k_scale / v_scale as in pkv_paged_kv_append_fp8; else
 *                 ignored)
 *   planned       0: plan and run; PKV_PLANNED: run over the plan
 *                 pkv_decode_plan wrote; PKV_PLANNED | PKV_INPUTS_READY: that,
 *                 and the caller guarantees that no work still pending on
 *                 `stream` when this call is made writes the pools, the block
 *                 tables, seq_lens or the workspace's plan (within a decode
 *                 step: every layer after the first, whose pool only its own
 *                 call writes).  Each CTA then reads its work item, stages its
 *                 block-table slice and starts its first tile loads while the
 *                 preceding kernel finishes (programmatic dependent launch),
 *                 and waits for that kernel before it reads q, k, v or
 *                 slot_mapping; the chunk that receives the new token is never
 *                 loaded before its slot is written.  Results are the same bit
 *                 for bit.  Not for the call right after pkv_decode_plan (it
 *                 writes the plan) nor after pkv_copy_blocks / swap / append
 *                 into the same pools.  16-bit pools only (ignored for E4M3).
 *                 Any other value is PKV_ERR_INVALID.
 *   other arguments as pkv_paged_attention_decode / _planned.
 * A non-negative slot that is not that position's slot (or a sequence of
 * length 0 with one) is not written and raises the error word's bounds bit.
 * The block holding position seq_lens[s] - 1 must not be read by another
 * sequence of the call (the block manager's copy-on-write gives every
 * sequence its own last block before it appends).
 */
#define PKV_PLANNED 1
#define PKV_INPUTS_READY 2
PKV_API pkv_status pkv_paged_kv_append_decode(void* out, const void* q, const void* k, const void* v,
                                      void* key_cache, void* value_cache, const int64_t* slot_mapping,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                      int64_t sum_seq_lens, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale, pkv_dtype dt,
                                      pkv_dtype kv_dt, const float* k_scale, const float* v_scale,
                                      void* workspace, size_t workspace_bytes, int partition_tokens,
                                      int planned, void* stream);

/*
 * paged_attention_verify -- num_queries query tokens per sequence over its
 * paged K/V, causal among themselves (the verification step of speculative
 * decoding).
 *
 * P1 §4.4.2 (the target model takes the K draft tokens as input and computes
 * their distributions in one forward pass); P3 §4.2 (speculative_verify:
 * the large model scores all gamma candidates in one pass over the prefix KV);
 * P2 §5.2 (the candidates' KV lives in the same block structure).  The last
 * num_queries positions of sequence s hold the query tokens' own K/V (written
 * by pkv_paged_kv_append first); query token i (0-based) attends over
 * positions t < seq_lens[s] - num_queries + i + 1, otherwise exactly as
 * pkv_paged_attention_decode.  num_queries = 1 is the decode call.
 *
 *   out, q        [num_seqs][num_queries][num_heads][head_dim]
 *   workspace     pkv_decode_workspace_bytes(num_seqs, num_heads * num_queries,
 *                 num_kv_heads, head_dim, max_seq_len, partition_tokens) bytes
 *   num_queries   in [1, 64]; seq_lens[s] should be 0 or >= num_queries (a
 *                 query token that sees no position gets a zero output)
 *   sum_seq_lens  the sum of seq_lens if known, else 0; it only sizes the
 *                 grid, as for pkv_paged_attention_decode_planned
 * A KV head serves R = (num_heads / num_kv_heads) * num_queries query rows.
 * R > 16: the tensor-core verify kernel (tcgen05), 64 rows per CTA when
 * R <= 64, else 128 (head_groups = ceil(R / 128)), K/V streamed once per
 * row group; R <= 16: the decode kernel's multi-query form, 8 rows per CTA.
 */
PKV_API pkv_status pkv_paged_attention_verify(void* out, const void* q, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                      int max_seq_len, int64_t sum_seq_lens, int num_heads, int num_kv_heads,
                                      int head_dim, int block_size, int64_t num_blocks, float scale,
                                      pkv_dtype dt, int num_queries, void* workspace, size_t workspace_bytes,
                                      int partition_tokens, void* stream);

/*
 * 8-bit KV cache (E4M3) -- P3 §6.2 (KV cache quantization: attention reads
 * low-precision K/V, saving memory and bandwidth with little accuracy loss).
 * The page names no format; these calls use OCP FP8 E4M3 codes (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, largest finite 448, no
 * infinities) with one float32 scale per KV head for K and one for V: the
 * element a code stands for is e4m3_value(code) * scale[kv_head].
 *
 * pkv_paged_kv_append_fp8: as pkv_paged_kv_append into uint8 pools; element
 * (t, h, i) becomes e4m3(float32(k[t][h][i]) / k_scale[h]) (IEEE division,
 * round to nearest even, magnitudes above 448 saturate to 448, NaN stays
 * NaN); likewise V with v_scale.
 *   k, v              [T][num_kv_heads][head_dim] fp16 / bf16 (`dt`), 16-byte aligned
 *   key_cache,
 *   value_cache       uint8 [num_blocks][block_size][num_kv_heads][head_dim], 8-byte aligned
 *   k_scale, v_scale  device float32 [num_kv_heads], each > 0 (not checked)
 */
PKV_API pkv_status pkv_paged_kv_append_fp8(const void* k, const void* v, void* key_cache, void* value_cache,
                                   const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                                   int block_size, int num_kv_heads, int head_dim, pkv_dtype dt,
                                   const float* k_scale, const float* v_scale, void* stream);

/*
 * pkv_paged_attention_decode_fp8: pkv_paged_attention_decode over uint8 E4M3
 * pools, K_t = e4m3_value(code) * k_scale[g] and V_t = e4m3_value(code) *
 * v_scale[g] for KV head g; q and out are fp16 / bf16 (`dt`).  Same
 * workspace, partitioning and plan.  head_dim 128 only.  The tensor cores
 * run in f16: every E4M3 value is exact in f16, and q is converted to f16
 * (exact for |q| < 65504; a bf16 query beyond f16's range is not supported).
 */
PKV_API pkv_status pkv_paged_attention_decode_fp8(void* out, const void* q, const void* key_cache,
                                          const void* value_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                          int max_seq_len, int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int64_t num_blocks, float scale, pkv_dtype dt,
                                          const float* k_scale, const float* v_scale, void* workspace,
                                          size_t workspace_bytes, int partition_tokens, void* stream);

/*
 * pkv_paged_attention_verify_fp8: pkv_paged_attention_verify over uint8 E4M3
 * pools (P1 §4.4.2 and P3 §4.2: the draft tokens scored in one pass; P3 §6.2:
 * over the low-precision K/V), with K and V as in
 * pkv_paged_attention_decode_fp8 and the causal mask of
 * pkv_paged_attention_verify.  q, out [num_seqs][num_queries][num_heads][128]
 * in dt (PKV_F16 or PKV_BF16).  Query rows are served 8 per CTA (the decode
 * kernel's multi-query form), so the CTAs of a KV head with many rows read
 * the same tiles; they run side by side (row groups are adjacent in the
 * grid), so L2 serves all but the first read, but each does the full
 * per-position work: R rows cost R / 8 CTAs' worth of arithmetic.
 */
PKV_API pkv_status pkv_paged_attention_verify_fp8(void* out, const void* q, const void* key_cache,
                                          const void* value_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                          int max_seq_len, int64_t sum_seq_lens, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                          float scale, pkv_dtype dt, const float* k_scale,
                                          const float* v_scale, int num_queries, void* workspace,
                                          size_t workspace_bytes, int partition_tokens, void* stream);

/*
 * copy_blocks -- the copy-on-write block copy at a fork.
 *
 * P2 §3.1 (the scheduler output's blocks_to_copy, "用于 Copy-on-Write") and
 * §3.3; P1 §4.2.2 (a writer to a shared block copies it, then writes); P4 §五.
 * For every pair i and every layer l:
 *     key_caches[l][dst_i] = key_caches[l][src_i];  value_caches[l][dst_i] = value_caches[l][src_i]
 * bit for bit, where (src_i, dst_i) = src_dst_pairs[i].
 *
 *   key_caches, value_caches  HOST arrays of num_layers device pointers, each a
 *                             pool [num_blocks][block_size][num_kv_heads][head_dim]
 *   src_dst_pairs             DEVICE int64 [num_pairs][2]
 *   dt                        the pools' element type (PKV_F16, PKV_BF16 or PKV_E4M3)
 * Destinations must be distinct and must not appear as a source (the pairs
 * are applied concurrently).  num_pairs == 0 or num_layers == 0 is a no-op.
 */
PKV_API pkv_status pkv_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                           const int64_t* src_dst_pairs, int64_t num_pairs, int64_t num_blocks,
                           int block_size, int num_kv_heads, int head_dim, pkv_dtype dt, void* stream);

/*
 * swap_blocks -- move blocks between the device pool and a host pool
 * (preemption by swapping).
 *
 * P2 §3.1 (the scheduler output's blocks_to_swap_in / blocks_to_swap_out) and
 * §3.2 (Swapping: a preempted request's blocks are copied from GPU memory to
 * CPU memory, freeing the GPU blocks, and copied back when it resumes); P1
 * §4.2.4 (--swap-space).  For every pair i and every layer l:
 *     dst_key_caches[l][dst_i] = src_key_caches[l][src_i], and the same for V,
 * bit for bit, where (src_i, dst_i) = src_dst_pairs[i].
 *
 *   src_*_caches, dst_*_caches  HOST arrays of num_layers pointers, each a pool
 *                 [num_blocks][block_size][num_kv_heads][head_dim] that the GPU
 *                 can address: device memory, or pinned host memory (cudaHostAlloc,
 *                 or torch pin_memory; pinned memory is mapped under unified
 *                 addressing).  Swap-out: device -> host; swap-in: host -> device.
 *   src_dst_pairs DEVICE int64 [num_pairs][2]; a source block id in
 *                 [0, src_num_blocks), a destination id in [0, dst_num_blocks)
 * Destinations must be distinct.  num_pairs == 0 or num_layers == 0 is a no-op.
 */
PKV_API pkv_status pkv_swap_blocks(void* const* src_key_caches, void* const* src_value_caches,
                           void* const* dst_key_caches, void* const* dst_value_caches, int num_layers,
                           const int64_t* src_dst_pairs, int64_t num_pairs, int64_t src_num_blocks,
                           int64_t dst_num_blocks, int block_size, int num_kv_heads, int head_dim,
                           pkv_dtype dt, void* stream);

/*
 * Device error word: bit 0 = a block id or slot out of range was skipped,
 * bit 1 = a pipeline wait gave up after its time limit.  Reads the word of
 * the current device after synchronising it, stores it in *value and, if
 * `reset` is non-zero, clears it.  Debug/test use; not for the hot path.
 */
PKV_API pkv_status pkv_device_error(unsigned int* value, int reset);

/*
 * paged_attention_decode_static -- pkv_paged_attention_decode for callers that
 * cannot allocate device memory.
 *
 * The source pages have no counterpart: this entry point exists for how the
 * library is called, not for what it computes.  Some callers have no way to
 * call cudaMalloc: a plugin inside a host engine that owns the device's whole
 * memory budget and hands the plugin only its input and output buffers, or a
 * serving loop that reserves all device memory at start-up and must not
 * allocate afterwards.  They cannot provide the decode workspace, so this call
 * uses a scratch array built into the library instead.  It computes exactly
 * what pkv_paged_attention_decode computes (same arguments, minus workspace),
 * through the same kernels.
 *
 *   - The scratch is a file-scope device array of PKV_STATIC_DECODE_SCRATCH_BYTES
 *     bytes.  Every GPU that loads the library holds it until the process exits.
 *   - A batch whose workspace (pkv_decode_workspace_bytes for the same
 *     arguments) exceeds that size is rejected with PKV_ERR_WORKSPACE and a
 *     message giving both sizes; nothing is launched.
 *   - The call allocates and frees nothing.  The first call on a device looks
 *     up the array's device address (cudaGetSymbolAddress) with that device
 *     current and caches it; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     the counters a call needs zeroed are cleared on `stream` by the call
 *     itself.  Calls whose kernels overlap on the GPU (other streams, other
 *     host threads) race on the array: order them on one stream.
 *   - The cached address belongs to the device's context at the first call.
 *     After cudaDeviceReset (or any reset of the primary context) it is
 *     stale: do not call this entry point again in that process.
 */
#define PKV_STATIC_DECODE_SCRATCH_BYTES ((size_t)32 << 20)

PKV_API pkv_status pkv_paged_attention_decode_static(void* out, const void* q, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                      int max_seq_len, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, float scale, pkv_dtype dt,
                                      int partition_tokens, void* stream);

/*
 * Host block manager (host memory only; no GPU call).
 *
 * P2 §2.3 (BlockEngine: free blocks in a FIFO list; allocate takes
 * ceil(num_tokens / block_size) blocks from its front; append_slot gives the
 * slot of a sequence's next token, taking a new block when the last one is
 * full, or reports exhaustion so the scheduler can preempt; free returns the
 * blocks to the back of the list) and §3.3 (forked samples share prefix
 * blocks); P1 §4.2.2 (a writer to a shared block copies it first); P4 §五
 * (shared blocks are reference counted and not freed while shared).
 *
 * One manager per pool; not thread-safe.  Every call checks before it changes
 * anything: PKV_ERR_OOM and PKV_ERR_INVALID leave the manager as it was.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of blocks 0..num_blocks-1; `free_order` (host, optional) is the
 * initial order of the free list (a permutation of the pool), NULL = 0, 1, ...
 * Returns NULL on bad arguments or allocation failure. */
PKV_API pkv_block_manager* pkv_bm_create(int64_t num_blocks, int block_size, const int64_t* free_order);
PKV_API void pkv_bm_destroy(pkv_block_manager* bm);
PKV_API int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm);
/* Tokens held by a sequence, or -1 if the id is unknown. */
PKV_API int64_t pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq_id);
/* Sequences sharing a block (0 = free), or -1 for an id outside the pool. */
PKV_API int pkv_bm_refcount(const pkv_block_manager* bm, int64_t block);

/* A new sequence holding num_tokens tokens (its prompt) in fresh blocks. */
PKV_API pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, int64_t num_tokens);
/* child_id shares every block of parent_id (parallel sampling, beam search). */
PKV_API pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);
/* Drop a sequence; blocks no other sequence holds go back to the free list. */
PKV_API pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);

/*
 * One new token for each of n distinct sequences.  slots[i] receives the flat
 * slot (physical_block * block_size + offset) of seq_ids[i]'s new token.  A
 * sequence whose last block is partly filled and shared gets a private copy
 * first: (shared block, new block) is appended to cow_pairs (host int64
 * [cow_capacity][2]) and *num_cow counts the pairs, to be passed to
 * pkv_copy_blocks before the slot writes.  PKV_ERR_OOM if the free list cannot
 * cover every sequence of the call.
 */
PKV_API pkv_status pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int64_t n, int64_t* slots,
                                       int64_t* cow_pairs, int64_t cow_capacity, int64_t* num_cow);

/* Block tables (host int32 [n][max_blocks_per_seq], rows padded with `pad`)
 * and lengths (host int32 [n]) of n sequences, the decode call's inputs. */
PKV_API pkv_status pkv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int64_t n,
                                       int32_t* tables, int max_blocks_per_seq, int32_t pad, int32_t* seq_lens);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
