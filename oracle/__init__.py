"""CPU oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import or run anything in this package.  The product library never calls it
and shares no code, header, table or helper with it.

Plain, single-threaded NumPy in float64.  Every function cites the passage of
the source pages that defines it.  The pages are four web articles on
PagedAttention / vLLM, cited by title and section:

* P1 "vLLM核心概念：PagedAttention原理、KV Cache分页管理、连续批处理、投机解码概览"
* P2 "LLM 推理引擎内部原理：PagedAttention、Continuous Batching 与现代推理架构剖析"
* P3 "LLM 推理优化深度实战：从 PagedAttention 到 Speculative Decoding 的工程架构"
* P4 the tbr8.org PagedAttention article (its title is not in the extract; cited
  by host and section heading)

Readings taken where the pages are silent or garbled (each is pinned by a
test in ``tests/test_oracle_pins.py``):

* query head h reads KV head ``h // (num_heads // num_kv_heads)`` (contiguous
  GQA grouping; P4 §2.2 gives only the shapes);
* the softmax runs over all positions t < seq_len of the sequence (P4 §2.2's
  pseudocode applies it to one scalar score, which is garbled; P2 §2.4 says
  the softmax and the V weighting follow the scores);
* the block table is indexed by the logical block index (P2 §2.4's listing
  indexes it by its length, a typo);
* a slot < 0 in ``slot_mapping`` writes nothing; seq_len = 0 gives zeros;
* ``seq_lens`` count the token appended in the same step.

Parity unpinned: P3 §一's "≈512MB" KV-size example; its own formula with its
stated L=80, d=8192, n=2048 gives 5 GiB, and no head count reproduces 512 MB,
so no test can pin it.
"""
from __future__ import annotations

import numpy as np

F16 = "f16"
BF16 = "bf16"
E4M3 = "e4m3"    # 8-bit KV cache elements (see ``e4m3_value``)


# --------------------------------------------------------------------------
# element decoding
# --------------------------------------------------------------------------
def decode_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """fp16 / bf16 bit patterns (uint16) or E4M3 codes (uint8) -> float64, exactly."""
    if dtype == E4M3:
        return e4m3_value(bits)
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# 8-bit KV cache elements (P3 §6.2: KV cache quantization, attention on
# low-precision K/V).  The page names no format; the reading taken is the OCP
# FP8 E4M3 format ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3
# mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448.  A
# per-KV-head scale multiplies the decoded element.
# --------------------------------------------------------------------------
def e4m3_value(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) -> float64, exactly, from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((e == 15) & ((c & 7) == 7), np.nan, out)


_E4M3_POS = e4m3_value(np.arange(0x7F, dtype=np.uint8))     # codes 0x00..0x7E: 0 .. 448, increasing


def e4m3_quantize(x: np.ndarray) -> np.ndarray:
    """float32 values -> E4M3 codes: round to nearest, ties to the even code;
    magnitudes above 448 (and infinities) become 448; NaN becomes 0x7F; the
    sign is kept, so tiny negatives give -0 (0x80)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 1, 0x7E)   # first grid value >= a
    lo = hi - 1
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a >= 448.0, 0x7E, code)
    code = np.where(a == 0.0, 0, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


def append_fp8_ref(key_cache: np.ndarray, value_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
                   slot_mapping: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray, dtype: str) -> None:
    """Quantize each new token's K/V rows into its slot of an E4M3 pool.

    As ``append_ref`` (P2 §2.3 slot, P1 §4.2.2), with element (t, h, i) stored
    as e4m3_quantize(float32(k[t, h, i]) / float32(k_scale[h])): the division
    in float32, as the kernel does it.  Caches are uint8 [NB, bs, Hkv, d];
    k, v are fp16 / bf16 bits [T, Hkv, d]; scales float32 [Hkv].
    """
    bs = key_cache.shape[1]
    ks = np.asarray(k_scale, dtype=np.float32)[:, None]
    vs = np.asarray(v_scale, dtype=np.float32)[:, None]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, o = physical_location(int(slot), bs)
        key_cache[b, o] = e4m3_quantize(decode_bits(k[t], dtype).astype(np.float32) / ks)
        value_cache[b, o] = e4m3_quantize(decode_bits(v[t], dtype).astype(np.float32) / vs)


# --------------------------------------------------------------------------
# sizes (P4 §一 formula; P2 §1.1 and §4.1 worked numbers)
# --------------------------------------------------------------------------
def kv_cache_bytes(num_layers: int, seq_len: int, num_kv_heads: int, head_dim: int,
                   dtype_size: int = 2) -> int:
    """Bytes of K plus V for ``seq_len`` tokens: 2 * L * S * H_kv * d * bytes.

    P4 §一 (``kv_cache_size``).  P2 §1.1 writes the same product with D for
    one head's width.
    """
    return 2 * num_layers * seq_len * num_kv_heads * head_dim * dtype_size


def num_logical_blocks(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of ``num_tokens`` occupies: ceil(num_tokens / block_size).

    P3 §2.1 (``BlockTable.num_blocks``); P4 §3 (``allocate``: 50 tokens -> 4
    blocks of 16, 4096 -> 256).
    """
    return (num_tokens + block_size - 1) // block_size


# --------------------------------------------------------------------------
# slot arithmetic (P2 §2.3 BlockEngine.append_slot; P4 §2.1 three-level map)
# --------------------------------------------------------------------------
def slot_for_position(block_table_row, pos: int, block_size: int) -> int:
    """Flat slot of logical position ``pos``: physical_block * block_size + offset.

    P2 §2.3: a token that lands in the last block at ``len % block_size`` gets
    ``blocks[-1] * block_size + len % block_size``; P4 §2.1: token t lives in
    logical block t // block_size, mapped through the table.
    """
    return int(block_table_row[pos // block_size]) * block_size + pos % block_size


def physical_location(slot: int, block_size: int):
    """(physical block, offset in block) of a flat slot."""
    return slot // block_size, slot % block_size


# --------------------------------------------------------------------------
# cache writes (bitwise; operate on uint16 bit arrays in place)
# --------------------------------------------------------------------------
def append_ref(key_cache: np.ndarray, value_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
               slot_mapping: np.ndarray) -> None:
    """Write each new token's K/V rows into its slot.

    Caches are [num_blocks, block_size, num_kv_heads, head_dim]; k, v are
    [T, num_kv_heads, head_dim].  For token t with slot >= 0:
    cache[slot // bs, slot % bs, :, :] = k[t] (P2 §2.3 slot, P1 §4.2.2 "增长").
    A negative slot writes nothing.
    """
    bs = key_cache.shape[1]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, o = physical_location(int(slot), bs)
        key_cache[b, o] = k[t]
        value_cache[b, o] = v[t]


def copy_blocks_ref(key_caches, value_caches, pairs) -> None:
    """Copy-on-write block copy: for each (src, dst), cache[dst] = cache[src], every layer.

    P2 §3.1 (``blocks_to_copy`` of the scheduler output, "用于 Copy-on-Write")
    and §3.3; P1 §4.2.2 ("复制该块后再写入"); P4 §五.  Pairs are applied in order.
    """
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        for kc, vc in zip(key_caches, value_caches):
            kc[dst] = kc[src]
            vc[dst] = vc[src]


def swap_blocks_ref(src_key_caches, src_value_caches, dst_key_caches, dst_value_caches, pairs) -> None:
    """Preemption swap: for each (src, dst), dst_cache[dst] = src_cache[src], every layer.

    P2 §3.1 (``blocks_to_swap_in`` / ``blocks_to_swap_out``) and §3.2 (a
    preempted request's blocks are copied to CPU memory and back).  The two
    pools may differ in size; a block keeps its contents, only its id changes.
    """
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        for sk, sv, dk, dv in zip(src_key_caches, src_value_caches, dst_key_caches, dst_value_caches):
            dk[dst] = sk[src]
            dv[dst] = sv[src]


# --------------------------------------------------------------------------
# attention (P4 §2.2 paged_attention_kernel, read per the module docstring)
# --------------------------------------------------------------------------
def gather_sequence(cache: np.ndarray, block_table_row, seq_len: int, kv_head: int,
                    dtype: str) -> np.ndarray:
    """Contiguous float64 [seq_len, head_dim] rows of one KV head of one sequence.

    Logical block j is physical block table[j]; within it token offset o is
    position j * block_size + o; positions >= seq_len are never read (P4 §2.2:
    the loop breaks at seq_len; the last block is partly filled).
    """
    bs = cache.shape[1]
    pieces = []
    for j in range(num_logical_blocks(seq_len, bs)):
        b = int(block_table_row[j])
        n = min(bs, seq_len - j * bs)          # the last block is filled up to seq_len
        pieces.append(cache[b, :n, kv_head])
    if not pieces:
        return np.zeros((0, cache.shape[3]), dtype=np.float64)
    return decode_bits(np.concatenate(pieces, axis=0), dtype)


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Textbook single-query attention: softmax_t(scale * q.K_t) weighted sum of V_t.

    z_t = scale * <q, K_t>;  p_t = exp(z_t - max z);  out = sum_t p_t V_t / sum_t p_t.
    P4 §2.2 (score = dot(q, k) / sqrt(head_dim), weighted by V); subtracting the
    maximum leaves the result unchanged and keeps exp finite.
    """
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    z = scale * (K @ q)
    p = np.exp(z - z.max())
    return (p @ V) / p.sum()


def attention_ref(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                  block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
                  num_kv_heads: int, dtype: str) -> np.ndarray:
    """Paged single-query attention for a batch; float64 [B, num_heads, head_dim].

    q: uint16 bits [B, Hq, d]; caches: uint16 bits [NB, bs, Hkv, d];
    block_tables: int [B, W]; seq_lens: int [B].  Query head h of sequence s
    attends over the gathered K/V of KV head h // (Hq / Hkv).
    """
    B, Hq, d = q.shape
    G = Hq // num_kv_heads
    out = np.zeros((B, Hq, d), dtype=np.float64)
    for s in range(B):
        L = int(seq_lens[s])
        for g in range(num_kv_heads):
            K = gather_sequence(key_cache, block_tables[s], L, g, dtype)
            V = gather_sequence(value_cache, block_tables[s], L, g, dtype)
            for h in range(g * G, (g + 1) * G):
                out[s, h] = softmax_attention(decode_bits(q[s, h], dtype), K, V, scale)
    return out


def attention_fp8_ref(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                      block_tables: np.ndarray, seq_lens: np.ndarray, scale: float, num_kv_heads: int,
                      q_dtype: str, k_scale: np.ndarray, v_scale: np.ndarray) -> np.ndarray:
    """Paged single-query attention over an E4M3 pool; float64 [B, num_heads, head_dim].

    As ``attention_ref`` (P4 §2.2) with K_t = e4m3_value(code) * k_scale[g] and
    V_t = e4m3_value(code) * v_scale[g] for KV head g (P3 §6.2: attention on
    the low-precision K/V).  q: fp16 / bf16 bits [B, Hq, d]; caches uint8.
    """
    B, Hq, d = q.shape
    G = Hq // num_kv_heads
    ks = np.asarray(k_scale, dtype=np.float32).astype(np.float64)
    vs = np.asarray(v_scale, dtype=np.float32).astype(np.float64)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    for s in range(B):
        L = int(seq_lens[s])
        for g in range(num_kv_heads):
            K = gather_sequence(key_cache, block_tables[s], L, g, E4M3) * ks[g]
            V = gather_sequence(value_cache, block_tables[s], L, g, E4M3) * vs[g]
            for h in range(g * G, (g + 1) * G):
                out[s, h] = softmax_attention(decode_bits(q[s, h], q_dtype), K, V, scale)
    return out


def verify_attention_ref(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                         block_tables: np.ndarray, seq_lens: np.ndarray, scale: float, num_kv_heads: int,
                         dtype: str) -> np.ndarray:
    """Multi-query paged attention; float64 [B, nq, num_heads, head_dim].

    q: uint16 bits [B, nq, Hq, d].  The last nq positions of sequence s are the
    query tokens' own (P1 §4.4.2: the target model scores all draft tokens in
    one pass; P3 §4.2 speculative_verify).  Query token i sees the prefix and
    the query tokens before it and itself, i.e. positions t < L_s - nq + i + 1
    (causal).  A query that sees no position gets zeros.
    """
    B, nq, Hq, d = q.shape
    G = Hq // num_kv_heads
    out = np.zeros((B, nq, Hq, d), dtype=np.float64)
    for s in range(B):
        L = int(seq_lens[s])
        for g in range(num_kv_heads):
            K = gather_sequence(key_cache, block_tables[s], L, g, dtype)
            V = gather_sequence(value_cache, block_tables[s], L, g, dtype)
            for i in range(nq):
                vis = L - nq + i + 1
                if L <= 0 or vis <= 0:
                    continue
                for h in range(g * G, (g + 1) * G):
                    out[s, i, h] = softmax_attention(decode_bits(q[s, i, h], dtype), K[:vis], V[:vis], scale)
    return out


def verify_attention_fp8_ref(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                             block_tables: np.ndarray, seq_lens: np.ndarray, scale: float, num_kv_heads: int,
                             q_dtype: str, k_scale: np.ndarray, v_scale: np.ndarray) -> np.ndarray:
    """Multi-query paged attention over an E4M3 pool; float64 [B, nq, num_heads, head_dim].

    ``verify_attention_ref`` (P1 §4.4.2, P3 §4.2: the causal mask among the
    query tokens) with the K/V of ``attention_fp8_ref`` (P3 §6.2: K_t =
    e4m3_value(code) * k_scale[g], V_t = e4m3_value(code) * v_scale[g]).
    q: fp16 / bf16 bits [B, nq, Hq, d]; caches uint8.
    """
    B, nq, Hq, d = q.shape
    G = Hq // num_kv_heads
    ks = np.asarray(k_scale, dtype=np.float32).astype(np.float64)
    vs = np.asarray(v_scale, dtype=np.float32).astype(np.float64)
    out = np.zeros((B, nq, Hq, d), dtype=np.float64)
    for s in range(B):
        L = int(seq_lens[s])
        for g in range(num_kv_heads):
            K = gather_sequence(key_cache, block_tables[s], L, g, E4M3) * ks[g]
            V = gather_sequence(value_cache, block_tables[s], L, g, E4M3) * vs[g]
            for i in range(nq):
                vis = L - nq + i + 1
                if L <= 0 or vis <= 0:
                    continue
                for h in range(g * G, (g + 1) * G):
                    out[s, i, h] = softmax_attention(decode_bits(q[s, i, h], q_dtype), K[:vis], V[:vis], scale)
    return out


# --------------------------------------------------------------------------
# split-K pieces: partial softmax over a slice of positions and its merge
# --------------------------------------------------------------------------
def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """(m, l, o) over one slice of positions: m = max z, l = sum exp(z - m), o = sum exp(z - m) V.

    The slice's softmax numerator and denominator relative to its own maximum;
    ``merge_partials`` recombines slices into the softmax over their union.
    """
    z = scale * (K @ q)
    m = z.max()
    p = np.exp(z - m)
    return m, p.sum(), p @ V


def merge_partials(ms, ls, os) -> np.ndarray:
    """Combine slice partials: M = max m_p; out = sum e^(m_p-M) o_p / sum e^(m_p-M) l_p."""
    ms = np.asarray(ms, dtype=np.float64)
    M = ms.max()
    w = np.exp(ms - M)
    num = sum(wi * np.asarray(oi, dtype=np.float64) for wi, oi in zip(w, os))
    den = float(np.dot(w, np.asarray(ls, dtype=np.float64)))
    return num / den


# --------------------------------------------------------------------------
# one decode step: copy-on-write copies, slot writes, attention
# --------------------------------------------------------------------------
def decode_step_ref(key_caches, value_caches, copy_pairs, k_new, v_new, slot_mapping,
                    q, block_tables, seq_lens, scale: float, num_kv_heads: int, dtype: str,
                    layers=None):
    """Apply one step to copies of the caches and return (per-layer outputs, caches).

    Order: copy-on-write copies (P2 §3.3, at the fork), then the new tokens'
    slot writes (P1 §4.2.2), then attention over [0, seq_len) (P4 §2.2).  Every
    layer gets the same copies and slot writes with its own K/V; ``layers``
    restricts the attention to a subset of layers.
    """
    kcs = [np.array(k, copy=True) for k in key_caches]
    vcs = [np.array(v, copy=True) for v in value_caches]
    if copy_pairs is not None and len(copy_pairs):
        copy_blocks_ref(kcs, vcs, copy_pairs)
    outs = {}
    for l in range(len(kcs)):
        kn = k_new[l] if isinstance(k_new, (list, tuple)) else k_new
        vn = v_new[l] if isinstance(v_new, (list, tuple)) else v_new
        append_ref(kcs[l], vcs[l], kn, vn, slot_mapping)
        if layers is None or l in layers:
            ql = q[l] if isinstance(q, (list, tuple)) else q
            outs[l] = attention_ref(ql, kcs[l], vcs[l], block_tables, seq_lens, scale,
                                    num_kv_heads, dtype)
    return outs, kcs, vcs


# --------------------------------------------------------------------------
# host block manager (P2 §2.3 BlockEngine, §3.3; P1 §4.2.2; P4 §五)
# --------------------------------------------------------------------------
class BlockEngineRef:
    """Plain reference of the host block manager.

    P2 §2.3: the free blocks form a FIFO list; ``allocate`` takes
    ceil(tokens / block_size) blocks from its front; the next token of a
    sequence goes to ``blocks[-1] * bs + len % bs`` unless the last block is
    full (``len % bs == 0``), in which case a block is taken from the front;
    an empty list means "no slot" (the scheduler must preempt); ``free``
    returns blocks to the back.  P2 §3.3 / P4 §五: a fork shares the parent's
    blocks, each block counting its holders, and a block is only returned when
    no sequence holds it.  P1 §4.2.2: a sequence about to write into a block
    that another sequence also holds first copies it into a block of its own.
    Calls that cannot complete change nothing and return False.
    """

    def __init__(self, num_blocks, block_size, free_order=None):
        from collections import deque

        self.bs = block_size
        self.free_list = deque(range(num_blocks) if free_order is None else [int(b) for b in free_order])
        self.ref = [0] * num_blocks
        self.tables = {}
        self.lens = {}

    def allocate(self, seq_id, num_tokens):
        if seq_id in self.tables or num_tokens < 0:
            return False
        n = num_logical_blocks(num_tokens, self.bs)
        if n > len(self.free_list):
            return False
        blocks = [self.free_list.popleft() for _ in range(n)]
        for b in blocks:
            self.ref[b] = 1
        self.tables[seq_id] = blocks
        self.lens[seq_id] = num_tokens
        return True

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            return False
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1
        return True

    def free(self, seq_id):
        if seq_id not in self.tables:
            return False
        for b in self.tables.pop(seq_id):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free_list.append(b)
        del self.lens[seq_id]
        return True

    def _blocks_needed(self, seq_ids):
        """Free blocks the call takes: one per sequence whose last block is full,
        and one per copy-on-write.  A shared block is copied by each writer only
        while another sequence still holds it (P1 §4.2.2), so of its r holders,
        k of them writing in this call, min(k, r - 1) copy it and the last holder
        writes in place."""
        full = 0
        writers = {}
        for s in seq_ids:
            last = self.tables[s][-1] if self.tables[s] else None
            if self.lens[s] % self.bs == 0:
                full += 1
            elif self.ref[last] > 1:
                writers[last] = writers.get(last, 0) + 1
        return full + sum(min(k, self.ref[b] - 1) for b, k in writers.items())

    def append_slots(self, seq_ids):
        """One token for each sequence; (slots, copy-on-write pairs) or None."""
        if len(set(seq_ids)) != len(seq_ids) or any(s not in self.tables for s in seq_ids):
            return None
        if self._blocks_needed(seq_ids) > len(self.free_list):
            return None
        slots, pairs = [], []
        for s in seq_ids:
            L, t = self.lens[s], self.tables[s]
            if L % self.bs == 0:
                b = self.free_list.popleft()
                self.ref[b] = 1
                t.append(b)
            elif self.ref[t[-1]] > 1:
                b = self.free_list.popleft()
                self.ref[b] = 1
                self.ref[t[-1]] -= 1
                pairs.append((t[-1], b))
                t[-1] = b
            slots.append(slot_for_position(t, L, self.bs))
            self.lens[s] = L + 1
        return slots, pairs
