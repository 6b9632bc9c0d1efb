"""Pins of the CPU oracle to what the pages and the mathematics fix.

No GPU.  Each check compares the oracle with something other than itself: the
pages' printed numbers and worked examples (``tests/golden``), closed forms,
invariants, special cases, brute force, and an independent indexing route.
``test_planted_mistakes_are_caught`` plants plausible mistakes in the oracle
(on the CPU) and requires at least one pin to fail for each.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import BF16, F16, NAN_BITS, f32_to_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def bits(x, dtype=F16):
    return f32_to_bits(np.asarray(x, dtype=np.float32), dtype)


def contiguous_pool(K, V, block_size, dtype=F16, perm=None, extra_blocks=0):
    """Place per-sequence contiguous K/V [L, Hkv, d] (float arrays) into a paged pool.

    Returns (kc, vc, table_row).  ``perm`` gives the physical id of each logical
    block; unused slots are NaN.
    """
    L, Hkv, d = K.shape
    nb = -(-L // block_size)
    NB = nb + extra_blocks
    if perm is None:
        perm = list(range(nb))
    nan = NAN_BITS[dtype]
    kc = np.full((NB, block_size, Hkv, d), nan, dtype=np.uint16)
    vc = np.full((NB, block_size, Hkv, d), nan, dtype=np.uint16)
    kb, vb = bits(K, dtype), bits(V, dtype)
    for t in range(L):
        kc[perm[t // block_size], t % block_size] = kb[t]
        vc[perm[t // block_size], t % block_size] = vb[t]
    return kc, vc, np.asarray(perm, dtype=np.int64)


# ---------------------------------------------------------------- element decoding
def test_decode_bits_known_patterns():
    f16 = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF], dtype=np.uint16)
    assert oracle.decode_bits(f16, F16).tolist() == [1.0, -2.0, 2.0 ** -24, 65504.0]
    b16 = np.array([0x3F80, 0xC000, 0x3E80, 0x0001], dtype=np.uint16)
    assert oracle.decode_bits(b16, BF16).tolist() == [1.0, -2.0, 0.25, 2.0 ** -133]


# ---------------------------------------------------------------- sizes
def test_kv_cache_bytes_exact_examples():
    g = _gold("kv_size_examples.json")
    for e in g["kv_cache_size_exact"]:
        got = oracle.kv_cache_bytes(e["num_layers"], e["seq_len"], e["num_kv_heads"], e["head_dim"], e["dtype_size"])
        assert got == e["bytes"], e["cite"]
    # P2 §1.1 "≈ 80 MB" is 80 MiB; P2 §4.1 "≈ 16 KB" is 16 KiB
    assert oracle.kv_cache_bytes(80, 2048, 1, 128, 2) == 80 * 2 ** 20
    assert oracle.kv_cache_bytes(32, 1, 1, 128, 2) == 16 * 2 ** 10


def test_kv_cache_bytes_printed_5_and_2_gib():
    """P4 §一 prints 5.00 GB and 2.00 GB.  The formula as written gives 1.25 / 0.50 GiB
    with the stated 8 KV heads; the printed values are exactly those of 32 KV heads.
    The ratio 5.00 / 2.00 = 80 / 32 holds for any head count."""
    g = _gold("kv_size_examples.json")
    for e in g["kv_cache_size_printed"]:
        stated = oracle.kv_cache_bytes(e["num_layers"], e["seq_len"], e["num_kv_heads_stated"], e["head_dim"], e["dtype_size"])
        assert stated / 2 ** 30 == e["formula_gib_with_stated_heads"]
        repro = oracle.kv_cache_bytes(e["num_layers"], e["seq_len"], e["num_kv_heads_reproducing_print"], e["head_dim"], e["dtype_size"])
        assert f"{repro / 2 ** 30:.2f}" == f"{e['printed_gib']:.2f}"
    a, b = g["kv_cache_size_printed"]
    for h in (1, 8, 32):
        r = oracle.kv_cache_bytes(a["num_layers"], 4096, h, 128, 2) / oracle.kv_cache_bytes(b["num_layers"], 4096, h, 128, 2)
        assert r == a["printed_gib"] / b["printed_gib"]
    assert oracle.kv_cache_bytes(80, 4096, 8, 128, 2) == 1342177280


def test_pool_sizing_printed_numbers():
    g = _gold("kv_size_examples.json")
    p2, p4a, p4b = g["pool_sizing"]
    # P2 §4.1: 61 GB / 16 KB ≈ 3.8M tokens, / 16 ≈ 237,500 blocks (decimal units)
    per_tok = oracle.kv_cache_bytes(32, 1, 1, 128, 2)
    tokens = p2["kv_budget_decimal_gb"] * 1e9 / (p2["per_token_bytes_decimal_kb"] * 1e3)
    assert f"{tokens / 1e6:.1f}M" == "3.8M"
    assert round(tokens / 1e5) * 1e5 / p2["block_size"] == p2["blocks_printed"]
    assert per_tok == 16384
    # P4 §4.2: 56 GB / 0.125 MB = 448,000 blocks(=tokens) ; x16 = 7,168,000 ; /4096 = 1750 ≈ 1700
    per_tok = oracle.kv_cache_bytes(32, 1, 8, 128, 2)
    assert per_tok / 2 ** 20 == p4a["per_token_mib"]
    n = int(p4a["kv_budget_decimal_gb"] * 1000 / (per_tok / 2 ** 20))
    assert n == p4a["blocks_printed"]
    assert n * p4a["block_size"] == p4a["tokens_printed"]
    assert abs(n * p4a["block_size"] / p4a["context"] - p4a["seqs_printed_approx"]) < 100
    # P4 §7.3: reproduces with one token's bytes per "block"; the listing's
    # block_size factor gives 30,310, which the page does not print
    kv_avail = p4b["gpu_memory_gb"] * p4b["gpu_util"] - p4b["model_weight_gb"]
    assert f"{kv_avail:.1f}" == f"{p4b['kv_available_printed_gb']:.1f}"
    per_tok = oracle.kv_cache_bytes(p4b["num_layers"], 1, p4b["num_kv_heads"], p4b["head_dim"], p4b["dtype_size"])
    # 0.3125 printed as 0.313 (half-up rounding; Python's format rounds the tie to even)
    assert math.floor(per_tok / 2 ** 20 * 1000 + 0.5) / 1000 == p4b["block_mb_printed"]
    nb = int(kv_avail * 1024 ** 3 / per_tok)
    assert nb == p4b["num_blocks_printed"]
    assert nb * p4b["block_size"] == p4b["max_tokens_printed"]
    assert nb * p4b["block_size"] // p4b["avg_context"] == p4b["recommended_seqs_printed"]
    per_blk = oracle.kv_cache_bytes(p4b["num_layers"], p4b["block_size"], p4b["num_kv_heads"], p4b["head_dim"], p4b["dtype_size"])
    assert int(kv_avail * 1024 ** 3 / per_blk) == p4b["num_blocks_from_listing_as_printed"]


def test_num_logical_blocks():
    g = _gold("kv_size_examples.json")
    for c in g["block_counts"]:
        for n, want in c["cases"]:
            assert oracle.num_logical_blocks(n, c["block_size"]) == want
    for bs in (8, 16, 32):
        for n in range(0, 200):
            nb = oracle.num_logical_blocks(n, bs)
            assert nb * bs >= n and (nb - 1) * bs < max(n, 1)
            # at most one block is partly filled (P3 §2.2: waste below one block)
            assert nb * bs - n < bs


# ---------------------------------------------------------------- slots
def test_slot_placements_three_level_map():
    g = _gold("block_mapping_examples.json")["three_level_map"]
    for pos, blk, off in g["placements"]:
        slot = oracle.slot_for_position(g["block_table"], pos, g["block_size"])
        assert oracle.physical_location(slot, g["block_size"]) == (blk, off)


def test_append_slot_examples():
    g = _gold("block_mapping_examples.json")["append_slot"]
    bs = g["block_size"]
    for c in g["cases"]:
        blocks = list(c["blocks"])
        if c["new_block"] is not None:
            assert c["current_len"] % bs == 0 and c["current_len"] == len(blocks) * bs
            blocks.append(c["new_block"])
        assert oracle.slot_for_position(blocks, c["current_len"], bs) == c["slot"]
    fig = _gold("block_mapping_examples.json")["pagedattention_figure"]
    # every position of request A lands in the figure's blocks, in order
    tA = fig["tables"]["A"]
    seen = [oracle.physical_location(oracle.slot_for_position(tA, p, 16), 16)[0] for p in range(64)]
    assert seen == [b for b in tA for _ in range(16)]


def test_block_engine_ref_append_slot_examples():
    """The reference block manager hands out the pages' append_slot slots (P2 §2.3)."""
    g = _gold("block_mapping_examples.json")["append_slot"]
    bs = g["block_size"]
    for c in g["cases"]:
        first = list(c["blocks"]) + ([c["new_block"]] if c["new_block"] is not None else [])
        NB = max(first) + 4
        order = first + [b for b in range(NB) if b not in first]
        eng = oracle.BlockEngineRef(NB, bs, free_order=order)
        assert eng.allocate(0, c["current_len"]) and eng.tables[0] == list(c["blocks"])
        slots, pairs = eng.append_slots([0])
        assert slots == [c["slot"]] and pairs == []
        if c["new_block"] is not None:
            assert eng.tables[0][-1] == c["new_block"]


def test_block_engine_ref_invariants_under_random_operations():
    """Every block is free or held, never both; a block's count is the number of
    sequences holding it; a failed call changes nothing (P2 §2.3, §3.3; P4 §五)."""
    rng = np.random.default_rng(9)
    NB, bs = 24, 4
    eng = oracle.BlockEngineRef(NB, bs, free_order=rng.permutation(NB))
    live, nxt = [], 0

    def check():
        held = {}
        for t in eng.tables.values():
            for b in t:
                held[b] = held.get(b, 0) + 1
        free = list(eng.free_list)
        assert len(set(free)) == len(free) and not set(free) & set(held)
        assert len(free) + len(held) == NB
        assert all(eng.ref[b] == n for b, n in held.items()) and all(eng.ref[b] == 0 for b in free)
        for sid, t in eng.tables.items():
            assert len(t) == oracle.num_logical_blocks(eng.lens[sid], bs)

    for _ in range(400):
        op = rng.integers(4)
        if op == 0:
            if eng.allocate(nxt, int(rng.integers(0, 13))):
                live.append(nxt)
            nxt += 1
        elif op == 1 and live:
            if eng.fork(live[int(rng.integers(len(live)))], nxt):
                live.append(nxt)
            nxt += 1
        elif op == 2 and live:
            sid = live.pop(int(rng.integers(len(live))))
            assert eng.free(sid)
        elif live:
            pick = list(rng.choice(live, size=min(len(live), int(rng.integers(1, 4))), replace=False))
            before = (list(eng.free_list), {k: list(v) for k, v in eng.tables.items()}, dict(eng.lens))
            r = eng.append_slots([int(x) for x in pick])
            if r is None:
                assert (list(eng.free_list), eng.tables, eng.lens) == before
            else:
                slots, pairs = r
                assert len(set(slots)) == len(slots)
                for src, dst in pairs:
                    assert eng.ref[dst] == 1 and src != dst
        check()


# ---------------------------------------------------------------- cache writes
def _rand_pool(rng, NB, bs, Hkv, d, dtype=F16):
    return (bits(rng.standard_normal((NB, bs, Hkv, d)), dtype),
            bits(rng.standard_normal((NB, bs, Hkv, d)), dtype))


def test_append_ref_matches_torch_index_route():
    rng = np.random.default_rng(0)
    NB, bs, Hkv, d, T = 11, 16, 3, 8, 9
    kc, vc = _rand_pool(rng, NB, bs, Hkv, d)
    k = bits(rng.standard_normal((T, Hkv, d)))
    v = bits(rng.standard_normal((T, Hkv, d)))
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    kc2, vc2 = kc.copy(), vc.copy()
    oracle.append_ref(kc2, vc2, k, v, slots)
    # independent route: torch CPU advanced indexing on the flat slot view
    tk = torch.from_numpy(kc.astype(np.int32)).view(NB * bs, Hkv, d)
    tv = torch.from_numpy(vc.astype(np.int32)).view(NB * bs, Hkv, d)
    keep = torch.from_numpy(slots >= 0)
    s = torch.from_numpy(slots)[keep]
    tk[s] = torch.from_numpy(k.astype(np.int32))[keep]
    tv[s] = torch.from_numpy(v.astype(np.int32))[keep]
    assert np.array_equal(kc2, tk.view(NB, bs, Hkv, d).numpy().astype(np.uint16))
    assert np.array_equal(vc2, tv.view(NB, bs, Hkv, d).numpy().astype(np.uint16))
    # the -1 entry wrote nothing: exactly T-1 slots changed
    changed = np.any(kc2.reshape(NB * bs, -1) != kc.reshape(NB * bs, -1), axis=1)
    assert set(np.nonzero(changed)[0].tolist()) == set(slots[slots >= 0].tolist())


def test_copy_blocks_ref_cow_example():
    g = _gold("block_mapping_examples.json")["cow_samples"]
    rng = np.random.default_rng(1)
    NB, bs, Hkv, d = 12, 16, 2, 8
    layers = [_rand_pool(rng, NB, bs, Hkv, d) for _ in range(3)]
    kcs = [l[0].copy() for l in layers]
    vcs = [l[1].copy() for l in layers]
    # sample 2 and 3 get private copies of the shared last block (Block2) in Block5, Block7
    pairs = np.array([[g["shared"][-1], g["private"][0][0]], [g["shared"][-1], g["private"][1][0]]])
    oracle.copy_blocks_ref(kcs, vcs, pairs)
    for (k0, v0), k1, v1 in zip(layers, kcs, vcs):
        for src, dst in pairs:
            assert np.array_equal(k1[dst], k0[src]) and np.array_equal(v1[dst], v0[src])
        untouched = [b for b in range(NB) if b not in pairs[:, 1]]
        assert np.array_equal(k1[untouched], k0[untouched]) and np.array_equal(v1[untouched], v0[untouched])


def test_swap_round_trip_preserves_attention():
    """Swapping a sequence's blocks out to a host pool and back in under new ids
    (P2 §3.2) leaves its attention unchanged once its table names the new ids."""
    rng = np.random.default_rng(13)
    NB, bs, Hkv, d, L = 20, 8, 2, 16, 37
    kc, vc = _rand_pool(rng, NB, bs, Hkv, d)
    table = np.array([3, 17, 0, 11, 5], dtype=np.int64)
    q = bits(rng.standard_normal((1, 4, d)))
    before = oracle.attention_ref(q, kc, vc, table[None], np.array([L]), 0.25, Hkv, F16)
    host_k = np.zeros((8, bs, Hkv, d), np.uint16)
    host_v = np.zeros((8, bs, Hkv, d), np.uint16)
    out_pairs = np.stack([table, np.arange(5)], axis=1)
    oracle.swap_blocks_ref([kc], [vc], [host_k], [host_v], out_pairs)
    assert all(np.array_equal(host_k[j], kc[b]) for j, b in enumerate(table))
    kc2 = np.full_like(kc, NAN_BITS[F16])
    vc2 = np.full_like(vc, NAN_BITS[F16])
    new_ids = np.array([9, 2, 14, 19, 6], dtype=np.int64)
    oracle.swap_blocks_ref([host_k], [host_v], [kc2], [vc2], np.stack([np.arange(5), new_ids], axis=1))
    after = oracle.attention_ref(q, kc2, vc2, new_ids[None], np.array([L]), 0.25, Hkv, F16)
    assert np.array_equal(before, after)


# ---------------------------------------------------------------- attention
def att_contig(q, K, V, scale, bs=16, dtype=F16, perm=None):
    """Oracle attention for one sequence with one KV head given float K/V [L, d]."""
    L, d = K.shape
    kc, vc, table = contiguous_pool(K[:, None, :], V[:, None, :], bs, dtype, perm=perm,
                                    extra_blocks=0 if perm is None else max(perm) + 1 - (-(-L // bs)))
    qb = bits(np.asarray(q)[None, None, :], dtype)
    return oracle.attention_ref(qb, kc, vc, table[None, :], np.array([L]), scale, 1, dtype)[0, 0]


def check_closed_form_two_tokens():
    """Two keys with scores ln 3 and 0 give weights 3/4 and 1/4 (logistic closed form)."""
    d = 4
    scale = 0.5
    q = np.array([2.0, 0, 0, 0])
    K = np.array([[math.log(3.0), 0, 0, 0], [0, 0, 0, 0]])
    # ln 3 is not representable; use the key value fp16 actually stores
    k0 = float(oracle.decode_bits(bits([math.log(3.0)]), F16)[0])
    V = np.array([[1.0, 0, 2, 0], [0, 1, 0, -4]])
    w0 = math.exp(scale * 2.0 * k0) / (math.exp(scale * 2.0 * k0) + 1.0)
    want = w0 * V[0] + (1 - w0) * V[1]
    got = att_contig(q, K, V, scale)
    assert np.allclose(got, want, rtol=0, atol=1e-14), (got, want)
    assert abs(w0 - 0.75) < 1e-3


def check_single_token_returns_v():
    rng = np.random.default_rng(2)
    K = rng.standard_normal((1, 64))
    V = rng.standard_normal((1, 64))
    got = att_contig(rng.standard_normal(64), K, V, 0.125)
    assert np.array_equal(got, oracle.decode_bits(bits(V[0]), F16))


def check_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(3)
    L, d = 37, 16
    K = np.repeat(rng.standard_normal((1, d)), L, axis=0)
    V = rng.standard_normal((L, d))
    Vr = oracle.decode_bits(bits(V), F16)
    got = att_contig(rng.standard_normal(d), K, V, 0.25)
    assert np.allclose(got, Vr.mean(axis=0), rtol=0, atol=1e-14)
    got0 = att_contig(rng.standard_normal(d), rng.standard_normal((L, d)), V, 0.0)
    assert np.allclose(got0, Vr.mean(axis=0), rtol=0, atol=1e-14)


def check_dominant_key():
    """One key scoring 60 above the rest carries all but ~e^-60 of the weight."""
    L, d = 20, 4
    K = np.zeros((L, d))
    K[13, 0] = 60.0
    V = np.arange(L * d, dtype=np.float64).reshape(L, d) / 8.0
    got = att_contig(np.array([1.0, 0, 0, 0]), K, V, 1.0)
    assert np.allclose(got, V[13], rtol=0, atol=1e-14)


def check_large_scores_stay_finite():
    L, d = 8, 4
    K = np.full((L, d), 60000.0)
    K[5] = 65000.0
    V = np.eye(L, d) + 1.0
    got = att_contig(np.array([1.0, 1, 1, 1]), K, V, 1.0)
    assert np.all(np.isfinite(got)) and np.allclose(got, V[5], atol=0)


def check_gqa_mapping():
    """KV head g holds V = g + 1 everywhere and constant keys, so out[h] = h // G + 1."""
    Hq, Hkv, d, L, bs = 12, 3, 8, 21, 8
    G = Hq // Hkv
    rng = np.random.default_rng(4)
    K = np.ones((L, Hkv, d))
    V = np.zeros((L, Hkv, d))
    for g in range(Hkv):
        V[:, g, :] = g + 1.0
    kc, vc, table = contiguous_pool(K, V, bs)
    q = bits(rng.standard_normal((1, Hq, d)))
    out = oracle.attention_ref(q, kc, vc, table[None], np.array([L]), 0.3, Hkv, F16)
    for h in range(Hq):
        assert np.all(out[0, h] == h // G + 1.0)


def check_gqa_equals_replicated_mha():
    rng = np.random.default_rng(5)
    Hq, Hkv, d, L, bs = 8, 2, 16, 30, 8
    G = Hq // Hkv
    K = rng.standard_normal((L, Hkv, d))
    V = rng.standard_normal((L, Hkv, d))
    q = bits(rng.standard_normal((1, Hq, d)))
    kc, vc, table = contiguous_pool(K, V, bs)
    gqa = oracle.attention_ref(q, kc, vc, table[None], np.array([L]), 0.25, Hkv, F16)
    kr, vr, table2 = contiguous_pool(np.repeat(K, G, axis=1), np.repeat(V, G, axis=1), bs)
    mha = oracle.attention_ref(q, kr, vr, table2[None], np.array([L]), 0.25, Hq, F16)
    assert np.array_equal(gqa, mha)


def check_permutation_and_block_size_invariance():
    rng = np.random.default_rng(6)
    L, d = 75, 16
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    ident = att_contig(q, K, V, 0.25, bs=16)
    nb = -(-L // 16)
    perm = list(rng.permutation(nb + 6)[:nb])
    permuted = att_contig(q, K, V, 0.25, bs=16, perm=perm)
    bs32 = att_contig(q, K, V, 0.25, bs=32)
    bs8 = att_contig(q, K, V, 0.25, bs=8, perm=list(rng.permutation(40)[:10]))
    assert np.array_equal(ident, permuted) and np.array_equal(ident, bs32) and np.array_equal(ident, bs8)
    # and the paged result equals attention over the contiguous rows directly
    Kr = oracle.decode_bits(bits(K), F16)
    Vr = oracle.decode_bits(bits(V), F16)
    qr = oracle.decode_bits(bits(q), F16)
    z = 0.25 * Kr @ qr
    p = np.exp(z - z.max())
    assert np.allclose(ident, p @ Vr / p.sum(), rtol=0, atol=1e-14)


def check_brute_force_tiny():
    """Scalar Python loops straight from the definition, B<=3, L<=20, d<=8."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, d, bs = 3, 4, 2, 8, 4
    lens = np.array([1, 7, 20])
    NB = 16
    perm = rng.permutation(NB)
    tables = np.full((B, 5), 99, dtype=np.int64)
    nxt = 0
    for s in range(B):
        for j in range(-(-lens[s] // bs)):
            tables[s, j] = perm[nxt]
            nxt += 1
    kc = bits(rng.standard_normal((NB, bs, Hkv, d)))
    vc = bits(rng.standard_normal((NB, bs, Hkv, d)))
    q = bits(rng.standard_normal((B, Hq, d)))
    scale = 1 / math.sqrt(d)
    got = oracle.attention_ref(q, kc, vc, tables, lens, scale, Hkv, F16)
    f = lambda x: float(np.asarray(x, dtype=np.uint16).view(np.float16))
    for s in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            zs = []
            for t in range(lens[s]):
                b, o = tables[s, t // bs], t % bs
                zs.append(scale * sum(f(q[s, h, i]) * f(kc[b, o, g, i]) for i in range(d)))
            mx = max(zs)
            ws = [math.exp(z - mx) for z in zs]
            for i in range(d):
                num = sum(ws[t] * f(vc[tables[s, t // bs], t % bs, g, i]) for t in range(lens[s]))
                assert abs(got[s, h, i] - num / sum(ws)) < 1e-12


def check_tail_never_read():
    """Poisoned (NaN) slots past seq_len and poisoned table padding are never read."""
    rng = np.random.default_rng(8)
    L, d, bs = 19, 8, 16
    kc, vc, table = contiguous_pool(rng.standard_normal((L, 1, d)), rng.standard_normal((L, 1, d)), bs)
    padded = np.concatenate([table, [2 ** 31 - 1, 999]])
    out = oracle.attention_ref(bits(rng.standard_normal((1, 1, d))), kc, vc, padded[None], np.array([L]), 0.3, 1, F16)
    assert np.all(np.isfinite(out))


def check_merge_identity():
    rng = np.random.default_rng(9)
    L, d = 300, 32
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    whole = oracle.softmax_attention(q, K, V, 0.2)
    for cuts in ([150], [1, 299], [64, 128, 256], list(range(10, 300, 10))):
        edges = [0] + cuts + [L]
        parts = [oracle.partial_attention(q, K[a:b], V[a:b], 0.2) for a, b in zip(edges[:-1], edges[1:])]
        merged = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
        assert np.allclose(merged, whole, rtol=0, atol=1e-13)
    m, l, o = oracle.partial_attention(q, K, V, 0.2)
    assert np.allclose(o / l, whole, rtol=0, atol=1e-14)


def check_empty_sequence_is_zero():
    kc = np.zeros((2, 16, 1, 8), dtype=np.uint16)
    out = oracle.attention_ref(bits(np.ones((1, 1, 8))), kc, kc, np.array([[5, 5]]), np.array([0]), 0.3, 1, F16)
    assert np.array_equal(out, np.zeros((1, 1, 8)))


def check_cow_shared_equals_private():
    """Forked sequences reading shared prefix blocks give the same outputs as the
    same sequences with private copies of every block (P2 §3.3, P4 §五)."""
    rng = np.random.default_rng(10)
    bs, Hkv, Hq, d, P = 8, 2, 4, 8, 29
    n = 3
    sfx = [0, 5, 17]
    prefK = rng.standard_normal((P, Hkv, d))
    prefV = rng.standard_normal((P, Hkv, d))
    sK = [rng.standard_normal((s, Hkv, d)) for s in sfx]
    sV = [rng.standard_normal((s, Hkv, d)) for s in sfx]
    q = bits(rng.standard_normal((n, Hq, d)))
    lens = np.array([P + s for s in sfx])
    # shared: prefix blocks once; the partly filled last prefix block copied per fork
    nbp = -(-P // bs)
    NB = 64
    nan = NAN_BITS[F16]
    kc = np.full((NB, bs, Hkv, d), nan, np.uint16)
    vc = np.full((NB, bs, Hkv, d), nan, np.uint16)
    free = list(rng.permutation(NB))
    pref_blocks = [free.pop() for _ in range(nbp)]
    for t in range(P):
        kc[pref_blocks[t // bs], t % bs] = bits(prefK[t])
        vc[pref_blocks[t // bs], t % bs] = bits(prefV[t])
    tables = np.full((n, 8), 777, np.int64)
    pairs = []
    for f in range(n):
        tb = list(pref_blocks)
        if f > 0:
            dst = free.pop()
            pairs.append((tb[-1], dst))
            tb[-1] = dst
        tables[f, :len(tb)] = tb
    oracle.copy_blocks_ref([kc], [vc], pairs)
    for f in range(n):
        tb = list(tables[f, :nbp])
        for i in range(sfx[f]):
            t = P + i
            if t // bs >= len(tb):
                tb.append(free.pop())
            kc[tb[t // bs], t % bs] = bits(sK[f][i])
            vc[tb[t // bs], t % bs] = bits(sV[f][i])
        tables[f, :len(tb)] = tb
    shared = oracle.attention_ref(q, kc, vc, tables, lens, 0.35, Hkv, F16)
    # private: each sequence in its own contiguous pool
    for f in range(n):
        Kf = np.concatenate([prefK, sK[f]])
        Vf = np.concatenate([prefV, sV[f]])
        kp, vp, tp = contiguous_pool(Kf, Vf, bs)
        priv = oracle.attention_ref(q[f:f + 1], kp, vp, tp[None], lens[f:f + 1], 0.35, Hkv, F16)
        assert np.array_equal(shared[f], priv[0])


def check_verify_reduces_to_decode_and_truncation():
    """One query token is the decode call; query token i of nq equals the decode of the
    sequence cut at its causal limit L - nq + i + 1."""
    rng = np.random.default_rng(11)
    Hq, Hkv, d, bs, nq = 8, 2, 16, 8, 3
    lens = np.array([9, 30, 3])
    NB = 20
    perm = rng.permutation(NB)
    tables = np.full((3, 4), 77, np.int64)
    k = 0
    for s_ in range(3):
        for j in range(-(-lens[s_] // bs)):
            tables[s_, j] = perm[k]
            k += 1
    kc = bits(rng.standard_normal((NB, bs, Hkv, d)))
    vc = bits(rng.standard_normal((NB, bs, Hkv, d)))
    q = bits(rng.standard_normal((3, nq, Hq, d)))
    one = oracle.verify_attention_ref(q[:, :1], kc, vc, tables, lens, 0.3, Hkv, F16)
    assert np.array_equal(one[:, 0], oracle.attention_ref(q[:, 0], kc, vc, tables, lens, 0.3, Hkv, F16))
    got = oracle.verify_attention_ref(q, kc, vc, tables, lens, 0.3, Hkv, F16)
    for i in range(nq):
        cut = lens - nq + i + 1
        want = oracle.attention_ref(q[:, i], kc, vc, tables, cut, 0.3, Hkv, F16)
        assert np.array_equal(got[:, i], want)


def check_verify_is_causal():
    """Keys after a query's limit cannot move its output, however large their scores."""
    rng = np.random.default_rng(12)
    d, bs, nq, L = 8, 16, 4, 12
    K = rng.standard_normal((L, 1, d)) * 0.1
    V = rng.standard_normal((L, 1, d))
    q = bits(np.ones((1, nq, 1, d)))
    kc, vc, table = contiguous_pool(K, V, bs)
    base = oracle.verify_attention_ref(q, kc, vc, table[None], np.array([L]), 1.0, 1, F16)
    K2 = K.copy()
    K2[L - 1] = 50.0                          # only query nq-1 may see position L-1
    kc2, vc2, _ = contiguous_pool(K2, V, bs)
    moved = oracle.verify_attention_ref(q, kc2, vc2, table[None], np.array([L]), 1.0, 1, F16)
    assert np.array_equal(base[0, :nq - 1], moved[0, :nq - 1])
    assert np.allclose(moved[0, nq - 1, 0], oracle.decode_bits(bits(V[L - 1, 0]), F16), atol=1e-10)


PINS = [check_closed_form_two_tokens, check_single_token_returns_v, check_identical_keys_give_mean_of_v,
        check_dominant_key, check_large_scores_stay_finite, check_gqa_mapping, check_gqa_equals_replicated_mha,
        check_permutation_and_block_size_invariance, check_brute_force_tiny, check_tail_never_read,
        check_merge_identity, check_empty_sequence_is_zero, check_cow_shared_equals_private,
        check_verify_reduces_to_decode_and_truncation, check_verify_is_causal]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_attention_pin(pin):
    pin()


# ---------------------------------------------------------------- planted mistakes
def _softmax_no_scale(q, K, V, scale):
    z = K @ q
    p = np.exp(z - z.max())
    return (p @ V) / p.sum()


def _softmax_kv_swapped(q, K, V, scale):
    z = scale * (V @ q)
    p = np.exp(z - z.max())
    return (p @ K) / p.sum()


def _softmax_unnormalised(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    z = scale * (K @ q)
    p = np.exp(z - z.max())
    return p @ V


def _softmax_sign(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    z = -scale * (K @ q)
    p = np.exp(z - z.max())
    return (p @ V) / p.sum()


def _softmax_no_max(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    with np.errstate(over="ignore", invalid="ignore"):
        p = np.exp(scale * (K @ q))
        return (p @ V) / p.sum()


def _gather_ignores_table(cache, row, L, g, dtype):
    bs = cache.shape[1]
    pieces = [cache[j, :min(bs, L - j * bs), g] for j in range(-(-L // bs))]
    return oracle.decode_bits(np.concatenate(pieces), dtype) if pieces else np.zeros((0, cache.shape[3]))


def _gather_off_by_one(cache, row, L, g, dtype):
    bs = cache.shape[1]
    L2 = L + 1
    pieces = [cache[int(row[j]), :min(bs, L2 - j * bs), g] for j in range(-(-L2 // bs))]
    return oracle.decode_bits(np.concatenate(pieces), dtype) if pieces else np.zeros((0, cache.shape[3]))


def _attention_mod_mapping(q, kc, vc, tables, lens, scale, Hkv, dtype):
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d))
    for s in range(B):
        for h in range(Hq):
            g = h % Hkv
            K = oracle.gather_sequence(kc, tables[s], int(lens[s]), g, dtype)
            V = oracle.gather_sequence(vc, tables[s], int(lens[s]), g, dtype)
            out[s, h] = oracle.softmax_attention(oracle.decode_bits(q[s, h], dtype), K, V, scale)
    return out


def _merge_wrong_weight(ms, ls, os):
    ms = np.asarray(ms)
    w = np.exp(ms.max() - ms)
    return sum(wi * oi for wi, oi in zip(w, os)) / float(np.dot(w, ls))


def _verify_with_limit(limit, head_map=lambda h, G, Hkv: h // G):
    """verify_attention_ref with query token i seeing positions t < limit(L, nq, i)."""
    def run(q, kc, vc, tables, lens, scale, Hkv, dtype):
        B, nq, Hq, d = q.shape
        G = Hq // Hkv
        out = np.zeros((B, nq, Hq, d))
        for s in range(B):
            L = int(lens[s])
            for h in range(Hq):
                g = head_map(h, G, Hkv)
                K = oracle.gather_sequence(kc, tables[s], L, g, dtype)
                V = oracle.gather_sequence(vc, tables[s], L, g, dtype)
                for i in range(nq):
                    vis = min(L, limit(L, nq, i))
                    if L <= 0 or vis <= 0:
                        continue
                    out[s, i, h] = oracle.softmax_attention(oracle.decode_bits(q[s, i, h], dtype), K[:vis], V[:vis],
                                                            scale)
        return out
    return run


def _verify_excludes_itself(*a):
    return _verify_with_limit(lambda L, nq, i: L - nq + i)(*a)


def _verify_sees_next_token(*a):
    return _verify_with_limit(lambda L, nq, i: L - nq + i + 2)(*a)


def _verify_reversed_queries(*a):
    return _verify_with_limit(lambda L, nq, i: L - i)(*a)


def _verify_no_causal_mask(*a):
    return _verify_with_limit(lambda L, nq, i: L)(*a)


def _verify_mod_mapping(*a):
    return _verify_with_limit(lambda L, nq, i: L - nq + i + 1, head_map=lambda h, G, Hkv: h % Hkv)(*a)


MUTANTS = [("softmax_attention", _softmax_no_scale), ("softmax_attention", _softmax_kv_swapped),
           ("softmax_attention", _softmax_unnormalised), ("softmax_attention", _softmax_sign),
           ("softmax_attention", _softmax_no_max), ("gather_sequence", _gather_ignores_table),
           ("gather_sequence", _gather_off_by_one), ("attention_ref", _attention_mod_mapping),
           ("merge_partials", _merge_wrong_weight), ("verify_attention_ref", _verify_excludes_itself),
           ("verify_attention_ref", _verify_sees_next_token), ("verify_attention_ref", _verify_reversed_queries),
           ("verify_attention_ref", _verify_no_causal_mask), ("verify_attention_ref", _verify_mod_mapping)]


def test_verify_mutant_scaffold_unmutated_passes_every_pin(monkeypatch):
    """The scaffold the verify mutants share, with the right causal limit and GQA mapping,
    passes every pin: what the pins catch in the mutants is the planted change."""
    monkeypatch.setattr(oracle, "verify_attention_ref", _verify_with_limit(lambda L, nq, i: L - nq + i + 1))
    for pin in PINS:
        pin()


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=lambda x: getattr(x, "__name__", x))
def test_planted_mistakes_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(oracle, name, mutant)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant.__name__}"
