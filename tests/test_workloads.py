"""The seeded workloads are well formed (no GPU).

Checks the generated structure against the oracle's own derivations: every
slot the generator hands to the append equals the oracle's slot for that
position, the pools' sizes follow the KV-size formula, and the poison layout
is exactly "no token yet" so a skipped write or copy shows up as NaN.
"""
import numpy as np
import pytest

import oracle
import workloads as W


@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "llama2_70b_mixed_bs16", "llama2_70b_mixed_bs32",
                                  "cow_fork", "cow_fork_partial", "llama2_70b_step"])
def test_structure(name):
    spec = W.SPECS[name]
    wl = W.build(spec, values="none")
    bs = spec.block_size
    B = spec.num_seqs
    assert wl.seq_lens.shape == (B,) and wl.block_tables.shape[0] == B
    # table width is the longest sequence's block count (padding is poison)
    assert wl.block_tables.shape[1] == oracle.num_logical_blocks(wl.max_seq_len, bs)
    used = []
    for s in range(B):
        nb = oracle.num_logical_blocks(int(wl.seq_lens[s]), bs)
        row = wl.block_tables[s]
        assert np.all((row[:nb] >= 0) & (row[:nb] < wl.num_blocks))
        assert np.all((row[nb:] >= wl.num_blocks))
        used.extend(row[:nb].tolist())
    # pool bytes per layer = the KV-size formula over num_blocks * block_size tokens
    assert wl.pool_bytes_per_layer() == oracle.kv_cache_bytes(1, wl.num_blocks * bs, spec.num_kv_heads,
                                                              spec.head_dim, 2)
    # appended slots are the oracle's slots of each sequence's newest positions
    slots = set(int(x) for x in wl.slot_mapping if x >= 0)
    for s in range(B):
        L = int(wl.seq_lens[s])
        if spec.fork is None or L > spec.fork[2]:
            assert oracle.slot_for_position(wl.block_tables[s], L - 1, bs) in slots
    if spec.fork is None:
        assert len(set(used)) == len(used)          # no sharing without a fork
        assert wl.num_tokens == B and np.all(wl.slot_mapping >= 0)
        # valid-before-step slots are exactly positions [0, L-1)
        assert wl.valid_slots.sum() == int(wl.seq_lens.sum()) - B
    else:
        reqs, n, P, lo, hi = spec.fork
        assert wl.copy_pairs.shape == (reqs * (n - 1), 2)
        assert len(set(wl.copy_pairs[:, 1].tolist())) == len(wl.copy_pairs)
        assert not set(wl.copy_pairs[:, 1].tolist()) & set(wl.copy_pairs[:, 0].tolist())
        assert np.all((wl.seq_lens >= P + lo) & (wl.seq_lens <= P + hi))
        # forks of one request share every prefix block but the copied last one
        nbp = oracle.num_logical_blocks(P, bs)
        t = wl.block_tables
        assert np.array_equal(t[0, :nbp - 1], t[1, :nbp - 1]) and t[0, nbp - 1] != t[1, nbp - 1]


def test_lengths_and_shapes_follow_the_recipe():
    """The configurations' shapes and length distributions as the recipe states them (the
    workload table of the measurement section): a generator drift here would move every
    benchmark number without any test of the kernels noticing."""
    shape = lambda n: (W.SPECS[n].num_heads, W.SPECS[n].num_kv_heads, W.SPECS[n].head_dim, W.SPECS[n].block_size,
                       W.SPECS[n].dtype)
    wl = W.build(W.SPECS["tiny"], values="none")
    assert wl.seq_lens.tolist() == [1, 17, 33, 50] and shape("tiny") == (4, 4, 64, 16, W.F16)
    for name in ("llama3_8b", "llama3_8b_fp8"):
        L = W.build(W.SPECS[name], values="none").seq_lens
        assert len(L) == 64 and L.min() >= 512 and L.max() <= 4096 and shape(name) == (32, 8, 128, 16, W.BF16)
        assert L.min() < 800 and L.max() > 3800 and 1900 < L.mean() < 2700     # U[512, 4096]: mean 2304
    for name, bs in (("llama2_70b_mixed_bs16", 16), ("llama2_70b_mixed_bs32", 32)):
        L = W.build(W.SPECS[name], values="none").seq_lens
        assert len(L) == 128 and L.min() >= 32 and L.max() <= 8192 and shape(name) == (64, 8, 128, bs, W.F16)
        # lognormal, median 500, sigma 1.2: the sample median of 128 lies within about 0.3 of ln 500
        assert 370 < np.median(L) < 680 and np.std(np.log(L)) > 0.9
    a = W.build(W.SPECS["llama2_70b_mixed_bs16"], values="none").seq_lens
    b = W.build(W.SPECS["llama2_70b_mixed_bs32"], values="none").seq_lens
    assert np.array_equal(a, b)                                              # same lengths at both block sizes
    for name, prefix in (("cow_fork", 1024), ("cow_fork_partial", 1020)):
        wl = W.build(W.SPECS[name], values="none")
        assert wl.spec.num_seqs == 768 and shape(name) == (32, 8, 128, 8, W.F16)
        sfx = wl.seq_lens - prefix
        assert sfx.min() >= 0 and sfx.max() <= 512 and sfx.max() > 480 and 200 < sfx.mean() < 310
    wl = W.build(W.SPECS["llama2_70b_step"], values="none")
    assert wl.spec.num_layers == 80 and (wl.seq_lens == 4096).all() and len(wl.seq_lens) == 16
    assert shape("llama2_70b_step") == (64, 8, 128, 16, W.BF16)


def test_tiny_values_and_poison():
    wl = W.build(W.SPECS["tiny"])
    assert wl.num_blocks == 32 and wl.seq_lens.tolist() == [1, 17, 33, 50]
    kc = wl.key_caches[0]
    nan = W.NAN_BITS["f16"]
    assert np.all((kc == nan).all(axis=(2, 3)) == ~wl.valid_slots)
    # the oracle step over the tiny workload is finite: appended tokens fill the NaN slots it reads
    outs, kcs, vcs = oracle.decode_step_ref(wl.key_caches, wl.value_caches, wl.copy_pairs, wl.k_new, wl.v_new,
                                            wl.slot_mapping, wl.q, wl.block_tables, wl.seq_lens, wl.scale,
                                            wl.spec.num_kv_heads, wl.spec.dtype)
    assert np.all(np.isfinite(outs[0]))
    # without the append the newest position is NaN and so is the output
    bad = oracle.attention_ref(wl.q, wl.key_caches[0], wl.value_caches[0], wl.block_tables, wl.seq_lens,
                               wl.scale, 4, "f16")
    assert np.all(np.isnan(bad))


def test_seeded_reproducible():
    a = W.build(W.SPECS["tiny"])
    b = W.build(W.SPECS["tiny"])
    for x, y in [(a.q, b.q), (a.key_caches[0], b.key_caches[0]), (a.block_tables, b.block_tables)]:
        assert np.array_equal(x, y)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -9, 3.0], dtype=np.float32)
    got = W.f32_to_bits(x, W.BF16)
    # ties go to even mantissa: 1+2^-8 -> 1.0 ; 1+3*2^-8 -> 1+2^-6 ; -1-2^-9 -> -1.0
    assert got.tolist() == [0x3F80, 0x3F82, 0xBF80, 0x4040]


def test_e4m3_pools_finite_where_valid_and_poisoned_elsewhere():
    wl = W.build(W.small_spec(kv_dtype=W.E4M3, lens=("fixed", (5, 40, 17, 1)), num_seqs=4))
    for kc in (wl.key_caches[0], wl.value_caches[0]):
        assert kc.dtype == np.uint8
        vals = kc[wl.valid_slots]
        assert not np.any((vals & 0x7F) == W.E4M3_NAN)           # no NaN code in a slot that holds a token
        assert np.all(kc[~wl.valid_slots] == W.E4M3_NAN)
    assert len(wl.k_scales) == 1 and wl.k_scales[0].dtype == np.float32 and np.all(wl.k_scales[0] > 0)
    assert wl.pool_bytes_per_layer() == 2 * int(np.prod(wl.pool_shape()))


def test_bench_dtype_override():
    """bench.py --dtype runs a workload in the other 16-bit type, everything else unchanged."""
    import argparse
    import bench

    for name in ("llama3_8b", "llama2_70b_mixed_bs16", "llama3_8b_fp8"):
        base = W.SPECS[name]
        for dt in (W.F16, W.BF16):
            s = bench.workload_spec(argparse.Namespace(workload=name, dtype=dt))
            assert s.dtype == dt and s.kv_dtype == base.kv_dtype
            assert (s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, s.block_size, s.seed, s.lens) == \
                (base.num_seqs, base.num_heads, base.num_kv_heads, base.head_dim, base.block_size, base.seed, base.lens)
        assert bench.workload_spec(argparse.Namespace(workload=name, dtype=None)) is base
