"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Slot writes and block copies must match bit for bit; attention outputs within
max-abs-error 2e-3 (fp16) / 1e-2 (bf16) of the float64 oracle.  Every batch,
from the edge cases to the full-size workloads run in the launch
configuration the benchmark times (automatic partition size), is compared
element by element over every output and every cache element it checks.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import (TOL, DeviceStep, max_abs_err, mean_abs_err, oracle_attention, oracle_caches_after_step, to_bits,
                         to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0, "a kernel raised the device error word"


def full_check(wl, step, layers=(0,)):
    """Every output and every cache element of the given layers against the oracle."""
    for l in layers:
        kc, vc = oracle_caches_after_step(wl, wl.key_caches[l], wl.value_caches[l])
        assert np.array_equal(to_bits(step.kc[l]), kc), "key cache differs from the oracle after the step"
        assert np.array_equal(to_bits(step.vc[l]), vc), "value cache differs from the oracle after the step"
        ref = oracle_attention(wl, kc, vc)
        err = max_abs_err(step.out[l], ref)
        assert err <= TOL[wl.spec.dtype], f"max abs err {err}"
        assert torch.isfinite(step.out[l]).all()


def test_tiny_step():
    wl = W.build(W.SPECS["tiny"])
    step = DeviceStep(wl)
    step.run()
    torch.cuda.synchronize()
    full_check(wl, step)


EDGE = [
    dict(num_heads=8, num_kv_heads=2, head_dim=128, block_size=16, dtype=W.F16, lens=("fixed", (5, 40, 17))),
    dict(num_heads=8, num_kv_heads=8, head_dim=64, block_size=8, dtype=W.BF16,
         lens=("fixed", (1, 8, 9, 63, 64, 65, 200))),
    dict(num_heads=32, num_kv_heads=4, head_dim=128, block_size=32, dtype=W.BF16,
         lens=("fixed", (0, 1, 31, 32, 33, 1000, 129))),
    dict(num_heads=16, num_kv_heads=1, head_dim=128, block_size=16, dtype=W.F16, lens=("fixed", (300, 77))),
    dict(num_heads=12, num_kv_heads=4, head_dim=64, block_size=16, dtype=W.F16, lens=("fixed", (100, 5, 64))),
    dict(num_heads=64, num_kv_heads=8, head_dim=128, block_size=8, dtype=W.F16,
         lens=("fixed", (2047, 513, 4096, 1))),
]


@pytest.mark.parametrize("partition_tokens", [0, 64, 128, 4096])
@pytest.mark.parametrize("case", range(len(EDGE)))
def test_edge_cases(case, partition_tokens):
    kw = dict(EDGE[case])
    kw["num_seqs"] = len(kw["lens"][1])
    wl = W.build(W.small_spec(seed=100 + case, **kw))
    step = DeviceStep(wl, partition_tokens=partition_tokens)
    step.run()
    torch.cuda.synchronize()
    full_check(wl, step)


def test_split_and_single_pass_agree_and_repeat_bitwise():
    wl = W.build(W.small_spec(num_seqs=5, num_heads=32, num_kv_heads=8, dtype=W.BF16, lens=("fixed", (3000, 700, 64, 65, 1500))))
    outs = []
    for p in (64, 256, 4096, 256):
        step = DeviceStep(wl, partition_tokens=p)
        step.run()
        outs.append(step.out[0].clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[1], outs[3]), "same partition size must repeat bit for bit"
    ref = oracle_attention(wl, *oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0]))
    for o in outs:
        assert max_abs_err(o, ref) <= TOL[W.BF16]


def test_block_size_and_placement_invariance():
    """The same logical K/V under bs 16 and bs 32 and two physical permutations gives
    bit-identical outputs (positions are consumed in the same 64-position chunks)."""
    base = W.build(W.small_spec(num_seqs=4, num_heads=16, num_kv_heads=4, block_size=16,
                                lens=("fixed", (900, 33, 257, 64)), pool=("headroom", 0.3)))
    kc0, vc0 = oracle_caches_after_step(base, base.key_caches[0], base.value_caches[0])
    outs = []
    for bs, seed in ((16, 1), (32, 2), (32, 3)):
        rng = np.random.default_rng(seed)
        L = base.seq_lens
        nb = [oracle.num_logical_blocks(int(x), bs) for x in L]
        NB = sum(nb) + 5
        perm = rng.permutation(NB)
        H, d = base.spec.num_kv_heads, base.spec.head_dim
        kc = np.full((NB, bs, H, d), W.NAN_BITS[W.F16], np.uint16)
        vc = kc.copy()
        tables = np.full((4, max(nb)), NB + 3, np.int32)
        nxt = 0
        for s in range(4):
            K = np.concatenate([kc0[base.block_tables[s, j]] for j in range(oracle.num_logical_blocks(int(L[s]), 16))])[:L[s]]
            V = np.concatenate([vc0[base.block_tables[s, j]] for j in range(oracle.num_logical_blocks(int(L[s]), 16))])[:L[s]]
            for j in range(nb[s]):
                b = perm[nxt]
                nxt += 1
                tables[s, j] = b
                rows = K[j * bs:(j + 1) * bs]
                kc[b, :len(rows)] = rows
                vc[b, :len(rows)] = V[j * bs:(j + 1) * bs]
        dk, dv = to_dev(kc, W.F16), to_dev(vc, W.F16)
        q = to_dev(base.q, W.F16)
        out = torch.empty_like(q)
        pkv.paged_attention_decode(out, q, dk, dv, torch.from_numpy(tables).cuda(), torch.from_numpy(L).cuda(),
                                   base.scale, max_seq_len=int(L.max()), partition_tokens=4096)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ---------------------------------------------------------------- the plan kernel and the full grid
@pytest.mark.parametrize("partition_tokens", [0, 64])
def test_batch_above_plan_limit_runs_the_full_grid(partition_tokens):
    """More sequences than the plan kernel lists: the full (head group, partition,
    sequence) grid, whose CTAs past their sequence's end return at once."""
    B = pkv.PLAN_MAX_SEQS + 77
    wl = W.build(W.small_spec(num_seqs=B, num_heads=8, num_kv_heads=2, head_dim=64, seed=501,
                              lens=("uniform", 0, 150), pool=("headroom", 0.1)))
    step = DeviceStep(wl, partition_tokens=partition_tokens)
    step.run()
    torch.cuda.synchronize()
    full_check(wl, step)
    s = wl.spec
    assert pkv.decode_plan_partition_tokens(step.workspace, B, s.num_heads, s.num_kv_heads) == -1


def test_plan_partition_size_bounds():
    """Automatic: at least the host's size, a multiple of 64, within the staged
    table, and no larger than the longest sequence needs; explicit: unchanged."""
    wl = W.build(W.small_spec(num_seqs=6, num_heads=32, num_kv_heads=8, dtype=W.BF16, seed=502,
                              lens=("fixed", (5000, 3000, 64, 1, 2100, 700))))
    s = wl.spec
    for p in (0, 192):
        step = DeviceStep(wl, partition_tokens=p)
        step.run()
        got = pkv.decode_plan_partition_tokens(step.workspace, s.num_seqs, s.num_heads, s.num_kv_heads)
        if p:
            assert got == p
        else:
            lo = pkv.decode_partition_tokens(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len)
            assert got % 64 == 0 and lo <= got <= max(lo, 512 * s.block_size, -(-int(wl.seq_lens.max()) // 64) * 64)
        torch.cuda.synchronize()
        full_check(wl, step)


@pytest.mark.parametrize("num_seqs", [5, pkv.PLAN_MAX_SEQS + 3])
def test_lengths_above_max_seq_len_are_clamped_and_flagged(num_seqs):
    """A length above max_seq_len breaks the call's precondition: the call attends
    over max_seq_len positions and raises the bounds bit (planned and full grid)."""
    rng = np.random.default_rng(503)
    lens = rng.integers(1, 300, size=num_seqs)
    lens[:3] = (299, 150, 40)
    wl = W.build(W.small_spec(num_seqs=num_seqs, num_heads=8, num_kv_heads=2, head_dim=64, seed=504,
                              lens=("fixed", tuple(int(x) for x in lens)), pool=("headroom", 0.1)))
    step = DeviceStep(wl)
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    cap = 100
    out = torch.full_like(step.q, float("nan"))
    pkv.paged_attention_decode(out, step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=cap, partition_tokens=64)
    torch.cuda.synchronize()
    assert pkv.device_error(reset=True) & 1, "a length above max_seq_len must raise the bounds bit"
    kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, np.minimum(wl.seq_lens, cap), wl.scale,
                               wl.spec.num_kv_heads, wl.spec.dtype)
    assert max_abs_err(out, ref) <= TOL[wl.spec.dtype]


# ---------------------------------------------------------------- full-size workloads
FULL = ["llama3_8b", "llama2_70b_mixed_bs16", "llama2_70b_mixed_bs32", "cow_fork", "cow_fork_partial"]


@pytest.mark.parametrize("mode", ["separate", "fused"])
@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name, mode):
    """separate: append then decode calls; fused: the benchmark's launches (one plan with the
    lengths' sum, then the fused slot write + decode over it)."""
    wl = W.build(W.SPECS[name], values="none")
    if mode == "fused" and wl.num_tokens != wl.spec.num_seqs:
        pytest.skip("this step writes several slots per sequence: the benchmark launches the append")
    step = DeviceStep(wl, pools="device")
    pre_k, pre_v = to_bits(step.kc[0]), to_bits(step.vc[0])
    step.run() if mode == "separate" else step.run_planned_fused()
    torch.cuda.synchronize()
    s = wl.spec
    part = pkv.decode_plan_partition_tokens(step.workspace, s.num_seqs, s.num_heads, s.num_kv_heads)
    assert part % 64 == 0 and part >= pkv.decode_partition_tokens(s.num_seqs, s.num_heads, s.num_kv_heads,
                                                                   s.head_dim, wl.max_seq_len)
    kc, vc = oracle_caches_after_step(wl, pre_k, pre_v)
    assert np.array_equal(to_bits(step.kc[0]), kc)
    assert np.array_equal(to_bits(step.vc[0]), vc)
    assert torch.isfinite(step.out[0]).all()
    ref = oracle_attention(wl, kc, vc)              # every sequence, every head
    err = max_abs_err(step.out[0], ref)
    print(f"{name} ({mode}): max abs err {err:.3g}, mean {mean_abs_err(step.out[0], ref):.3g} over all "
          f"{s.num_seqs} sequences x {s.num_heads} heads")
    assert err <= TOL[wl.spec.dtype], f"{name}: max abs err {err}"


@pytest.mark.parametrize("mode", ["separate", "fused", "fused_inputs_ready"])
def test_full_size_80_layer_step(mode):
    wl = W.build(W.SPECS["llama2_70b_step"], values="none")
    step = DeviceStep(wl, pools="device")
    check_layers = (0, 41, 79)
    pre = {l: (to_bits(step.kc[l]), to_bits(step.vc[l])) for l in check_layers}
    step.run() if mode == "separate" else step.run_planned_fused(inputs_ready=mode == "fused_inputs_ready")
    torch.cuda.synchronize()
    for l in range(80):
        assert torch.isfinite(step.out[l]).all(), f"layer {l}"
    for l in check_layers:
        kc, vc = oracle_caches_after_step(wl, *pre[l])
        assert np.array_equal(to_bits(step.kc[l]), kc) and np.array_equal(to_bits(step.vc[l]), vc)
        ref = oracle_attention(wl, kc, vc)          # all 16 sequences, every head
        err = max_abs_err(step.out[l], ref)
        print(f"llama2_70b_step ({mode}) layer {l}: max abs err {err:.3g}, mean {mean_abs_err(step.out[l], ref):.3g} "
              f"over all sequences x heads")
        assert err <= TOL[W.BF16], f"layer {l}: {err}"


# ---------------------------------------------------------------- copy-on-write, append, errors
def test_copy_blocks_bit_exact_multi_layer():
    rng = np.random.default_rng(11)
    NB, bs, H, d = 40, 8, 8, 128
    layers = 3
    kcs = [W.normal_bits(rng, (NB, bs, H, d), W.F16) for _ in range(layers)]
    vcs = [W.normal_bits(rng, (NB, bs, H, d), W.F16) for _ in range(layers)]
    pairs = np.array([[0, 5], [3, 7], [0, 9], [12, 39]], dtype=np.int64)
    dk = [to_dev(x, W.F16) for x in kcs]
    dv = [to_dev(x, W.F16) for x in vcs]
    pkv.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    oracle.copy_blocks_ref(kcs, vcs, pairs)
    for l in range(layers):
        assert np.array_equal(to_bits(dk[l]), kcs[l]) and np.array_equal(to_bits(dv[l]), vcs[l])


def test_append_padding_and_empty():
    rng = np.random.default_rng(12)
    NB, bs, H, d = 6, 16, 2, 64
    kc = W.normal_bits(rng, (NB, bs, H, d), W.BF16)
    vc = W.normal_bits(rng, (NB, bs, H, d), W.BF16)
    k = W.normal_bits(rng, (5, H, d), W.BF16)
    v = W.normal_bits(rng, (5, H, d), W.BF16)
    slots = np.array([3, -1, 95, 17, -5], dtype=np.int64)
    dk, dv = to_dev(kc, W.BF16), to_dev(vc, W.BF16)
    pkv.paged_kv_append(to_dev(k, W.BF16), to_dev(v, W.BF16), dk, dv, torch.from_numpy(slots).cuda())
    # zero tokens is a no-op
    pkv.paged_kv_append(to_dev(k[:0], W.BF16), to_dev(v[:0], W.BF16), dk, dv, torch.from_numpy(slots[:0]).cuda())
    torch.cuda.synchronize()
    oracle.append_ref(kc, vc, k, v, slots)
    assert np.array_equal(to_bits(dk), kc) and np.array_equal(to_bits(dv), vc)


def test_out_of_range_ids_are_skipped_and_flagged():
    wl = W.build(W.small_spec(lens=("fixed", (40, 20, 5))))
    step = DeviceStep(wl)
    step.block_tables[1, 0] = wl.num_blocks + 100       # a block id past the pool
    step.slot_mapping[2] = wl.num_blocks * wl.spec.block_size + 3   # a slot past the pool
    before = to_bits(step.kc[0])
    step.run()
    err = pkv.device_error(reset=True)
    assert err & 1, "out-of-range ids must raise the bounds bit"
    assert torch.isfinite(step.out[0][0]).all() and torch.isfinite(step.out[0][1]).all()
    after = to_bits(step.kc[0])
    ref_k, _ = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    changed = np.any(after.reshape(-1, wl.spec.num_kv_heads * wl.spec.head_dim) != before.reshape(-1, wl.spec.num_kv_heads * wl.spec.head_dim), axis=1)
    # only the two in-range slots were written
    assert set(np.nonzero(changed)[0].tolist()) <= set(int(s) for s in wl.slot_mapping[:2])


def test_host_validation_errors():
    wl = W.build(W.small_spec(lens=("fixed", (300, 20, 5))))
    step = DeviceStep(wl, partition_tokens=64)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode(step.out[0], step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens,
                                   wl.scale, max_seq_len=300, workspace=small, partition_tokens=64)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode(step.out[0], step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens,
                                   wl.scale, max_seq_len=300, workspace=step.workspace, partition_tokens=100)
    assert e.value.status == pkv.PKV_ERR_INVALID
    with pytest.raises(ValueError):
        pkv.paged_kv_append(step.k_new.cpu(), step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
