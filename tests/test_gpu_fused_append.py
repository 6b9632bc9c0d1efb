"""GPU parity of the fused slot write + decode call (pkv_paged_kv_append_decode).

The fused call must leave the pools exactly as the oracle's append leaves
them (bit for bit, 16-bit and E4M3 pools), return outputs within the dtype's
tolerance of the oracle's attention, and return the very same output bits as
the separate append and decode calls on the same inputs.  Misuse (a slot that
is not the position seq_len - 1 of its sequence) writes nothing and raises the
error word's bounds bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, max_abs_err, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0, "a kernel raised the device error word"


def cuda_of(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


CASES = [
    dict(num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16,
         lens=("fixed", (1, 15, 16, 17, 64, 65, 1000, 2049, 0))),
    dict(num_heads=8, num_kv_heads=8, head_dim=64, block_size=8, dtype=W.F16, lens=("fixed", (3, 300, 129, 0, 64))),
    dict(num_heads=64, num_kv_heads=8, head_dim=128, block_size=32, dtype=W.F16, lens=("uniform", 1, 3000)),
    dict(num_heads=24, num_kv_heads=2, head_dim=128, block_size=16, dtype=W.BF16, lens=("fixed", (700, 5, 4096))),
    dict(num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16, kv_dtype=W.E4M3,
         lens=("fixed", (1, 64, 65, 2049, 0, 333))),
    dict(num_heads=64, num_kv_heads=8, head_dim=128, block_size=8, dtype=W.F16, kv_dtype=W.E4M3,
         lens=("uniform", 1, 2500)),
]


def build(case, seed):
    kw = dict(CASES[case])
    kw["num_seqs"] = len(kw["lens"][1]) if kw["lens"][0] == "fixed" else 24
    wl = W.build(W.small_spec(seed=seed, **kw))
    assert wl.num_tokens == wl.spec.num_seqs      # one new token (or a padding entry) per sequence
    return wl


def device_pools(wl, layer=0):
    s = wl.spec
    if s.fp8:
        return cuda_of(wl.key_caches[layer]), cuda_of(wl.value_caches[layer])
    return to_dev(wl.key_caches[layer], s.dtype), to_dev(wl.value_caches[layer], s.dtype)


def pool_bits(t):
    return t.cpu().numpy() if t.dtype == torch.uint8 else to_bits(t)


def oracle_step(wl, layer=0):
    s = wl.spec
    kc, vc = wl.key_caches[layer].copy(), wl.value_caches[layer].copy()
    if s.fp8:
        ks, vs = wl.k_scales[layer], wl.v_scales[layer]
        oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, ks, vs, s.dtype)
        ref = oracle.attention_fp8_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                       ks, vs)
    else:
        oracle.append_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping)
        ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    return kc, vc, ref


class Inputs:
    def __init__(self, wl, layer=0):
        s = wl.spec
        self.q = to_dev(wl.q, s.dtype)
        self.k = to_dev(wl.k_new, s.dtype)
        self.v = to_dev(wl.v_new, s.dtype)
        self.slots = cuda_of(wl.slot_mapping)
        self.tables = cuda_of(wl.block_tables)
        self.lens = cuda_of(wl.seq_lens)
        self.ks = cuda_of(wl.k_scales[layer]) if s.fp8 else None
        self.vs = cuda_of(wl.v_scales[layer]) if s.fp8 else None
        self.total = int(wl.seq_lens.sum())


def fused(wl, x, kc, vc, part, planned, ws):
    out = torch.full_like(x.q, float("nan"))
    pkv.paged_kv_append_decode(out, x.q, x.k, x.v, kc, vc, x.slots, x.tables, x.lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=ws, partition_tokens=part, planned=planned,
                               sum_seq_lens=x.total if planned else 0, k_scale=x.ks, v_scale=x.vs)
    return out


def unfused(wl, x, kc, vc, part):
    out = torch.full_like(x.q, float("nan"))
    if wl.spec.fp8:
        pkv.paged_kv_append_fp8(x.k, x.v, kc, vc, x.slots, x.ks, x.vs)
        pkv.paged_attention_decode_fp8(out, x.q, kc, vc, x.tables, x.lens, x.ks, x.vs, wl.scale,
                                       max_seq_len=wl.max_seq_len, partition_tokens=part)
    else:
        pkv.paged_kv_append(x.k, x.v, kc, vc, x.slots)
        pkv.paged_attention_decode(out, x.q, kc, vc, x.tables, x.lens, wl.scale, max_seq_len=wl.max_seq_len,
                                   partition_tokens=part)
    return out


@pytest.mark.parametrize("planned", [False, True])
@pytest.mark.parametrize("partition_tokens", [0, 64, 1024])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_matches_oracle_and_separate_calls(case, partition_tokens, planned):
    wl = build(case, 700 + case)
    s = wl.spec
    x = Inputs(wl)
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len, partition_tokens)
    kc, vc = device_pools(wl)
    if planned:
        pkv.decode_plan(ws, x.tables, x.lens, s.num_heads, kc, wl.max_seq_len, partition_tokens, sum_seq_lens=x.total)
    out = fused(wl, x, kc, vc, partition_tokens, planned, ws)
    kc2, vc2 = device_pools(wl)
    out2 = unfused(wl, x, kc2, vc2, partition_tokens)
    torch.cuda.synchronize()
    rk, rv, ref = oracle_step(wl)
    assert np.array_equal(pool_bits(kc), rk) and np.array_equal(pool_bits(vc), rv)
    assert torch.isfinite(out).all()
    err = max_abs_err(out, ref)
    assert err <= TOL[s.dtype], f"max abs err {err}"
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "fused and separate calls differ"


@pytest.mark.parametrize("partition_tokens", [0, 64])
@pytest.mark.parametrize("case", [0, 1, 2, 3, 4])
def test_inputs_ready_layers_match(case, partition_tokens):
    """One plan, then four layers' fused calls, every layer after the first with inputs_ready
    (its work item, table slice and first tiles are read before it waits for the preceding
    launch): the pools bit-exact against the oracle's append, the outputs bit-identical to the
    same calls without the flag and within tolerance of the oracle.  Case 0's short sequences
    put the new token in the first chunks (loaded only after its slot is written); case 3's 12
    query heads per KV head give two CTAs per KV head writing the same slot; case 4 (E4M3)
    accepts the flag and runs as without it."""
    wl = build(case, 900 + case)
    s = wl.spec
    x = Inputs(wl)
    layers = 4
    rk, rv, ref = oracle_step(wl)
    outs = {}
    for ready in (False, True):
        ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len,
                                 partition_tokens)
        pools = [device_pools(wl) for _ in range(layers)]
        pkv.decode_plan(ws, x.tables, x.lens, s.num_heads, pools[0][0], wl.max_seq_len, partition_tokens,
                        sum_seq_lens=x.total)
        outs[ready] = []
        for l, (kc, vc) in enumerate(pools):
            out = torch.full_like(x.q, float("nan"))
            pkv.paged_kv_append_decode(out, x.q, x.k, x.v, kc, vc, x.slots, x.tables, x.lens, wl.scale,
                                       max_seq_len=wl.max_seq_len, workspace=ws, partition_tokens=partition_tokens,
                                       planned=True, sum_seq_lens=x.total, k_scale=x.ks, v_scale=x.vs,
                                       inputs_ready=ready and l > 0)
            outs[ready].append(out)
        torch.cuda.synchronize()
        for kc, vc in pools:
            assert np.array_equal(pool_bits(kc), rk) and np.array_equal(pool_bits(vc), rv)
    for l in range(layers):
        assert torch.equal(outs[True][l].view(torch.int16), outs[False][l].view(torch.int16)), f"layer {l}"
        err = max_abs_err(outs[True][l], ref)
        assert err <= TOL[s.dtype], f"layer {l}: max abs err {err}"


def test_inputs_ready_needs_a_plan():
    wl = build(0, 950)
    x = Inputs(wl)
    kc, vc = device_pools(wl)
    out = torch.empty_like(x.q)
    with pytest.raises(ValueError):
        pkv.paged_kv_append_decode(out, x.q, x.k, x.v, kc, vc, x.slots, x.tables, x.lens, wl.scale,
                                   max_seq_len=wl.max_seq_len, inputs_ready=True)


@pytest.mark.parametrize("case", [0, 4])
def test_plan_once_fused_layers(case):
    """One plan, then the fused call on several layers' pools (the tickets reset between runs)."""
    wl = build(case, 740 + case)
    s = wl.spec
    x = Inputs(wl)
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len)
    pools = [device_pools(wl) for _ in range(3)]
    pkv.decode_plan(ws, x.tables, x.lens, s.num_heads, pools[0][0], wl.max_seq_len, sum_seq_lens=x.total)
    outs = [fused(wl, x, kc, vc, 0, True, ws) for kc, vc in pools]
    torch.cuda.synchronize()
    rk, rv, ref = oracle_step(wl)
    for (kc, vc), out in zip(pools, outs):
        assert np.array_equal(pool_bits(kc), rk) and np.array_equal(pool_bits(vc), rv)
        assert max_abs_err(out, ref) <= TOL[s.dtype]
        assert torch.equal(out.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("case", [0, 4])
def test_fused_full_size_batch(case):
    """The llama3_8b-shaped batch (64 sequences, 32 q / 8 kv heads) through the fused call, sampled."""
    spec = W.SPECS["llama3_8b_fp8" if case == 4 else "llama3_8b"]
    wl = W.build(spec, values="none")
    s = wl.spec
    x = Inputs(wl)
    kc, vc = W.device_pools(wl, 0, "cuda")
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len)
    pkv.decode_plan(ws, x.tables, x.lens, s.num_heads, kc, wl.max_seq_len, sum_seq_lens=x.total)
    out = fused(wl, x, kc, vc, 0, True, ws)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    kb, vb = pool_bits(kc), pool_bits(vc)
    # the new tokens landed, bit for bit (E4M3: the oracle's codes)
    seqs = np.random.default_rng(5).choice(s.num_seqs, 5, replace=False)
    ko, vo = kb.copy(), vb.copy()
    if s.fp8:
        oracle.append_fp8_ref(ko, vo, wl.k_new, wl.v_new, wl.slot_mapping, wl.k_scales[0], wl.v_scales[0], s.dtype)
        ref = oracle.attention_fp8_ref(wl.q[seqs], kb, vb, wl.block_tables[seqs], wl.seq_lens[seqs], wl.scale,
                                       s.num_kv_heads, s.dtype, wl.k_scales[0], wl.v_scales[0])
    else:
        oracle.append_ref(ko, vo, wl.k_new, wl.v_new, wl.slot_mapping)
        ref = oracle.attention_ref(wl.q[seqs], kb, vb, wl.block_tables[seqs], wl.seq_lens[seqs], wl.scale,
                                   s.num_kv_heads, s.dtype)
    assert np.array_equal(ko, kb) and np.array_equal(vo, vb)
    assert max_abs_err(out, ref, seqs) <= TOL[s.dtype]


@pytest.mark.parametrize("planned", [False, True])
def test_fused_refuses_a_foreign_slot(planned):
    """A slot that is not position seq_len - 1 of its sequence (or a slot for an empty
    sequence) is not written and raises the bounds bit; the other sequences are unaffected."""
    wl = build(0, 760)
    s = wl.spec
    x = Inputs(wl)
    lens = wl.seq_lens
    bad, empty = 6, int(np.nonzero(lens == 0)[0][0])
    slots = wl.slot_mapping.copy()
    free = np.nonzero(~wl.valid_slots.reshape(-1))[0]
    free = free[~np.isin(free, slots)]
    slots[bad] = free[0]                            # a free slot of the pool, not position L - 1
    slots[empty] = free[1]
    x.slots = cuda_of(slots)
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len)
    kc, vc = device_pools(wl)
    if planned:
        pkv.decode_plan(ws, x.tables, x.lens, s.num_heads, kc, wl.max_seq_len, sum_seq_lens=x.total)
    out = fused(wl, x, kc, vc, 0, planned, ws)
    torch.cuda.synchronize()
    assert pkv.device_error(reset=True) & 1, "the bounds bit must be raised"
    good = wl.slot_mapping.copy()
    good[[bad, empty]] = -1                        # what must have been written: every other sequence's token
    rk, rv = wl.key_caches[0].copy(), wl.value_caches[0].copy()
    oracle.append_ref(rk, rv, wl.k_new, wl.v_new, good)
    assert np.array_equal(pool_bits(kc), rk) and np.array_equal(pool_bits(vc), rv)
    others = np.array([i for i in range(s.num_seqs) if i not in (bad, empty)])
    ref = oracle.attention_ref(wl.q[others], rk, rv, wl.block_tables[others], lens[others], wl.scale,
                               s.num_kv_heads, s.dtype)
    assert max_abs_err(out, ref, others) <= TOL[s.dtype]


def test_fused_host_validation():
    wl = build(1, 770)
    s = wl.spec
    x = Inputs(wl)
    kc, vc = device_pools(wl)
    out = torch.empty_like(x.q)
    with pytest.raises(ValueError):                 # one new row per sequence
        pkv.paged_kv_append_decode(out, x.q, x.k[:-1], x.v[:-1], kc, vc, x.slots[:-1], x.tables, x.lens)
    with pytest.raises(ValueError):                 # slots are int64
        pkv.paged_kv_append_decode(out, x.q, x.k, x.v, kc, vc, x.slots.int(), x.tables, x.lens)


def test_fused_above_plan_limit_full_grid():
    """More sequences than the plan lists (the decode runs its full 3-D grid): the fused write
    is made by the CTA of the last partition, as with a plan."""
    B = pkv.PLAN_MAX_SEQS + 76
    rng = np.random.default_rng(790)
    lens = rng.integers(1, 700, B)
    lens[rng.random(B) < 0.05] = 0
    wl = W.build(W.small_spec(num_seqs=B, num_heads=16, num_kv_heads=4, head_dim=128, block_size=16, dtype=W.F16,
                              seed=791, lens=("fixed", tuple(int(x) for x in lens)), pool=("headroom", 0.1)))
    s = wl.spec
    x = Inputs(wl)
    kc, vc = device_pools(wl)
    out = fused(wl, x, kc, vc, 256, False, None)
    torch.cuda.synchronize()
    rk, rv = wl.key_caches[0].copy(), wl.value_caches[0].copy()
    oracle.append_ref(rk, rv, wl.k_new, wl.v_new, wl.slot_mapping)
    assert np.array_equal(pool_bits(kc), rk) and np.array_equal(pool_bits(vc), rv)
    seqs = np.random.default_rng(792).choice(B, 40, replace=False)
    ref = oracle.attention_ref(wl.q[seqs], rk, rv, wl.block_tables[seqs], wl.seq_lens[seqs], wl.scale,
                               s.num_kv_heads, s.dtype)
    assert torch.isfinite(out).all()
    assert max_abs_err(out, ref, seqs) <= TOL[s.dtype]
