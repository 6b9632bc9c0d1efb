"""GPU parity of paged_attention_verify (multi-query, causal) against the oracle.

The last num_queries positions of each sequence are the query tokens' own K/V;
query token i sees positions < L - num_queries + i + 1.  Cases cover query
rows that fit one 8-row group and several, more than 16 rows per KV head (the
tensor-core kernel: M = 64 tiles partly and wholly filled, M = 128 tiles, two
row groups per KV head), with and without the lengths' sum, one and several
partitions (merged from shared memory or, past what the ring holds, from
global memory), query tokens that see nothing in a late partition, an empty
sequence, both head sizes and every block size.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, DeviceStep, max_abs_err, mean_abs_err, oracle_caches_after_step, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0


CASES = [
    dict(num_heads=16, num_kv_heads=4, head_dim=128, block_size=16, dtype=W.BF16, nq=2,
         lens=("fixed", (2, 40, 1025, 300))),
    dict(num_heads=64, num_kv_heads=8, head_dim=128, block_size=8, dtype=W.F16, nq=4,
         lens=("fixed", (4, 1025, 700, 64, 65))),
    dict(num_heads=4, num_kv_heads=4, head_dim=64, block_size=32, dtype=W.F16, nq=3, lens=("fixed", (3, 17, 2000))),
    dict(num_heads=12, num_kv_heads=4, head_dim=128, block_size=16, dtype=W.BF16, nq=5, lens=("fixed", (130, 5, 513))),
    # more than 16 rows per KV head: the tensor-core verify kernel (an M = 64 tile up to 64 rows)
    dict(num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16, nq=5,
         lens=("fixed", (5, 6, 64, 65, 1500, 3000))),
    dict(num_heads=16, num_kv_heads=2, head_dim=128, block_size=32, dtype=W.F16, nq=8, lens=("fixed", (8, 900, 77))),
    dict(num_heads=8, num_kv_heads=1, head_dim=64, block_size=8, dtype=W.BF16, nq=10, lens=("fixed", (10, 400, 1025))),
    dict(num_heads=64, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.F16, nq=3, lens=("fixed", (0, 3, 2049, 700))),
    # 128 rows per KV head at head_dim 128 (the M = 128 tile), and 160 (two row groups, the second
    # holding 32 rows)
    dict(num_heads=64, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16, nq=16,
         lens=("fixed", (16, 1500, 3000))),
    dict(num_heads=32, num_kv_heads=4, head_dim=128, block_size=16, dtype=W.F16, nq=20,
         lens=("fixed", (20, 700, 2100))),
    # exactly 32 rows per KV head at head_dim 64 (an M = 64 tile, half of it empty rows)
    dict(num_heads=16, num_kv_heads=2, head_dim=64, block_size=16, dtype=W.BF16, nq=4,
         lens=("fixed", (4, 31, 33, 95, 97, 2100))),
]


@pytest.mark.parametrize("with_sum", [False, True])
@pytest.mark.parametrize("partition_tokens", [0, 64, 1024])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_verify_matches_oracle(case, partition_tokens, with_sum):
    kw = dict(CASES[case])
    nq = kw.pop("nq")
    kw["num_seqs"] = len(kw["lens"][1])
    wl = W.build(W.small_spec(seed=300 + case, **kw))
    step = DeviceStep(wl)
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    rng = np.random.default_rng(case)
    s = wl.spec
    q = W.normal_bits(rng, (s.num_seqs, nq, s.num_heads, s.head_dim), s.dtype)
    qd = to_dev(q, s.dtype)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_attention_verify(out, qd, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, partition_tokens=partition_tokens,
                               sum_seq_lens=int(wl.seq_lens.sum()) if with_sum else 0)
    torch.cuda.synchronize()
    kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    ref = oracle.verify_attention_ref(q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    assert torch.isfinite(out).all()
    err = max_abs_err(out, ref)
    assert err <= TOL[s.dtype], f"max abs err {err}"


# The benchmarked verify launches at full size (their workloads, query counts, workspace and
# lengths' sum): the 70B-shaped mixed batch at 32, 64 and 128 rows per KV head (tensor-core
# tiles of M = 64 half and wholly filled, then M = 128) and the 8B-shaped batch at 32 and 64 rows.
FULL = [("llama2_70b_mixed_bs16", 4), ("llama2_70b_mixed_bs16", 8), ("llama2_70b_mixed_bs16", 16),
        ("llama3_8b", 8), ("llama3_8b", 16)]


@pytest.mark.parametrize("name,nq", FULL)
def test_full_size_verify(name, nq):
    """Every output of every sequence against the oracle."""
    wl = W.build(W.SPECS[name], values="none")
    s = wl.spec
    assert len(wl.copy_pairs) == 0 and int(wl.seq_lens.min()) >= nq   # the query tokens' own slots exist
    step = DeviceStep(wl, pools="device")
    pre_k, pre_v = to_bits(step.kc[0]), to_bits(step.vc[0])
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    rng = np.random.default_rng(900 + nq)
    q = W.normal_bits(rng, (s.num_seqs, nq, s.num_heads, s.head_dim), s.dtype)
    qd = to_dev(q, s.dtype)
    out = torch.full_like(qd, float("nan"))
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads * nq, s.num_kv_heads, s.head_dim, wl.max_seq_len, 0, "cuda")
    pkv.paged_attention_verify(out, qd, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=ws, sum_seq_lens=int(wl.seq_lens.sum()))
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    kc, vc = oracle_caches_after_step(wl, pre_k, pre_v)
    ref = oracle.verify_attention_ref(q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    err = max_abs_err(out, ref)
    print(f"{name} verify nq={nq}: max abs err {err:.3g}, mean {mean_abs_err(out, ref):.3g} over all "
          f"{s.num_seqs} sequences x {nq} queries x "
          f"{s.num_heads} heads")
    assert err <= TOL[s.dtype], f"max abs err {err}"


def test_one_query_verify_is_the_decode_call():
    wl = W.build(W.small_spec(num_seqs=4, num_heads=32, num_kv_heads=8, dtype=W.BF16,
                              lens=("fixed", (900, 33, 2049, 1))))
    step = DeviceStep(wl, partition_tokens=256)
    step.run()
    out = torch.empty_like(step.q).unsqueeze(1)
    pkv.paged_attention_verify(out, step.q.unsqueeze(1).contiguous(), step.kc[0], step.vc[0], step.block_tables,
                               step.seq_lens, wl.scale, max_seq_len=wl.max_seq_len, partition_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], step.out[0])
