"""GPU parity at long context: one sequence of 64K or 128K positions beside short ones.

Long sequences are why the pages page the KV cache at all ("tbr8.org PagedAttention
article" §一: the cache of one 4096-token sequence already runs to gigabytes at 80
layers; "vLLM核心概念" §4.2: blocks are allocated as the sequence grows).  Here one
sequence's blocks span a table of 4K to 8K entries, its partitions number 16 to 256
(the merge of many partials, not only the single-pass form for up to four), and a
one-position sequence shares the batch.  Every output is compared with the oracle,
through the separate calls and through the benchmark's planned, fused launch; the
tensor-core verify kernel (64 rows per KV head) and the decode over E4M3 pools run
the same 128K-position batch.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import (TOL, DeviceStep, max_abs_err, mean_abs_err, oracle_attention, oracle_caches_after_step,
                         to_bits, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0


LONG = [
    # 128K positions, GQA 4, bf16, block size 16 (8192 table entries), with a 77- and a 1-position sequence
    dict(num_seqs=3, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16, seed=71,
         lens=("fixed", (131072, 77, 1)), pool=("headroom", 0.05)),
    # 64K + 13 positions (a ragged last block), GQA 8, fp16, block size 32
    dict(num_seqs=2, num_heads=64, num_kv_heads=8, head_dim=128, block_size=32, dtype=W.F16, seed=72,
         lens=("fixed", (65549, 4096)), pool=("headroom", 0.05)),
    # one 66000-position sequence over a single KV head (8 query heads): the automatic size
    # must keep it within the 512 partitions a call accepts
    dict(num_seqs=1, num_heads=8, num_kv_heads=1, head_dim=128, block_size=16, dtype=W.F16, seed=76,
         lens=("fixed", (66000,)), pool=("headroom", 0.05)),
]


@pytest.mark.parametrize("partition_tokens", [0, 512])
@pytest.mark.parametrize("mode", ["separate", "fused"])
@pytest.mark.parametrize("case", range(len(LONG)))
def test_long_context_matches_oracle(case, mode, partition_tokens):
    wl = W.build(W.small_spec(**LONG[case]), values="none")
    s = wl.spec
    step = DeviceStep(wl, pools="device", partition_tokens=partition_tokens)
    pre_k, pre_v = to_bits(step.kc[0]), to_bits(step.vc[0])
    step.run() if mode == "separate" else step.run_planned_fused()
    torch.cuda.synchronize()
    kc, vc = oracle_caches_after_step(wl, pre_k, pre_v)
    assert np.array_equal(to_bits(step.kc[0]), kc) and np.array_equal(to_bits(step.vc[0]), vc)
    assert torch.isfinite(step.out[0]).all()
    ref = oracle_attention(wl, kc, vc)
    err = max_abs_err(step.out[0], ref)
    print(f"long context {wl.max_seq_len} ({mode}, partition {partition_tokens}): max abs err {err:.3g}, "
          f"mean {mean_abs_err(step.out[0], ref):.3g}")
    assert err <= TOL[s.dtype], f"max abs err {err}"


def _f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("partition_tokens", [0, 512])
def test_long_context_verify_matches_oracle(partition_tokens):
    """8 query tokens x GQA 8 = 64 rows per KV head (the tensor-core verify kernel) over a
    128K-position sequence beside shorter ones.  The long sequence's outputs average some
    48K effective positions, so they are small: besides the batch's absolute bound, its
    error is held to 1% of its largest output, which a wrong partition or merge breaks."""
    wl = W.build(W.small_spec(num_seqs=3, num_heads=64, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16,
                              seed=73, lens=("fixed", (131072, 77, 40)), pool=("headroom", 0.05)), values="none")
    s, nq = wl.spec, 8
    step = DeviceStep(wl, pools="device")
    pre_k, pre_v = to_bits(step.kc[0]), to_bits(step.vc[0])
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    q = W.normal_bits(np.random.default_rng(74), (s.num_seqs, nq, s.num_heads, s.head_dim), s.dtype)
    qd = to_dev(q, s.dtype)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_attention_verify(out, qd, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, partition_tokens=partition_tokens,
                               sum_seq_lens=int(wl.seq_lens.sum()))
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    kc, vc = oracle_caches_after_step(wl, pre_k, pre_v)
    ref = oracle.verify_attention_ref(q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    err = max_abs_err(out, ref)
    err_long = max_abs_err(out[:1], ref[:1])
    top_long = float(np.abs(ref[0]).max())
    print(f"long context verify ({partition_tokens}): max abs err {err:.3g}, mean {mean_abs_err(out, ref):.3g}; "
          f"128K sequence: max abs err {err_long:.3g}, largest output {top_long:.3g}; per sequence "
          f"{[round(max_abs_err(out[i:i + 1], ref[i:i + 1]), 5) for i in range(s.num_seqs)]}")
    assert err <= TOL[s.dtype], f"max abs err {err}"
    assert err_long <= 0.01 * top_long, f"128K sequence: max abs err {err_long} against outputs up to {top_long}"


@pytest.mark.parametrize("partition_tokens", [0, 512])
def test_long_context_fp8_matches_oracle(partition_tokens):
    """A 128K-position sequence over E4M3 pools (quantizing append, then decode)."""
    wl = W.build(W.small_spec(num_seqs=3, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16,
                              seed=75, kv_dtype=W.E4M3, lens=("fixed", (131072, 77, 1)), pool=("headroom", 0.05)),
                 values="none")
    s = wl.spec
    dk, dv = W.device_pools(wl, 0, "cuda")
    kc, vc = dk.cpu().numpy().copy(), dv.cpu().numpy().copy()
    ks, vs = wl.k_scales[0], wl.v_scales[0]
    pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv, _dev(wl.slot_mapping),
                            _f32(ks), _f32(vs))
    q = to_dev(wl.q, s.dtype)
    out = torch.empty_like(q)
    pkv.paged_attention_decode_fp8(out, q, dk, dv, _dev(wl.block_tables), _dev(wl.seq_lens), _f32(ks), _f32(vs),
                                   wl.scale, max_seq_len=wl.max_seq_len, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, ks, vs, s.dtype)
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    ref = oracle.attention_fp8_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                   ks, vs)
    err = max_abs_err(out, ref)
    print(f"long context E4M3 ({partition_tokens}): max abs err {err:.3g}, mean {mean_abs_err(out, ref):.3g}")
    assert err <= TOL[s.dtype], f"max abs err {err}"
