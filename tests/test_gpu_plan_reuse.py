"""Plan once, run per layer: one work list serves every layer of a step.

Each planned run must equal, bit for bit, the single call (plan + run) on the
same layer, and the oracle within tolerance; a run repeated on the same plan
must repeat bit for bit (the merging CTA resets its ticket); a run whose
arguments do not fit its plan raises the bounds bit and stays in range.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, DeviceStep, max_abs_err, oracle_caches_after_step, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0, "a kernel raised the device error word"


@pytest.mark.parametrize("with_sum", [False, True])
@pytest.mark.parametrize("partition_tokens", [0, 64])
def test_plan_once_run_every_layer(partition_tokens, with_sum):
    wl = W.build(W.small_spec(num_seqs=6, num_heads=32, num_kv_heads=8, dtype=W.BF16, num_layers=3, seed=701,
                              lens=("fixed", (1500, 33, 700, 1, 2049, 64))))
    step = DeviceStep(wl, partition_tokens=partition_tokens)
    s = wl.spec
    total = int(wl.seq_lens.sum()) if with_sum else 0       # sizes the grid tighter when given
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, s.num_heads, step.kc[0], wl.max_seq_len,
                    partition_tokens, sum_seq_lens=total)
    planned = []
    for l in range(3):
        pkv.paged_kv_append(step.k_new, step.v_new, step.kc[l], step.vc[l], step.slot_mapping)
        out = torch.empty_like(step.q)
        pkv.paged_attention_decode(out, step.q, step.kc[l], step.vc[l], step.block_tables, step.seq_lens, wl.scale,
                                   max_seq_len=wl.max_seq_len, workspace=step.workspace,
                                   partition_tokens=partition_tokens, planned=True, sum_seq_lens=total)
        planned.append(out)
    again = torch.empty_like(step.q)                 # the same plan once more: tickets were reset
    pkv.paged_attention_decode(again, step.q, step.kc[2], step.vc[2], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=step.workspace,
                               partition_tokens=partition_tokens, planned=True, sum_seq_lens=total)
    for l in range(3):                               # the single call (its own plan) on each layer
        step.decode(l)
    torch.cuda.synchronize()
    assert torch.equal(again, planned[2])
    for l in range(3):
        assert torch.equal(planned[l], step.out[l]), f"layer {l}"
        kc, vc = oracle_caches_after_step(wl, wl.key_caches[l], wl.value_caches[l])
        ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
        assert max_abs_err(planned[l], ref) <= TOL[s.dtype]


def test_fp8_plan_once_run_twice():
    wl = W.build(W.small_spec(num_seqs=5, num_heads=16, num_kv_heads=4, kv_dtype=W.E4M3, seed=702,
                              lens=("fixed", (900, 65, 3000, 17, 128))))
    s = wl.spec
    dk = torch.from_numpy(wl.key_caches[0]).cuda()
    dv = torch.from_numpy(wl.value_caches[0]).cuda()
    ks, vs = (torch.from_numpy(x).cuda() for x in (wl.k_scales[0], wl.v_scales[0]))
    tables = torch.from_numpy(wl.block_tables).cuda()
    lens = torch.from_numpy(wl.seq_lens).cuda()
    pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv,
                            torch.from_numpy(wl.slot_mapping).cuda(), ks, vs)
    q = to_dev(wl.q, s.dtype)
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len, 0, q.device)
    pkv.decode_plan(ws, tables, lens, s.num_heads, dk, wl.max_seq_len)
    outs = [torch.empty_like(q) for _ in range(3)]
    for o in outs[:2]:
        pkv.paged_attention_decode_fp8(o, q, dk, dv, tables, lens, ks, vs, wl.scale, max_seq_len=wl.max_seq_len,
                                       workspace=ws, planned=True)
    pkv.paged_attention_decode_fp8(outs[2], q, dk, dv, tables, lens, ks, vs, wl.scale, max_seq_len=wl.max_seq_len,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    kc, vc = wl.key_caches[0].copy(), wl.value_caches[0].copy()
    oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, wl.k_scales[0], wl.v_scales[0], s.dtype)
    ref = oracle.attention_fp8_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                   wl.k_scales[0], wl.v_scales[0])
    assert max_abs_err(outs[0], ref) <= TOL[s.dtype]


def test_run_with_arguments_the_plan_does_not_fit_is_flagged():
    """Plan for 6 sequences, run for the first 3: entries of sequences 3..5 are skipped
    and flagged; the first 3 sequences' outputs are still right."""
    wl = W.build(W.small_spec(num_seqs=6, num_heads=16, num_kv_heads=4, seed=703,
                              lens=("fixed", (300, 900, 40, 700, 1200, 5))))
    step = DeviceStep(wl, partition_tokens=128)
    s = wl.spec
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, s.num_heads, step.kc[0], wl.max_seq_len, 128)
    out = torch.full((3, s.num_heads, s.head_dim), float("nan"), dtype=torch.float16, device="cuda")
    pkv.paged_attention_decode(out, step.q[:3].contiguous(), step.kc[0], step.vc[0], step.block_tables[:3].contiguous(),
                               step.seq_lens[:3].contiguous(), wl.scale, max_seq_len=wl.max_seq_len,
                               workspace=step.workspace, partition_tokens=128, planned=True)
    torch.cuda.synchronize()
    assert pkv.device_error(reset=True) & 1, "entries past the run's batch must raise the bounds bit"
    kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    ref = oracle.attention_ref(wl.q[:3], kc, vc, wl.block_tables[:3], wl.seq_lens[:3], wl.scale, s.num_kv_heads,
                               s.dtype)
    assert max_abs_err(out, ref) <= TOL[s.dtype]


def test_full_grid_batch_plans_nothing_and_runs():
    B = pkv.PLAN_MAX_SEQS + 9
    wl = W.build(W.small_spec(num_seqs=B, num_heads=8, num_kv_heads=2, head_dim=64, seed=704,
                              lens=("uniform", 1, 100), pool=("headroom", 0.1)))
    step = DeviceStep(wl, partition_tokens=64)
    s = wl.spec
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, s.num_heads, step.kc[0], wl.max_seq_len, 64)
    out = torch.empty_like(step.q)
    pkv.paged_attention_decode(out, step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=step.workspace, partition_tokens=64,
                               planned=True)
    torch.cuda.synchronize()
    kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    assert max_abs_err(out, ref) <= TOL[s.dtype]


def test_wrong_length_sum_is_flagged():
    """A sum_seq_lens below the real sum sizes the grid too small: the plan flags it (and
    drops the entries past the grid, never writing out of range)."""
    wl = W.build(W.small_spec(num_seqs=8, num_heads=16, num_kv_heads=4, seed=705,
                              lens=("fixed", (3000, 2500, 40, 900, 1200, 5, 64, 2047))))
    step = DeviceStep(wl, partition_tokens=64)
    s = wl.spec
    pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
    wrong = int(wl.seq_lens.sum()) // 4
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, s.num_heads, step.kc[0], wl.max_seq_len, 64,
                    sum_seq_lens=wrong)
    out = torch.empty_like(step.q)
    pkv.paged_attention_decode(out, step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=step.workspace, partition_tokens=64,
                               planned=True, sum_seq_lens=wrong)
    torch.cuda.synchronize()
    assert pkv.device_error(reset=True) & 1, "a wrong length sum must raise the bounds bit"
    # planned again with the right sum, the same workspace gives the right answer
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, s.num_heads, step.kc[0], wl.max_seq_len, 64,
                    sum_seq_lens=int(wl.seq_lens.sum()))
    pkv.paged_attention_decode(out, step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=step.workspace, partition_tokens=64,
                               planned=True, sum_seq_lens=int(wl.seq_lens.sum()))
    torch.cuda.synchronize()
    kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    assert max_abs_err(out, ref) <= TOL[s.dtype]
