"""The calls captured in a CUDA graph: a serving loop replays one decode step.

A graph of (input copies, plan, fused slot write + decode) is captured once
through the public calls and replayed on new inputs copied into the same
buffers; every replay must match the oracle (bit-exact caches, outputs within
the dtype's tolerance) and equal an eager run of the same calls bit for bit.
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


@pytest.mark.parametrize("planned", [False, True])
def test_replayed_step_matches_oracle(planned):
    wl = W.build(W.small_spec(num_seqs=12, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=W.BF16,
                              seed=880, lens=("uniform", 1, 2500)))
    s = wl.spec
    rng = np.random.default_rng(881)
    # device buffers the graph reads; host tensors copied into them before each replay
    q = to_dev(wl.q, s.dtype)
    k = to_dev(wl.k_new, s.dtype)
    v = to_dev(wl.v_new, s.dtype)
    slots = torch.from_numpy(wl.slot_mapping).cuda()
    tables = torch.from_numpy(wl.block_tables).cuda()
    lens = torch.from_numpy(wl.seq_lens).cuda()
    kc, vc = to_dev(wl.key_caches[0], s.dtype), to_dev(wl.value_caches[0], s.dtype)
    out = torch.empty_like(q)
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len)

    def step():
        if planned:
            pkv.decode_plan(ws, tables, lens, s.num_heads, kc, wl.max_seq_len)
        pkv.paged_kv_append_decode(out, q, k, v, kc, vc, slots, tables, lens, wl.scale, max_seq_len=wl.max_seq_len,
                                   workspace=ws, planned=planned)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                      # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        step()
    torch.cuda.synchronize()

    for rep in range(3):
        # a new step's inputs into the captured buffers; the pools restart from the workload's
        qb = W.normal_bits(rng, wl.q.shape, s.dtype)
        kb = W.normal_bits(rng, wl.k_new.shape, s.dtype)
        vb = W.normal_bits(rng, wl.v_new.shape, s.dtype)
        for dst, src in ((q, qb), (k, kb), (v, vb)):
            dst.copy_(to_dev(src, s.dtype))
        kc.copy_(to_dev(wl.key_caches[0], s.dtype))
        vc.copy_(to_dev(wl.value_caches[0], s.dtype))
        g.replay()
        torch.cuda.synchronize()
        got, kg, vg = out.clone(), kc.clone(), vc.clone()
        # the same calls, eagerly, from the same pools
        kc.copy_(to_dev(wl.key_caches[0], s.dtype))
        vc.copy_(to_dev(wl.value_caches[0], s.dtype))
        step()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), out.view(torch.int16)), f"replay {rep} differs from the eager run"
        rk, rv = wl.key_caches[0].copy(), wl.value_caches[0].copy()
        oracle.append_ref(rk, rv, kb, vb, wl.slot_mapping)
        assert np.array_equal(to_bits(kg), rk) and np.array_equal(to_bits(vg), rv)
        ref = oracle.attention_ref(qb, rk, rv, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
        assert max_abs_err(got, ref) <= TOL[s.dtype]
