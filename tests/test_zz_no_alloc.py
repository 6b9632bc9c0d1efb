"""The allocation-free decode entry point, pkv_paged_attention_decode_static.

It serves callers that cannot call cudaMalloc (for example a plugin that a
host engine gives only its input and output buffers), so its split-K scratch
is an array built into the library.  These tests call it through the C ABI
and compare its output with the regular entry point (which takes a caller
workspace) on the same inputs: bit for bit, since both run the same kernels
at the same partition size, and against the CPU oracle.  The calls come in a
row with different batches, so every later call runs on scratch that an
earlier call left behind: explicit split partitions, the automatic partition
(the plan kernel zeroes the merge counters in the array), and a batch of
more sequences than the plan lists (the counters are cleared by a memset).

The file name makes pytest collect it last: a run that stops at the first
failure has already run every other test.  It builds and loads the library
itself, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, DeviceStep, max_abs_err, oracle_attention, oracle_caches_after_step
from paged_kv_cache_156_gb300 import _build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    return pkv.load()


def decode_static(lib, step, partition_tokens):
    wl, s = step.wl, step.wl.spec
    out = torch.full_like(step.q, float("nan"))
    st = lib.pkv_paged_attention_decode_static(
        out.data_ptr(), step.q.data_ptr(), step.kc[0].data_ptr(), step.vc[0].data_ptr(), step.block_tables.data_ptr(),
        step.block_tables.shape[1], step.seq_lens.data_ptr(), s.num_seqs, wl.max_seq_len, s.num_heads,
        s.num_kv_heads, s.head_dim, s.block_size, wl.num_blocks, wl.scale, 0 if s.dtype == W.F16 else 1,
        partition_tokens, torch.cuda.current_stream().cuda_stream)
    assert st == pkv.PKV_OK, lib.pkv_last_error()
    return out


CASES = {
    # split partitions at an explicit size
    "A": (W.small_spec(num_seqs=5, num_heads=32, num_kv_heads=8, dtype=W.BF16, seed=31,
                       lens=("fixed", (3000, 700, 64, 65, 1500))), 256),
    "B": (W.small_spec(num_seqs=4, num_heads=16, num_kv_heads=2, dtype=W.F16, block_size=32, seed=32,
                       lens=("fixed", (2049, 1, 513, 4000))), 512),
    # automatic partition size: the plan kernel picks it and zeroes the counters
    "C": (W.small_spec(num_seqs=7, num_heads=32, num_kv_heads=8, dtype=W.BF16, seed=33,
                       lens=("fixed", (5000, 1, 2100, 64, 3333, 700, 129))), 0),
    # more sequences than the plan lists: the full grid, counters cleared by a memset
    "D": (W.small_spec(num_seqs=pkv.PLAN_MAX_SEQS + 77, num_heads=8, num_kv_heads=2, head_dim=64, seed=34,
                       lens=("uniform", 0, 150), pool=("headroom", 0.1)), 64),
}


def test_static_decode_matches_workspace_decode_on_consecutive_calls(lib):
    steps = {}
    for name, (spec, p) in CASES.items():
        wl = W.build(spec)
        step = DeviceStep(wl, partition_tokens=p)
        pkv.paged_kv_append(step.k_new, step.v_new, step.kc[0], step.vc[0], step.slot_mapping)
        step.decode(0)                              # regular entry point, caller workspace
        kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
        steps[name] = (step, p, oracle_attention(wl, kc, vc))
    torch.cuda.synchronize()
    # calls in a row on the shared scratch, each after a different batch left its contents
    for name in ("A", "B", "A", "C", "D", "A", "C"):
        step, p, ref = steps[name]
        got = decode_static(lib, step, p)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert torch.equal(got.view(torch.int16), step.out[0].view(torch.int16)), \
            f"batch {name}: static-scratch decode differs from the workspace decode"
        err = max_abs_err(got, ref)
        assert err <= TOL[step.wl.spec.dtype], f"batch {name}: max abs err {err} against the oracle"
    assert pkv.device_error(reset=True) == 0


def test_static_decode_rejects_batches_beyond_the_scratch(lib):
    # 512 sequences x 64 heads x 64 partitions of fp32 partials is far beyond the built-in scratch;
    # the call must refuse before touching any pointer
    st = lib.pkv_paged_attention_decode_static(None, None, None, None, None, 64, None, 512, 4096, 64, 8, 128, 16,
                                               100000, 0.088, 0, 64, None)
    assert st == pkv.PKV_ERR_WORKSPACE
    assert b"built-in scratch" in lib.pkv_last_error()
