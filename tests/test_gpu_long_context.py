"""GPU parity at long context: one sequence of 64K or 128K positions beside short ones.

Long sequences are why the pages page the KV cache at all ("tbr8.org PagedAttention
article" §一: the cache of one 4096-token sequence already runs to gigabytes at 80
layers; "vLLM核心概念" §4.2: blocks are allocated as the sequence grows).  Here one
sequence's blocks span a table of 4K to 8K entries, its partitions number 16 to 256
(the merge of many partials, not only the single-pass form for up to four), and a
one-position sequence shares the batch.  Every output is compared with the oracle,
through the separate calls and through the benchmark's planned, fused launch.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import (TOL, DeviceStep, max_abs_err, mean_abs_err, oracle_attention, oracle_caches_after_step,
                         to_bits)

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
