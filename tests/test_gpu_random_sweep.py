"""Randomized GPU parity sweep: seeded random batches against the oracle, through the
separate calls and through one plan plus the fused slot write + decode.

Each case draws a shape (heads, KV heads, head size, block size, dtype), a
batch (sequence count, length distribution with ragged tails and empty
sequences), a partition size and a pool type (16-bit or E4M3), runs one step
(slot writes, then decode) through the C ABI and checks every cache byte and
every output against the oracle.  The draws are fixed by the seed, so a
failure reproduces.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, DeviceStep, max_abs_err, oracle_caches_after_step, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0, "a kernel raised the device error word"


def draw_case(seed):
    rng = np.random.default_rng(9000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 4, 5, 8, 12, 16]))
    d = int(rng.choice([64, 128]))
    fp8 = d == 128 and rng.random() < 0.35
    B = int(rng.integers(1, 40))
    kind = rng.integers(3)
    if kind == 0:
        lens = rng.integers(0, 300, B)
    elif kind == 1:
        lens = np.clip(np.rint(rng.lognormal(np.log(200), 1.3, B)), 1, 3000)
    else:
        lens = rng.integers(1, 5000, B)
    lens[rng.random(B) < 0.1] = 0
    spec = W.small_spec(num_seqs=B, num_heads=hkv * group, num_kv_heads=hkv, head_dim=d,
                        block_size=int(rng.choice([8, 16, 32])), dtype=str(rng.choice([W.F16, W.BF16])),
                        seed=500 + seed, lens=("fixed", tuple(int(x) for x in lens)),
                        pool=("headroom", float(rng.uniform(0.05, 0.5))), kv_dtype=W.E4M3 if fp8 else "")
    part = int(rng.choice([0, 0, 64, 192, 512, 2048]))
    return spec, part


@pytest.mark.parametrize("seed", range(24))
def test_random_batch_matches_oracle(seed):
    spec, part = draw_case(seed)
    wl = W.build(spec)
    s = wl.spec
    if s.fp8:
        dk, dv = (torch.from_numpy(x).cuda() for x in (wl.key_caches[0], wl.value_caches[0]))
        ks, vs = (torch.from_numpy(x).cuda() for x in (wl.k_scales[0], wl.v_scales[0]))
        slots = torch.from_numpy(wl.slot_mapping).cuda()
        pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv, slots, ks, vs)
        q = to_dev(wl.q, s.dtype)
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode_fp8(out, q, dk, dv, torch.from_numpy(wl.block_tables).cuda(),
                                       torch.from_numpy(wl.seq_lens).cuda(), ks, vs, wl.scale,
                                       max_seq_len=wl.max_seq_len, partition_tokens=part)
        torch.cuda.synchronize()
        kc, vc = wl.key_caches[0].copy(), wl.value_caches[0].copy()
        oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, wl.k_scales[0], wl.v_scales[0], s.dtype)
        assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
        ref = oracle.attention_fp8_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                       wl.k_scales[0], wl.v_scales[0])
    else:
        step = DeviceStep(wl, partition_tokens=part)
        step.run()
        torch.cuda.synchronize()
        out = step.out[0]
        kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
        assert np.array_equal(to_bits(step.kc[0]), kc) and np.array_equal(to_bits(step.vc[0]), vc)
        ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    assert torch.isfinite(out).all()
    err = max_abs_err(out, ref)
    assert err <= TOL[s.dtype], f"case {seed} ({s}, partition {part}): max abs err {err}"


@pytest.mark.parametrize("seed", range(24))
def test_random_batch_fused_planned(seed):
    """The same random batches through the benchmark's launches: one plan with the lengths'
    sum, then the slot write fused into the decode (16-bit or E4M3 pools)."""
    spec, part = draw_case(seed)
    wl = W.build(spec)
    s = wl.spec
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    q, k, v = to_dev(wl.q, s.dtype), to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype)
    tables, lens, slots = dev(wl.block_tables), dev(wl.seq_lens), dev(wl.slot_mapping)
    if s.fp8:
        kc, vc = dev(wl.key_caches[0]), dev(wl.value_caches[0])
        ks, vs = dev(wl.k_scales[0]), dev(wl.v_scales[0])
    else:
        kc, vc = to_dev(wl.key_caches[0], s.dtype), to_dev(wl.value_caches[0], s.dtype)
        ks = vs = None
    total = int(wl.seq_lens.sum())
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len, part)
    pkv.decode_plan(ws, tables, lens, s.num_heads, kc, wl.max_seq_len, part, sum_seq_lens=total)
    out = torch.full_like(q, float("nan"))
    pkv.paged_kv_append_decode(out, q, k, v, kc, vc, slots, tables, lens, wl.scale, max_seq_len=wl.max_seq_len,
                               workspace=ws, partition_tokens=part, planned=True, sum_seq_lens=total, k_scale=ks,
                               v_scale=vs)
    torch.cuda.synchronize()
    rk, rv = wl.key_caches[0].copy(), wl.value_caches[0].copy()
    if s.fp8:
        oracle.append_fp8_ref(rk, rv, wl.k_new, wl.v_new, wl.slot_mapping, wl.k_scales[0], wl.v_scales[0], s.dtype)
        assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)
        ref = oracle.attention_fp8_ref(wl.q, rk, rv, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                       wl.k_scales[0], wl.v_scales[0])
    else:
        oracle.append_ref(rk, rv, wl.k_new, wl.v_new, wl.slot_mapping)
        assert np.array_equal(to_bits(kc), rk) and np.array_equal(to_bits(vc), rv)
        ref = oracle.attention_ref(wl.q, rk, rv, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype)
    assert torch.isfinite(out).all()
    err = max_abs_err(out, ref)
    assert err <= TOL[s.dtype], f"case {seed} ({s}, partition {part}): max abs err {err}"
