"""GPU parity of the 8-bit (E4M3) KV cache calls against the oracle.

The quantizing append must match the oracle's codes bit for bit (both
divide by the scale in float32 and round to nearest even with saturation);
the decode over E4M3 pools must be within the query dtype's tolerance of the
oracle's float64 attention over the dequantized K/V.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, max_abs_err, mean_abs_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0, "a kernel raised the device error word"


def cuda_of(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_append_fp8_bit_exact(dtype):
    rng = np.random.default_rng(61)
    NB, bs, H, d, T = 12, 16, 4, 128, 37
    kc = np.full((NB, bs, H, d), W.E4M3_NAN, np.uint8)
    vc = kc.copy()
    x = rng.standard_normal((T, H, d)).astype(np.float32) * rng.choice([1e-4, 0.1, 1.0, 30.0, 300.0], (T, 1, 1))
    x[0, 0, :6] = [0.0, -0.0, np.inf, -np.inf, 1e30, -1e-30]
    k = W.f32_to_bits(x, dtype)
    v = W.f32_to_bits(-0.5 * x, dtype)
    slots = rng.choice(NB * bs, T, replace=False).astype(np.int64)
    slots[5] = -1
    ks = rng.uniform(0.01, 2.0, H).astype(np.float32)
    vs = rng.uniform(0.01, 2.0, H).astype(np.float32)
    dk, dv = cuda_of(kc), cuda_of(vc)
    pkv.paged_kv_append_fp8(to_dev(k, dtype), to_dev(v, dtype), dk, dv, cuda_of(slots), f32(ks), f32(vs))
    torch.cuda.synchronize()
    oracle.append_fp8_ref(kc, vc, k, v, slots, ks, vs, dtype)
    assert np.array_equal(dk.cpu().numpy(), kc)
    assert np.array_equal(dv.cpu().numpy(), vc)


CASES = [
    dict(num_heads=32, num_kv_heads=8, block_size=16, dtype=W.BF16, lens=("fixed", (1, 15, 16, 17, 64, 65, 1000, 2049))),
    dict(num_heads=64, num_kv_heads=8, block_size=8, dtype=W.F16, lens=("fixed", (300, 4096, 7, 129))),
    dict(num_heads=8, num_kv_heads=1, block_size=32, dtype=W.BF16, lens=("fixed", (0, 33, 700))),
    dict(num_heads=16, num_kv_heads=4, block_size=16, dtype=W.F16, lens=("uniform", 1, 900)),
]


@pytest.mark.parametrize("partition_tokens", [0, 64, 1024])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_fp8_step_matches_oracle(case, partition_tokens):
    kw = dict(CASES[case])
    kw["num_seqs"] = len(kw["lens"][1]) if kw["lens"][0] == "fixed" else 20
    wl = W.build(W.small_spec(seed=620 + case, head_dim=128, kv_dtype=W.E4M3, **kw))
    s = wl.spec
    dk, dv = cuda_of(wl.key_caches[0]), cuda_of(wl.value_caches[0])
    ks, vs = wl.k_scales[0], wl.v_scales[0]
    pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv, cuda_of(wl.slot_mapping),
                            f32(ks), f32(vs))
    q = to_dev(wl.q, s.dtype)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_fp8(out, q, dk, dv, cuda_of(wl.block_tables), cuda_of(wl.seq_lens), f32(ks), f32(vs), wl.scale,
                                   max_seq_len=wl.max_seq_len, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    kc, vc = wl.key_caches[0].copy(), wl.value_caches[0].copy()
    oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, ks, vs, s.dtype)
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    ref = oracle.attention_fp8_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                   ks, vs)
    assert torch.isfinite(out).all()
    err = max_abs_err(out, ref)
    assert err <= TOL[s.dtype], f"max abs err {err}"


def test_full_size_fp8_workload():
    wl = W.build(W.SPECS["llama3_8b_fp8"], values="none")
    s = wl.spec
    dk, dv = W.device_pools(wl, 0, "cuda")
    kc, vc = dk.cpu().numpy().copy(), dv.cpu().numpy().copy()     # the generator's pools, before the step
    ks, vs = wl.k_scales[0], wl.v_scales[0]
    pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv, cuda_of(wl.slot_mapping),
                            f32(ks), f32(vs))
    q = to_dev(wl.q, s.dtype)
    out = torch.empty_like(q)
    pkv.paged_attention_decode_fp8(out, q, dk, dv, cuda_of(wl.block_tables), cuda_of(wl.seq_lens), f32(ks), f32(vs), wl.scale,
                                   max_seq_len=wl.max_seq_len)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, ks, vs, s.dtype)
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    ref = oracle.attention_fp8_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                   ks, vs)                 # every sequence, every head
    err = max_abs_err(out, ref)
    print(f"llama3_8b_fp8: max abs err {err:.3g}, mean {mean_abs_err(out, ref):.3g} over all {s.num_seqs} sequences x "
          f"{s.num_heads} heads")
    assert err <= TOL[s.dtype], f"max abs err {err}"


def test_copy_and_swap_fp8_pools_bit_exact():
    rng = np.random.default_rng(63)
    NB, bs, H, d = 20, 16, 8, 128
    kc = W.random_e4m3_codes(rng, (NB, bs, H, d))
    vc = W.random_e4m3_codes(rng, (NB, bs, H, d))
    dk, dv = cuda_of(kc), cuda_of(vc)
    pairs = np.array([[1, 7], [3, 9], [4, 0]], np.int64)
    pkv.copy_blocks([dk], [dv], cuda_of(pairs))
    host_k = torch.zeros((5, bs, H, d), dtype=torch.uint8, pin_memory=True)
    host_v = torch.zeros_like(host_k, pin_memory=True)
    out_pairs = np.array([[2, 0], [11, 4]], np.int64)
    pkv.swap_blocks([dk], [dv], [host_k], [host_v], cuda_of(out_pairs))
    torch.cuda.synchronize()
    oracle.copy_blocks_ref([kc], [vc], pairs)
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    hk = np.zeros((5, bs, H, d), np.uint8)
    hv = hk.copy()
    oracle.swap_blocks_ref([kc], [vc], [hk], [hv], out_pairs)
    assert np.array_equal(host_k.numpy(), hk) and np.array_equal(host_v.numpy(), hv)


def test_fp8_host_validation():
    k8 = torch.zeros((4, 16, 2, 64), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 4, 64), dtype=torch.float16, device="cuda")
    one = torch.ones(2, dtype=torch.float32, device="cuda")
    tab = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:                 # head_dim 64: not built for E4M3 pools
        pkv.paged_attention_decode_fp8(torch.empty_like(q), q, k8, k8, tab, lens, one, one, max_seq_len=1)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    with pytest.raises(ValueError):                        # one scale per KV head
        pkv.paged_attention_decode_fp8(torch.empty_like(q), q, k8, k8, tab, lens, one[:1], one, max_seq_len=1)


VERIFY_CASES = [
    dict(num_heads=32, num_kv_heads=8, block_size=16, dtype=W.BF16, nq=4, lens=("fixed", (4, 70, 1025, 300, 2))),
    dict(num_heads=64, num_kv_heads=8, block_size=8, dtype=W.F16, nq=2, lens=("fixed", (2, 900, 129, 0))),
    dict(num_heads=16, num_kv_heads=2, block_size=32, dtype=W.BF16, nq=5, lens=("fixed", (5, 3000, 64, 65))),
    dict(num_heads=8, num_kv_heads=1, block_size=16, dtype=W.F16, nq=3, lens=("uniform", 3, 1500)),
]


@pytest.mark.parametrize("partition_tokens", [0, 64, 1024])
@pytest.mark.parametrize("case", range(len(VERIFY_CASES)))
def test_verify_fp8_matches_oracle(case, partition_tokens):
    """Several causal query tokens per sequence over E4M3 pools (rows per KV head from 4 to 40:
    one and several 8-row groups); the last nq positions are the queries' own, appended first."""
    kw = dict(VERIFY_CASES[case])
    nq = kw.pop("nq")
    kw["num_seqs"] = len(kw["lens"][1]) if kw["lens"][0] == "fixed" else 12
    wl = W.build(W.small_spec(seed=840 + case, head_dim=128, kv_dtype=W.E4M3, **kw))
    s = wl.spec
    dk, dv = cuda_of(wl.key_caches[0]), cuda_of(wl.value_caches[0])
    ks, vs = wl.k_scales[0], wl.v_scales[0]
    pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv, cuda_of(wl.slot_mapping),
                            f32(ks), f32(vs))
    rng = np.random.default_rng(850 + case)
    q = W.normal_bits(rng, (s.num_seqs, nq, s.num_heads, s.head_dim), s.dtype)
    qd = to_dev(q, s.dtype)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_attention_verify(out, qd, dk, dv, cuda_of(wl.block_tables), cuda_of(wl.seq_lens), wl.scale,
                               max_seq_len=wl.max_seq_len, partition_tokens=partition_tokens,
                               sum_seq_lens=int(wl.seq_lens.sum()), k_scale=f32(ks), v_scale=f32(vs))
    torch.cuda.synchronize()
    kc, vc = wl.key_caches[0].copy(), wl.value_caches[0].copy()
    oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, ks, vs, s.dtype)
    ref = oracle.verify_attention_fp8_ref(q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                          ks, vs)
    assert torch.isfinite(out).all()
    err = max_abs_err(out, ref)
    assert err <= TOL[s.dtype], f"max abs err {err}"


@pytest.mark.parametrize("nq", [4, 8])
def test_full_size_verify_fp8(nq):
    """The benchmarked E4M3 verify launches (the 8B-shaped batch, 16 and 32 rows per KV head, the
    benchmark's workspace and lengths' sum): every output of every sequence against the oracle."""
    wl = W.build(W.SPECS["llama3_8b_fp8"], values="none")
    s = wl.spec
    assert int(wl.seq_lens.min()) >= nq
    dk, dv = W.device_pools(wl, 0, "cuda")
    kc, vc = dk.cpu().numpy().copy(), dv.cpu().numpy().copy()     # the generator's pools, before the step
    ks, vs = wl.k_scales[0], wl.v_scales[0]
    pkv.paged_kv_append_fp8(to_dev(wl.k_new, s.dtype), to_dev(wl.v_new, s.dtype), dk, dv, cuda_of(wl.slot_mapping),
                            f32(ks), f32(vs))
    rng = np.random.default_rng(950 + nq)
    q = W.normal_bits(rng, (s.num_seqs, nq, s.num_heads, s.head_dim), s.dtype)
    qd = to_dev(q, s.dtype)
    out = torch.full_like(qd, float("nan"))
    ws = pkv.alloc_workspace(s.num_seqs, s.num_heads * nq, s.num_kv_heads, s.head_dim, wl.max_seq_len, 0, "cuda")
    pkv.paged_attention_verify(out, qd, dk, dv, cuda_of(wl.block_tables), cuda_of(wl.seq_lens), wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=ws, sum_seq_lens=int(wl.seq_lens.sum()),
                               k_scale=f32(ks), v_scale=f32(vs))
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    oracle.append_fp8_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping, ks, vs, s.dtype)
    ref = oracle.verify_attention_fp8_ref(q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, s.num_kv_heads, s.dtype,
                                          ks, vs)
    err = max_abs_err(out, ref)
    print(f"llama3_8b_fp8 verify nq={nq}: max abs err {err:.3g}, mean {mean_abs_err(out, ref):.3g} over all "
          f"{s.num_seqs} sequences x {nq} queries x "
          f"{s.num_heads} heads")
    assert err <= TOL[s.dtype], f"max abs err {err}"


def test_verify_fp8_one_query_is_the_decode_call():
    wl = W.build(W.small_spec(num_seqs=5, num_heads=32, num_kv_heads=8, head_dim=128, dtype=W.BF16, seed=860,
                              kv_dtype=W.E4M3, lens=("fixed", (900, 33, 2049, 1, 4000))))
    s = wl.spec
    dk, dv = cuda_of(wl.key_caches[0]), cuda_of(wl.value_caches[0])
    ks, vs = f32(wl.k_scales[0]), f32(wl.v_scales[0])
    q = to_dev(wl.q, s.dtype)
    tab, lens = cuda_of(wl.block_tables), cuda_of(wl.seq_lens)
    a = torch.empty_like(q)
    pkv.paged_attention_decode_fp8(a, q, dk, dv, tab, lens, ks, vs, wl.scale, max_seq_len=wl.max_seq_len,
                                   partition_tokens=256)
    b = torch.empty_like(q).unsqueeze(1)
    pkv.paged_attention_verify(b, q.unsqueeze(1).contiguous(), dk, dv, tab, lens, wl.scale,
                               max_seq_len=wl.max_seq_len, partition_tokens=256, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b[:, 0].view(torch.int16))
