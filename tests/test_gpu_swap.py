"""GPU parity of swap_blocks (preemption by swapping) against the oracle.

Swap-out copies blocks from device pools into pinned host pools, swap-in
copies them back under new block ids; both must match the oracle bit for bit,
and a decode over the swapped-in blocks (table rewritten to the new ids) must
give the same output, bit for bit, as the decode before the swap.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import DeviceStep, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0


def pinned_like(shape, dtype, fill_bits):
    t = torch.empty(shape, dtype=torch.int16, pin_memory=True)
    t.fill_(np.int16(np.uint16(fill_bits).view(np.int16)))
    return t.view(dtype)


@pytest.mark.parametrize("layers", [1, 3])
def test_swap_out_and_in_bit_exact(layers):
    rng = np.random.default_rng(40 + layers)
    NB, NH_host, bs, H, d = 50, 24, 16, 8, 128
    dt = W.BF16
    tdt = torch.bfloat16
    kcs = [W.normal_bits(rng, (NB, bs, H, d), dt) for _ in range(layers)]
    vcs = [W.normal_bits(rng, (NB, bs, H, d), dt) for _ in range(layers)]
    dk = [to_dev(x, dt) for x in kcs]
    dv = [to_dev(x, dt) for x in vcs]
    hk = [pinned_like((NH_host, bs, H, d), tdt, W.NAN_BITS[dt]) for _ in range(layers)]
    hv = [pinned_like((NH_host, bs, H, d), tdt, W.NAN_BITS[dt]) for _ in range(layers)]
    out_pairs = np.stack([rng.choice(NB, 20, replace=False), rng.choice(NH_host, 20, replace=False)], 1)
    pkv.swap_blocks(dk, dv, hk, hv, torch.from_numpy(out_pairs).cuda())
    torch.cuda.synchronize()
    ref_hk = [np.full((NH_host, bs, H, d), W.NAN_BITS[dt], np.uint16) for _ in range(layers)]
    ref_hv = [np.full((NH_host, bs, H, d), W.NAN_BITS[dt], np.uint16) for _ in range(layers)]
    oracle.swap_blocks_ref(kcs, vcs, ref_hk, ref_hv, out_pairs)
    for l in range(layers):
        assert np.array_equal(hk[l].view(torch.int16).numpy().view(np.uint16), ref_hk[l])
        assert np.array_equal(hv[l].view(torch.int16).numpy().view(np.uint16), ref_hv[l])
    # swap back in under new ids into a fresh device pool
    in_pairs = np.stack([out_pairs[:, 1], rng.choice(NB, 20, replace=False)], 1)
    dk2 = [to_dev(np.full((NB, bs, H, d), W.NAN_BITS[dt], np.uint16), dt) for _ in range(layers)]
    dv2 = [to_dev(np.full((NB, bs, H, d), W.NAN_BITS[dt], np.uint16), dt) for _ in range(layers)]
    pkv.swap_blocks(hk, hv, dk2, dv2, torch.from_numpy(in_pairs).cuda())
    torch.cuda.synchronize()
    ref_k2 = [np.full((NB, bs, H, d), W.NAN_BITS[dt], np.uint16) for _ in range(layers)]
    ref_v2 = [np.full((NB, bs, H, d), W.NAN_BITS[dt], np.uint16) for _ in range(layers)]
    oracle.swap_blocks_ref(ref_hk, ref_hv, ref_k2, ref_v2, in_pairs)
    for l in range(layers):
        assert np.array_equal(to_bits(dk2[l]), ref_k2[l]) and np.array_equal(to_bits(dv2[l]), ref_v2[l])


def test_decode_is_unchanged_by_a_swap_round_trip():
    """Preempt every sequence (swap all its blocks out), resume it under new ids."""
    wl = W.build(W.small_spec(num_seqs=4, num_heads=32, num_kv_heads=8, dtype=W.F16,
                              lens=("fixed", (700, 33, 1500, 64)), pool=("headroom", 1.2)))
    step = DeviceStep(wl, partition_tokens=256)
    step.run()
    before = step.out[0].clone()
    bs = wl.spec.block_size
    used = []
    for s in range(wl.spec.num_seqs):
        used.extend(wl.block_tables[s, :oracle.num_logical_blocks(int(wl.seq_lens[s]), bs)].tolist())
    used = np.array(used, dtype=np.int64)
    host_k = torch.empty((len(used),) + tuple(step.kc[0].shape[1:]), dtype=torch.float16, pin_memory=True)
    host_v = torch.empty_like(host_k, pin_memory=True)
    pkv.swap_blocks(step.kc, step.vc, [host_k], [host_v],
                    torch.from_numpy(np.stack([used, np.arange(len(used))], 1)).cuda())
    # resume into different physical blocks of a poisoned pool
    free = np.setdiff1d(np.arange(wl.num_blocks), used)
    rng = np.random.default_rng(5)
    new_ids = rng.permutation(np.concatenate([free, used]))[:len(used)]
    step.kc[0].view(torch.int16).fill_(np.int16(0x7E00))
    step.vc[0].view(torch.int16).fill_(np.int16(0x7E00))
    pkv.swap_blocks([host_k], [host_v], step.kc, step.vc,
                    torch.from_numpy(np.stack([np.arange(len(used)), new_ids], 1)).cuda())
    remap = dict(zip(used.tolist(), new_ids.tolist()))
    tables = wl.block_tables.copy()
    for s in range(wl.spec.num_seqs):
        for j in range(oracle.num_logical_blocks(int(wl.seq_lens[s]), bs)):
            tables[s, j] = remap[int(tables[s, j])]
    step.block_tables = torch.from_numpy(tables).cuda()
    step.decode(0)
    torch.cuda.synchronize()
    assert torch.equal(step.out[0], before)


def test_swap_rejects_unpinned_host_memory():
    t = torch.zeros(4, 16, 2, 64, dtype=torch.float16)
    d = torch.zeros(4, 16, 2, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        pkv.swap_blocks([d], [d], [t], [t], torch.zeros(1, 2, dtype=torch.int64, device="cuda"))
