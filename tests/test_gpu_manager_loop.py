"""A small serving loop driven by the native block manager, on the GPU.

The manager hands out blocks and slots, a fork shares a prompt, each decode
step appends one token per sequence (copy-on-write copies first), writes the
new K/V and attends; a sequence finishes and a new one arrives midway.  The
device pools must equal the oracle's bit for bit after every step and every
attention output must be within the fp16 tolerance of the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, to_bits, to_dev

pytestmark = pytest.mark.gpu


def test_manager_driven_decode_loop():
    rng = np.random.default_rng(77)
    NB, bs, Hq, Hkv, d = 96, 16, 16, 4, 128
    dt = W.F16
    bm = pkv.BlockManager(NB, bs, free_order=rng.permutation(NB))
    kc = np.full((NB, bs, Hkv, d), W.NAN_BITS[dt], np.uint16)
    vc = kc.copy()
    dk, dv = to_dev(kc, dt), to_dev(vc, dt)

    def write_tokens(seq_slots):
        slots = np.asarray(seq_slots, dtype=np.int64)
        k = W.normal_bits(rng, (len(slots), Hkv, d), dt)
        v = W.normal_bits(rng, (len(slots), Hkv, d), dt)
        oracle.append_ref(kc, vc, k, v, slots)
        pkv.paged_kv_append(to_dev(k, dt), to_dev(v, dt), dk, dv, torch.from_numpy(slots).cuda())

    def prompt(seq_id, L):
        bm.allocate(seq_id, L)
        t, _ = bm.block_tables([seq_id], max(1, -(-L // bs)))
        write_tokens([oracle.slot_for_position(t[0], p, bs) for p in range(L)])

    prompt(0, 37)
    prompt(1, 16)
    prompt(2, 70)
    bm.fork(0, 10)
    bm.fork(0, 11)
    live = [0, 1, 2, 10, 11]
    scale = 1.0 / np.sqrt(d)
    for step in range(6):
        if step == 3:
            bm.free(1)
            live.remove(1)
            prompt(20, 5)
            live.append(20)
        slots, cow = bm.append_slots(live)
        if len(cow):
            oracle.copy_blocks_ref([kc], [vc], cow)
            pkv.copy_blocks([dk], [dv], torch.from_numpy(cow).cuda())
        write_tokens(slots)
        Wd = max(-(-bm.seq_len(s) // bs) for s in live)
        tables, lens = bm.block_tables(live, Wd, pad=NB + 7)
        q = W.normal_bits(rng, (len(live), Hq, d), dt)
        out = torch.empty((len(live), Hq, d), dtype=torch.float16, device="cuda")
        pkv.paged_attention_decode(out, to_dev(q, dt), dk, dv, torch.from_numpy(tables).cuda(),
                                   torch.from_numpy(lens).cuda(), scale, max_seq_len=int(lens.max()),
                                   partition_tokens=64)
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(dk), kc) and np.array_equal(to_bits(dv), vc), f"pools differ at step {step}"
        ref = oracle.attention_ref(q, kc, vc, tables, lens, scale, Hkv, dt)
        err = float(np.abs(out.float().cpu().numpy() - ref).max())
        assert err <= TOL[dt], f"step {step}: {err}"
    assert pkv.device_error(reset=True) == 0
    # the fork's copy-on-write happened exactly once per child
    assert bm.refcount(int(tables[0, 0])) == 3 and bm.seq_len(10) == 37 + 6
