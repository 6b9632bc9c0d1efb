"""GPU parity of the shared-prefix decode: forked sequences served as units.

The plan kernel compares the block-table rows of adjacent sequences whose
first blocks agree (forks of one prompt, "LLM 推理引擎内部原理" §3.3) and, with
at most 4 query heads per KV head over 16-bit pools, serves up to 8 / G of
them in one CTA per KV head: the shared blocks once, then each member's own
blocks.  Every output must still be the oracle's attention of each sequence
over its own blocks (within tolerance), every cache byte the oracle's, for
fork batches of every block size and GQA ratio, explicit and automatic
partitions, through the separate calls and through the benchmark's launches
(one plan, then the slot write fused into the decode); and for hand-built
tables: members that share a partly filled block, a member whose length ends
inside the shared run, runs too short to share, units of 8.  The work list is
read back to check that units formed where they should and not elsewhere.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W
from gpu_harness import TOL, DeviceStep, max_abs_err, oracle_attention, oracle_caches_after_step, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.device_error(reset=True)
    yield
    assert pkv.device_error(reset=True) == 0, "a kernel raised the device error word"


def work_list(ws, num_seqs, num_heads, num_kv_heads):
    """Live entries of the plan in `ws`: (first sequence, partition, stream length,
    partition size, members, shared length).  Reads the workspace's layout: merge
    counters (one u32 per sequence and KV head group, padded to 256 bytes), then
    entries of eight int32."""
    group = num_heads // num_kv_heads
    nh = num_kv_heads * ((group + 7) // 8)
    off = (4 * num_seqs * nh + 255) // 256 * 256
    e = ws[off:].view(torch.int32).cpu().numpy()
    e = e[:8 * (e.size // 8)].reshape(-1, 8)
    out = []
    for r in e:                                     # live entries come first, then padding (sequence -1)
        if r[0] < 0 or r[4] < 1 or r[4] > 8 or (out and r[3] != out[0][3]):
            break
        out.append(tuple(int(x) for x in r[:6]))
    return out


def units_of(entries):
    """{first sequence: (members, shared length)} of the multi-sequence units."""
    return {r[0]: (r[4], r[5]) for r in entries if r[4] > 1}


def check_step(wl, step):
    kc, vc = oracle_caches_after_step(wl, wl.key_caches[0], wl.value_caches[0])
    assert np.array_equal(to_bits(step.kc[0]), kc) and np.array_equal(to_bits(step.vc[0]), vc)
    ref = oracle_attention(wl, kc, vc)
    assert torch.isfinite(step.out[0]).all()
    err = max_abs_err(step.out[0], ref)
    assert err <= TOL[wl.spec.dtype], f"max abs err {err}"
    return err


FORKS = [
    # (query heads, KV heads, block size, dtype, (requests, forks, prefix, suffix lo, suffix hi))
    (8, 2, 16, W.F16, (3, 3, 300, 0, 80)),       # G 4: units of 2 (+ 1), partly filled prefix block copied
    (32, 8, 8, W.F16, (4, 3, 1024, 0, 512)),     # the fork workload's shape, fewer requests
    (8, 4, 32, W.BF16, (3, 5, 640, 1, 200)),     # G 2: units of 4 (+ 1)
    (4, 4, 16, W.BF16, (2, 8, 520, 0, 300)),     # G 1: one unit of 8
    (16, 2, 16, W.F16, (2, 3, 700, 5, 60)),      # G 8: no units (the heads fill the CTA)
    (8, 2, 8, W.BF16, (2, 4, 257, 0, 3)),        # a prefix just above the sharing threshold, tiny suffixes
]


@pytest.mark.parametrize("partition_tokens", [0, 64, 256, 4096])
@pytest.mark.parametrize("case", range(len(FORKS)))
def test_fork_batch_matches_oracle(case, partition_tokens):
    hq, hkv, bs, dt, fork = FORKS[case]
    spec = W.small_spec(num_seqs=fork[0] * fork[1], num_heads=hq, num_kv_heads=hkv, block_size=bs, dtype=dt,
                        seed=1100 + case, lens=("fork",), fork=fork)
    wl = W.build(spec)
    step = DeviceStep(wl, partition_tokens=partition_tokens)
    step.run()
    torch.cuda.synchronize()
    check_step(wl, step)
    units = units_of(work_list(step.workspace, spec.num_seqs, hq, hkv))
    if hq // hkv > 4:
        assert not units, "no units when a sequence's heads fill the CTA"
    elif partition_tokens in (0, 4096):
        assert units, "forks that share their prefix must form units"
        for s0, (n, sh) in units.items():
            assert 2 <= n <= 8 // (hq // hkv) and sh >= 256
            # members are forks of the same request: the same first block
            assert len({int(wl.block_tables[s0 + j, 0]) for j in range(n)}) == 1


@pytest.mark.parametrize("partition_tokens", [0, 128])
@pytest.mark.parametrize("case", [0, 1, 3])
def test_fork_batch_fused_planned(case, partition_tokens):
    """The benchmark's launches: one plan (lengths' sum given), then the fused slot write +
    decode over it, twice (the plan serves every run)."""
    hq, hkv, bs, dt, fork = FORKS[case]
    fork = (fork[0], fork[1], (fork[2] // bs) * bs, fork[3], fork[4])   # whole prefix blocks: one slot per sequence
    spec = W.small_spec(num_seqs=fork[0] * fork[1], num_heads=hq, num_kv_heads=hkv, block_size=bs, dtype=dt,
                        seed=1200 + case, lens=("fork",), fork=fork)
    wl = W.build(spec)
    assert wl.num_tokens == spec.num_seqs
    step = DeviceStep(wl, partition_tokens=partition_tokens)
    step.run_planned_fused()
    first = step.out[0].clone()
    check_step(wl, step)
    assert units_of(work_list(step.workspace, spec.num_seqs, hq, hkv)), "forks must form units"
    # the same plan runs again over the step's result (the slot writes repeat the same bytes)
    pkv.paged_attention_decode(step.out[0], step.q, step.kc[0], step.vc[0], step.block_tables, step.seq_lens,
                               wl.scale, max_seq_len=wl.max_seq_len, workspace=step.workspace,
                               partition_tokens=partition_tokens, planned=True, sum_seq_lens=int(wl.seq_lens.sum()))
    torch.cuda.synchronize()
    assert torch.equal(first, step.out[0]), "a planned run must repeat bit for bit"


# ---------------------------------------------------------------- hand-built tables
def manual(tables, lens, appends, NB, bs=16, hq=8, hkv=2, d=128, dt=W.F16, seed=0):
    """A one-layer batch with the given block tables and lengths; `appends[s]`: sequence s
    writes its newest token (position L - 1) in this step.  Slots that hold no token
    before the step are NaN."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    width = max(len(t) for t in tables)
    bt = np.full((B, width), NB + 7, np.int64)
    bt[:, 1::2] = W.INT32_MAX
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    valid = np.zeros((NB, bs), bool)
    slots = []
    for t, L, ap in zip(tables, lens, appends):
        for p in range(L - (1 if ap else 0)):
            valid[t[p // bs], p % bs] = True
        slots.append(t[(L - 1) // bs] * bs + (L - 1) % bs if ap else -1)
    spec = W.small_spec(num_seqs=B, num_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=dt,
                        seed=seed, lens=("fixed", tuple(lens)))
    kc = W.normal_bits(rng, (NB, bs, hkv, d), dt)
    vc = W.normal_bits(rng, (NB, bs, hkv, d), dt)
    kc[~valid] = W.NAN_BITS[dt]
    vc[~valid] = W.NAN_BITS[dt]
    wl = W.Workload(spec=spec, num_blocks=NB, seq_lens=np.asarray(lens, np.int32), block_tables=bt.astype(np.int32),
                    q=W.normal_bits(rng, (B, hq, d), dt), k_new=W.normal_bits(rng, (B, hkv, d), dt),
                    v_new=W.normal_bits(rng, (B, hkv, d), dt), slot_mapping=np.asarray(slots, np.int64),
                    copy_pairs=np.zeros((0, 2), np.int64), valid_slots=valid)
    wl.key_caches, wl.value_caches = [kc], [vc]
    return wl


def permuted_blocks(n, NB, seed):
    return [int(b) for b in np.random.default_rng(seed).permutation(NB)[:n]]


def test_members_sharing_a_partly_filled_block():
    """Three sequences hold the same 19 blocks and 300 positions (the last block partly
    filled); none appends: the unit's stream is the shared prefix alone."""
    t = permuted_blocks(19, 40, 1)
    wl = manual([t, t, t], [300, 300, 300], [False] * 3, NB=40)
    for p in (0, 64):
        step = DeviceStep(wl, partition_tokens=p)
        step.run()
        torch.cuda.synchronize()
        check_step(wl, step)
        assert units_of(work_list(step.workspace, 3, 8, 2)) == {0: (2, 300)}


def test_member_ending_inside_the_shared_run():
    """A (1000 positions, 63 blocks) and B (1500 positions) share A's 63 blocks, A's last
    one partly filled (B holds its own positions 1000..1007 in the rest of it): the shared
    length is 1000, B's own segment starts inside that block."""
    blocks = permuted_blocks(94, 120, 2)
    A, Bt = blocks[:63], blocks[:63] + blocks[63:94]
    for appends in ([False, True], [False, False]):
        wl = manual([A, Bt], [1000, 1500], appends, NB=120, seed=3)
        for p in (0, 64, 1024):
            step = DeviceStep(wl, partition_tokens=p)
            step.run()
            torch.cuda.synchronize()
            check_step(wl, step)
            got = units_of(work_list(step.workspace, 2, 8, 2))
            if p == 0:
                assert got == {0: (2, 1000)}


def test_short_shared_runs_stay_separate():
    """Sharing fewer than 256 positions does not form a unit."""
    blocks = permuted_blocks(60, 80, 4)
    A = blocks[:10] + blocks[10:30]             # 10 shared blocks of 16: 160 positions
    Bt = blocks[:10] + blocks[30:55]
    wl = manual([A, Bt], [470, 395], [True, True], NB=80, seed=5)
    step = DeviceStep(wl)
    step.run()
    torch.cuda.synchronize()
    check_step(wl, step)
    assert not units_of(work_list(step.workspace, 2, 8, 2))


def test_fused_write_into_the_shared_prefix_is_refused():
    """A fused slot write whose position lies in the shared blocks would change what the
    other members read: it is refused (nothing written, bounds bit raised)."""
    t = permuted_blocks(19, 40, 6)
    wl = manual([t, t], [300, 300], [True, False], NB=40, seed=7)
    step = DeviceStep(wl)
    before = to_bits(step.kc[0])
    total = int(wl.seq_lens.sum())
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, 8, step.kc[0], wl.max_seq_len, 0,
                    sum_seq_lens=total)
    pkv.paged_kv_append_decode(step.out[0], step.q, step.k_new, step.v_new, step.kc[0], step.vc[0],
                               step.slot_mapping, step.block_tables, step.seq_lens, wl.scale,
                               max_seq_len=wl.max_seq_len, workspace=step.workspace, planned=True,
                               sum_seq_lens=total)
    torch.cuda.synchronize()
    assert pkv.device_error(reset=True) & 1, "a fused write into a shared block must raise the bounds bit"
    assert np.array_equal(to_bits(step.kc[0]), before), "nothing may be written"


def test_units_across_layers_of_a_planned_step():
    """One plan with units, three layers: each planned run equals the single call on its
    layer bit for bit and the oracle within tolerance."""
    spec = W.small_spec(num_seqs=6, num_heads=8, num_kv_heads=2, block_size=16, dtype=W.BF16, seed=1300,
                        lens=("fork",), fork=(2, 3, 512, 0, 100), num_layers=3)
    wl = W.build(spec)
    step = DeviceStep(wl)
    pkv.copy_blocks(step.kc, step.vc, step.copy_pairs)
    total = int(wl.seq_lens.sum())
    pkv.decode_plan(step.workspace, step.block_tables, step.seq_lens, 8, step.kc[0], wl.max_seq_len, 0,
                    sum_seq_lens=total)
    assert units_of(work_list(step.workspace, 6, 8, 2))
    planned = []
    for l in range(3):
        pkv.paged_kv_append(step.k_new, step.v_new, step.kc[l], step.vc[l], step.slot_mapping)
        out = torch.empty_like(step.q)
        pkv.paged_attention_decode(out, step.q, step.kc[l], step.vc[l], step.block_tables, step.seq_lens, wl.scale,
                                   max_seq_len=wl.max_seq_len, workspace=step.workspace, planned=True,
                                   sum_seq_lens=total)
        planned.append(out)
    for l in range(3):
        step.decode(l)
    torch.cuda.synchronize()
    for l in range(3):
        assert torch.equal(planned[l], step.out[l]), f"layer {l}"
        kc, vc = oracle_caches_after_step(wl, wl.key_caches[l], wl.value_caches[l])
        ref = oracle.attention_ref(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.scale, 2, W.BF16)
        assert max_abs_err(planned[l], ref) <= TOL[W.BF16]
