"""The native host block manager (pkv_bm_*) against the pages and the oracle.

No GPU: the manager is host code in the library.  Pins follow the pages'
worked behaviour; a randomized differential test drives the C++ manager and
the oracle's plain reference through the same operations.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_156_gb300 as pkv
from paged_kv_cache_156_gb300 import _build


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def test_allocate_ceil_blocks_and_fifo_order():
    bm = pkv.BlockManager(300, 16)
    bm.allocate(0, 50)                       # P4 §3: 50 tokens -> 4 blocks of 16
    bm.allocate(1, 4096)                     # 4096 -> 256
    t, L = bm.block_tables([0, 1], 256)
    assert t[0, :4].tolist() == [0, 1, 2, 3] and (t[0, 4:] == -1).all() and L.tolist() == [50, 4096]
    assert t[1].tolist() == list(range(4, 260))
    bm.free(0)                               # freed blocks go to the back of the list (P2 §2.3)
    bm.allocate(2, 40 * 16)
    t2, _ = bm.block_tables([2], 40)
    assert t2[0].tolist() == list(range(260, 300)) and bm.num_free_blocks == 4
    bm.allocate(3, 1)
    assert bm.block_tables([3], 1)[0][0, 0] == 0


def test_append_slot_matches_pages_arithmetic():
    bm = pkv.BlockManager(8, 16)
    bm.allocate(7, 20)                       # blocks 0, 1; next position 20 -> block 1 offset 4
    slots, cow = bm.append_slots([7])
    assert slots.tolist() == [1 * 16 + 4] and len(cow) == 0
    for _ in range(11):
        bm.append_slots([7])                 # fill to 32 tokens
    slots, _ = bm.append_slots([7])          # 32 % 16 == 0: a new block, offset 0
    assert slots.tolist() == [2 * 16] and bm.seq_len(7) == 33


def test_oom_changes_nothing():
    bm = pkv.BlockManager(4, 8)
    bm.allocate(0, 24)                       # 3 blocks
    bm.allocate(1, 8)                        # 1 block: pool empty
    with pytest.raises(pkv.PkvError) as e:
        bm.append_slots([0, 1])              # both need a new block
    assert e.value.status == pkv.PKV_ERR_OOM
    assert bm.seq_len(0) == 24 and bm.seq_len(1) == 8 and bm.num_free_blocks == 0
    with pytest.raises(pkv.PkvError):
        bm.allocate(2, 1)
    bm.free(1)
    slots, _ = bm.append_slots([0])
    assert slots.tolist() == [3 * 8]


def test_fork_shares_then_copies_on_write():
    bm = pkv.BlockManager(16, 16)
    bm.allocate(0, 40)                       # blocks 0,1,2 ; block 2 holds 8 tokens
    bm.fork(0, 1)
    bm.fork(0, 2)
    assert [bm.refcount(b) for b in range(3)] == [3, 3, 3]
    slots, cow = bm.append_slots([1, 2, 0])
    # 1 and 2 copy the shared partial block; 0, the last holder, writes in place
    assert cow.tolist() == [[2, 3], [2, 4]]
    assert slots.tolist() == [3 * 16 + 8, 4 * 16 + 8, 2 * 16 + 8]
    assert [bm.refcount(b) for b in range(5)] == [3, 3, 1, 1, 1]
    bm.free(0)
    bm.free(1)
    # blocks 2 (sequence 0's) and 3 (sequence 1's copy) are freed; 0 and 1 stay with sequence 2
    assert bm.refcount(0) == 1 and bm.refcount(2) == 0 and bm.num_free_blocks == 16 - 5 + 2
    bm.free(2)
    assert bm.num_free_blocks == 16


def test_last_holder_of_a_shared_block_needs_no_free_block():
    """Two forks share a partly filled block and both append with one block free:
    the first copies it, the second (now its only holder) writes in place, so the
    call fits (P1 §4.2.2: a block is copied only while another sequence holds it)."""
    for make in (lambda: pkv.BlockManager(3, 8), lambda: oracle.BlockEngineRef(3, 8)):
        bm = make()
        bm.allocate(0, 12)                   # blocks 0, 1; block 1 holds 4 tokens
        bm.fork(0, 1)
        bm.allocate(2, 1)                    # block 2: the pool is now empty
        bm.free(2)                           # one free block
        got = bm.append_slots([0, 1])
        assert got is not None
        slots, cow = got
        assert [tuple(int(x) for x in p) for p in cow] == [(1, 2)]
        assert [int(x) for x in slots] == [2 * 8 + 4, 1 * 8 + 4]
    # three holders, two of them writing: both copy (a third sequence still holds the block)
    bm = pkv.BlockManager(4, 8)
    ref = oracle.BlockEngineRef(4, 8)
    for m in (bm, ref):
        m.allocate(0, 12)
        m.fork(0, 1)
        m.fork(0, 2)
    slots, cow = bm.append_slots([0, 1])
    want = ref.append_slots([0, 1])
    assert cow.tolist() == [[1, 2], [1, 3]] and [tuple(p) for p in want[1]] == [(1, 2), (1, 3)]


def test_oracle_manager_follows_the_same_pages():
    """The oracle's reference manager pinned to the same worked behaviour directly, not only
    through the differential test: ceil-sized FIFO allocation with freed blocks at the back
    (P2 §2.3, P4 §3), and a fork's partly filled block copied by every writer but the last
    holder (P1 §4.2.2, P2 §3.3)."""
    eng = oracle.BlockEngineRef(300, 16)
    assert eng.allocate(0, 50) and eng.tables[0] == [0, 1, 2, 3]
    assert eng.allocate(1, 4096) and eng.tables[1] == list(range(4, 260))
    assert eng.free(0)
    assert eng.allocate(2, 40 * 16) and eng.tables[2] == list(range(260, 300)) and len(eng.free_list) == 4
    assert eng.allocate(3, 1) and eng.tables[3] == [0]
    eng = oracle.BlockEngineRef(16, 16)
    eng.allocate(0, 40)
    eng.fork(0, 1)
    eng.fork(0, 2)
    assert eng.ref[:3] == [3, 3, 3]
    slots, cow = eng.append_slots([1, 2, 0])
    assert cow == [(2, 3), (2, 4)] and slots == [3 * 16 + 8, 4 * 16 + 8, 2 * 16 + 8]
    assert eng.ref[:5] == [3, 3, 1, 1, 1]
    eng.free(0)
    eng.free(1)
    assert eng.ref[0] == 1 and eng.ref[2] == 0 and len(eng.free_list) == 16 - 5 + 2


def test_fork_at_block_boundary_needs_no_copy():
    bm = pkv.BlockManager(8, 16)
    bm.allocate(0, 32)
    bm.fork(0, 1)
    slots, cow = bm.append_slots([0, 1])     # full shared block: each takes a fresh block
    assert len(cow) == 0 and slots.tolist() == [2 * 16, 3 * 16]


def test_invalid_calls():
    bm = pkv.BlockManager(8, 16)
    bm.allocate(0, 10)
    for f in (lambda: bm.allocate(0, 5), lambda: bm.fork(9, 1), lambda: bm.free(9),
              lambda: bm.append_slots([0, 0]), lambda: bm.append_slots([5]),
              lambda: bm.block_tables([0], 0)):
        with pytest.raises(pkv.PkvError) as e:
            f()
        assert e.value.status == pkv.PKV_ERR_INVALID
    with pytest.raises(ValueError):
        pkv.BlockManager(4, 16, free_order=[0, 1, 1, 3])


def test_huge_allocation_is_refused_whole():
    """ceil(tokens / block_size) must not overflow: a request for INT64_MAX
    tokens needs more blocks than any pool holds, so it fails and takes none."""
    bm = pkv.BlockManager(8, 16)
    for n in (2 ** 63 - 1, 2 ** 63 - 16, 9 * 16):
        with pytest.raises(pkv.PkvError) as e:
            bm.allocate(1, n)
        assert e.value.status == pkv.PKV_ERR_OOM
        assert bm.seq_len(1) == -1 and bm.num_free_blocks == 8
    bm.allocate(1, 8 * 16)                   # exactly the pool
    assert bm.num_free_blocks == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_reference(seed):
    rng = np.random.default_rng(seed)
    NB, bs = int(rng.integers(20, 200)), int(rng.choice([8, 16, 32]))
    order = rng.permutation(NB)
    bm = pkv.BlockManager(NB, bs, free_order=order)
    ref = oracle.BlockEngineRef(NB, bs, free_order=order)
    live, next_id = [], 0
    for _ in range(400):
        op = rng.choice(["alloc", "fork", "append", "free"], p=[0.2, 0.15, 0.5, 0.15])
        if op == "alloc":
            n = int(rng.integers(0, 6 * bs))
            ok_ref = ref.allocate(next_id, n)
            try:
                bm.allocate(next_id, n)
                ok = True
            except pkv.PkvError:
                ok = False
            assert ok == ok_ref
            if ok:
                live.append(next_id)
            next_id += 1
        elif op == "fork" and live:
            p = int(rng.choice(live))
            assert ref.fork(p, next_id)
            bm.fork(p, next_id)
            live.append(next_id)
            next_id += 1
        elif op == "append" and live:
            ids = [int(x) for x in rng.choice(live, size=min(len(live), int(rng.integers(1, 6))), replace=False)]
            want = ref.append_slots(ids)
            try:
                got = bm.append_slots(ids)
            except pkv.PkvError as e:
                assert want is None and e.status == pkv.PKV_ERR_OOM
                continue
            assert want is not None
            assert got[0].tolist() == want[0] and [tuple(p) for p in got[1].tolist()] == want[1]
        elif op == "free" and live:
            s = int(live.pop(int(rng.integers(len(live)))))
            assert ref.free(s)
            bm.free(s)
        assert bm.num_free_blocks == len(ref.free_list)
    if live:
        W = max(len(ref.tables[s]) for s in live)
        t, L = bm.block_tables(live, W)
        for i, s in enumerate(live):
            assert t[i, :len(ref.tables[s])].tolist() == ref.tables[s] and L[i] == ref.lens[s]
        assert [bm.refcount(b) for b in range(NB)] == ref.ref
