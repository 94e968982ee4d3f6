"""Host block manager (free list, reference counts, on-demand allocation,
copy-on-write).  CPU only: the manager is host code in the library."""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_260_gb300 import PagedAttnError
from paged_kv_cache_260_gb300.block_manager import PA_ERR_OUT_OF_BLOCKS, BlockManager

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_260_gb300 import _build
    _build.build()


def test_page3_pool_state_from_on_demand_allocation():
    # The block-pool figure shows A in blocks 0,2,6, B in 1,4,7 and blocks 3, 5
    # empty.  Reading: a third request C took blocks while A and B grew and has
    # finished; allocating on demand in this order and releasing C gives exactly
    # the printed pool row.
    g = json.load(open(os.path.join(GOLDEN, "page3_block_table.json")))
    bm = BlockManager(g["pool_blocks"], g["block_size"])
    ids = {"A": 1, "B": 2, "C": 3}
    for r in ids.values():
        bm.add_sequence(r)
    for req in ["A", "B", "A", "C", "B", "C", "A", "B"]:     # one block's worth of tokens each
        bm.append(ids[req], g["block_size"])
    bm.free(ids["C"])
    for req in ("A", "B"):
        table, nb, ln = bm.block_table(ids[req], 3)
        assert table.tolist() == g["tables"][req] and nb == 3 and ln == 48
    st = bm.stats()
    assert st["free_blocks"] == len(g["free_blocks"])
    assert [b for b in range(g["pool_blocks"]) if bm.ref_count(b) == 0] == g["free_blocks"]


def test_waste_under_one_block_and_slots_follow_the_table():
    rng = np.random.default_rng(0)
    bm = BlockManager(4000)
    lens = {}
    for sid in range(60):
        bm.add_sequence(sid)
        lens[sid] = 0
    for _ in range(400):
        sid = int(rng.integers(60))
        n = int(rng.integers(1, 40))
        slots, cow = bm.append(sid, n)
        assert cow is None
        table, nb, ln = bm.block_table(sid, 256)
        for i, sl in enumerate(slots):
            t = lens[sid] + i
            assert sl == table[t // 16] * 16 + t % 16
        lens[sid] += n
        assert ln == lens[sid] and nb == -(-ln // 16)       # under one block of waste
    st = bm.stats()
    assert st["num_blocks"] - st["free_blocks"] == sum(-(-L // 16) for L in lens.values())


def test_out_of_blocks_changes_nothing():
    bm = BlockManager(4)
    bm.add_sequence(0)
    bm.append(0, 40)                                        # 3 blocks
    before = bm.stats()
    with pytest.raises(PagedAttnError) as e:
        bm.append(0, 40)                                    # needs 3 more, 1 free
    assert e.value.status == PA_ERR_OUT_OF_BLOCKS
    assert bm.stats() == before and bm.block_table(0, 8)[2] == 40
    bm.append(0, 8)                                         # fits the partial block + 1 new


def test_fork_and_copy_on_write():
    bm = BlockManager(64)
    bm.add_sequence(0)
    bm.append(0, 40)                                        # blocks 0,1,2; block 2 half full
    for c in (1, 2, 3):
        bm.fork(0, c)
    assert [bm.ref_count(b) for b in (0, 1, 2)] == [4, 4, 4]
    slots, cow = bm.append(1, 1)                            # write into the shared block
    assert cow == (2, 3)                                    # copy of block 2 into fresh block 3
    assert slots[0] == 3 * 16 + 8
    assert bm.ref_count(2) == 3 and bm.ref_count(3) == 1
    assert bm.append(1, 1)[1] is None                       # its own copy now
    assert bm.append(2, 1)[1] == (2, 4)
    assert bm.append(0, 1)[1] == (2, 5)                     # the parent copies too
    slots, cow = bm.append(3, 1)                            # last sharer keeps the original
    assert cow is None and slots[0] == 2 * 16 + 8
    assert bm.stats()["cow_copies"] == 3
    for sid in range(4):                                    # prompt blocks still shared
        assert bm.block_table(sid, 4)[0][:2].tolist() == [0, 1]


def test_block_aligned_prompt_needs_no_copy():
    bm = BlockManager(64)
    bm.add_sequence(0)
    bm.append(0, 32)
    bm.fork(0, 1)
    slots, cow = bm.append(1, 1)
    assert cow is None and slots[0] // 16 not in (0, 1)
    assert bm.ref_count(0) == 2 and bm.ref_count(1) == 2


def test_no_leak_and_reference_invariant():
    rng = np.random.default_rng(1)
    bm = BlockManager(3000)
    live = []
    for step in range(600):
        op = rng.integers(4)
        if op == 0 or not live:
            sid = step
            bm.add_sequence(sid)
            live.append(sid)
        elif op == 1:
            child = 100000 + step
            bm.fork(int(rng.choice(live)), child)
            live.append(child)
        elif op == 2:
            sid = int(rng.choice(live))
            slots, cow = bm.append(sid, int(rng.integers(1, 20)))
            # the block written to is owned by this sequence alone
            assert bm.ref_count(int(slots[-1]) // 16) == 1
        else:
            sid = live.pop(int(rng.integers(len(live))))
            bm.free(sid)
        total_refs = sum(bm.ref_count(b) for b in range(3000))
        assert total_refs == sum(bm.block_table(s, 256)[1] for s in live)
    for sid in live:
        bm.free(sid)
    st = bm.stats()
    assert st["free_blocks"] == 3000 and st["allocations"] == st["releases"]
    assert st["shared_blocks"] == 0 and st["num_sequences"] == 0


def test_bad_calls():
    bm = BlockManager(8)
    bm.add_sequence(5)
    with pytest.raises(PagedAttnError):
        bm.add_sequence(5)
    with pytest.raises(PagedAttnError):
        bm.append(6, 1)
    with pytest.raises(PagedAttnError):
        bm.fork(7, 8)
    with pytest.raises(PagedAttnError):
        bm.block_table(5, 0) if bm.append(5, 20) else None    # 2 blocks do not fit 0 entries
    assert bm.ref_count(99) == -1
    with pytest.raises(ValueError):
        BlockManager(0)
