"""Pins for the allocator model (oracle side): the pages' 100-token example,
waste confined to each sequence's last block, conservation of blocks and
references, copy-on-write only where branches diverge inside a shared block,
immediate reuse of freed blocks, and all-or-nothing failure."""
import json
import os
import random

from oracle import BlockAllocatorModel, OK, ERR_INVALID, ERR_OOM, blocks_needed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_invariants(m: BlockAllocatorModel):
    live = {}
    for s in m.sequences():
        table = m.block_table(s)
        n = m.num_tokens(s)
        # blocks are held only for tokens that exist: ceil(n / B) of them
        assert len(table) == blocks_needed(n, m.block_size)
        for b in table:
            live[b] = live.get(b, 0) + 1
    # conservation: every block is either free or referenced, never both
    assert m.num_free() + len(live) == m.num_blocks
    for b in range(m.num_blocks):
        assert m.refcount(b) == live.get(b, 0)
    occupied, allocated = m.waste()
    assert allocated == len(live) * m.block_size
    assert 0 <= allocated - occupied


def test_hundred_tokens_take_seven_blocks():
    g = json.load(open(os.path.join(GOLDEN, "block_table_example.json")))
    B = g["block_size"]
    m = BlockAllocatorModel(num_blocks=g["reserved_blocks"], block_size=B)
    assert m.add_seq(0, 0) == OK
    for _ in range(g["tokens"]):
        st, slot, src, dst = m.append_slot(0)
        assert st == OK and src == -1 and dst == -1
    assert len(m.block_table(0)) == g["blocks"]
    occupied, allocated = m.waste()
    assert (occupied, allocated) == (g["tokens"], g["slots"])
    # the same request as one prompt
    m2 = BlockAllocatorModel(num_blocks=g["reserved_blocks"], block_size=B)
    assert m2.add_seq(7, g["tokens"]) == OK
    assert len(m2.block_table(7)) == g["blocks"]
    # a 4096-token reservation would have held the whole pool
    assert m2.add_seq(8, g["reserved_tokens"]) == ERR_OOM
    assert m2.num_free() == g["reserved_blocks"] - g["blocks"]


def test_slots_walk_the_block_table():
    m = BlockAllocatorModel(num_blocks=8, block_size=4)
    m.add_seq(1, 0)
    slots = [m.append_slot(1)[1] for _ in range(10)]
    table = m.block_table(1)
    assert slots == [table[p // 4] * 4 + p % 4 for p in range(10)]


def test_freed_blocks_are_reused_without_compaction():
    m = BlockAllocatorModel(num_blocks=6, block_size=4)
    for s in range(3):
        assert m.add_seq(s, 8) == OK  # two blocks each: the pool is full
    assert m.add_seq(9, 1) == ERR_OOM
    middle = m.block_table(1)
    assert m.free_seq(1) == OK
    # the hole left in the middle is used at once
    assert m.add_seq(9, 8) == OK
    assert sorted(m.block_table(9)) == sorted(middle)
    check_invariants(m)


def test_beams_share_prefix_and_copy_only_a_partial_last_block():
    B = 16
    m = BlockAllocatorModel(num_blocks=256, block_size=B)
    assert m.add_seq(0, 1032) == OK  # 64 full blocks + 8 tokens
    for child in range(1, 8):
        assert m.fork(0, child) == OK
    shared = m.block_table(0)
    assert all(m.refcount(b) == 8 for b in shared)
    copies = []
    for beam in range(8):
        st, slot, src, dst = m.append_slot(beam)
        assert st == OK
        if src >= 0:
            copies.append((src, dst))
    # 8 beams diverge inside the shared last block: 7 copies, the last holder
    # writes in place
    assert len(copies) == 7
    assert all(src == shared[-1] for src, _ in copies)
    assert m.refcount(shared[-1]) == 1
    for b in shared[:-1]:
        assert m.refcount(b) == 8  # full prefix blocks stay shared
    check_invariants(m)


def test_full_shared_block_is_never_copied():
    m = BlockAllocatorModel(num_blocks=200, block_size=16)
    m.add_seq(0, 1024)  # exactly 64 full blocks
    for child in range(1, 8):
        m.fork(0, child)
    for beam in range(8):
        st, slot, src, dst = m.append_slot(beam)
        assert st == OK and src == -1
    check_invariants(m)


def test_failures_change_nothing():
    m = BlockAllocatorModel(num_blocks=3, block_size=2)
    m.add_seq(0, 5)  # 3 blocks, last one half full
    m.fork(0, 1)
    snap = (m.block_table(0), m.block_table(1), m.num_free(), [m.refcount(b) for b in range(3)])
    assert m.append_slot(1)[0] == ERR_OOM  # would need a copy, pool empty
    assert m.add_seq(2, 1) == ERR_OOM
    assert m.fork(0, 1) == ERR_INVALID
    assert m.free_seq(5) == ERR_INVALID
    assert m.append_slot(42)[0] == ERR_INVALID
    assert snap == (m.block_table(0), m.block_table(1), m.num_free(), [m.refcount(b) for b in range(3)])


def test_random_operation_sequences_keep_invariants():
    rnd = random.Random(11)
    for trial in range(30):
        B = rnd.choice([1, 2, 4, 8, 16])
        m = BlockAllocatorModel(num_blocks=rnd.randint(1, 64), block_size=B)
        next_id = 0
        for _ in range(300):
            seqs = m.sequences()
            op = rnd.random()
            if op < 0.25 or not seqs:
                m.add_seq(next_id, rnd.randint(0, 3 * B))
                next_id += 1
            elif op < 0.65:
                m.append_slot(rnd.choice(seqs))
            elif op < 0.8:
                m.fork(rnd.choice(seqs), next_id)
                next_id += 1
            else:
                m.free_seq(rnd.choice(seqs))
            check_invariants(m)
            # waste: only the last block of a sequence can be partly empty
            for s in m.sequences():
                n, t = m.num_tokens(s), m.block_table(s)
                assert len(t) * B - n < B or n == 0
