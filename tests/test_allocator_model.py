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


# -- prefix caching ("vLLM PagedAttention: Buoc dot pha ve thong luong suy luan LLM",
#    advanced features, "Prefix caching": a shared prompt prefix's KV is reused) --

def test_prefix_cache_shares_leading_full_blocks():
    m = BlockAllocatorModel(16, 16)
    system = list(range(100, 140))                       # a 40-token system prompt
    st, cached = m.add_seq_cached(0, system + [1, 2, 3])  # 43 tokens: blocks 0, 1, 2
    assert (st, cached) == (OK, 0) and m.block_table(0) == [0, 1, 2]
    st, cached = m.add_seq_cached(1, system + [7, 8])    # 42 tokens: the two full blocks are found
    assert (st, cached) == (OK, 32)
    assert m.block_table(1)[:2] == [0, 1] and m.block_table(1)[2] == 3
    assert m.refcount(0) == m.refcount(1) == 2 and m.refcount(2) == 1
    # the third block of the first prompt held tokens 32..42: not full, never registered
    # prompt 0: 2 full blocks, both new (misses); prompt 1: both found (hits)
    assert m.cache_stats() == {"hits": 2, "misses": 2, "cached_blocks": 2, "evictable_blocks": 0}


def test_prefix_cache_counts_only_full_blocks():
    m = BlockAllocatorModel(8, 4)
    st, c = m.add_seq_cached(0, [1, 2, 3, 4, 5, 6])   # one full block, one partial
    assert (st, c) == (OK, 0)
    st, c = m.add_seq_cached(1, [1, 2, 3, 4, 5, 6])   # the same prompt: only the full block is shared
    assert (st, c) == (OK, 4)
    assert m.block_table(1)[0] == m.block_table(0)[0] and m.block_table(1)[1] != m.block_table(0)[1]
    st, c = m.add_seq_cached(2, [1, 2, 3, 9, 5, 6])   # differs inside the first block: nothing shared
    assert (st, c) == (OK, 0)
    st, c = m.add_seq_cached(3, [1, 2, 3, 4])         # exactly the first block
    assert (st, c) == (OK, 4)


def test_prefix_cache_survives_free_and_evicts_tail_first():
    m = BlockAllocatorModel(6, 2)
    prompt = [5, 6, 7, 8, 9, 10]                      # three full blocks
    assert m.add_seq_cached(0, prompt) == (OK, 0)
    table = m.block_table(0)
    assert m.free_seq(0) == OK
    # nothing holds the blocks, yet they stay registered and count as free
    assert m.num_free() == 6 and m.cache_stats()["evictable_blocks"] == 3
    assert m.add_seq_cached(1, prompt) == (OK, 6)      # found again, same blocks
    assert m.block_table(1) == table and m.cache_stats()["evictable_blocks"] == 0
    assert m.free_seq(1) == OK
    # 3 free + 3 evictable; a 4-block prompt takes the free ones, then evicts the
    # prompt's last block first
    assert m.add_seq(2, 8) == OK
    assert m.cache_stats()["evictable_blocks"] == 2 and m.cache_stats()["cached_blocks"] == 2
    assert table[2] in m.block_table(2)
    # no room for the prompt's third block while sequence 2 holds the rest
    assert m.add_seq_cached(3, prompt) == (ERR_OOM, 0)
    assert m.free_seq(2) == OK
    assert m.add_seq_cached(3, prompt) == (OK, 4)      # the first two blocks are still there
    assert m.block_table(3)[:2] == table[:2]


def test_prefix_cache_oom_changes_nothing_and_clear_forgets():
    m = BlockAllocatorModel(3, 2)
    assert m.add_seq_cached(0, [1, 2, 3, 4]) == (OK, 0)
    before = (m.block_table(0), m.num_free(), m.cache_stats())
    assert m.add_seq_cached(1, [1, 2, 9, 9, 9, 9]) == (ERR_OOM, 0)   # needs 2 new blocks, 1 left
    assert (m.block_table(0), m.num_free(), m.cache_stats()) == before and 1 not in m.sequences()
    assert m.free_seq(0) == OK and m.cache_clear() == OK
    assert m.cache_stats()["cached_blocks"] == 0 and m.num_free() == 3
    assert m.add_seq_cached(1, [1, 2, 3, 4]) == (OK, 0)


# ---------------------------------------------------------------------------
# Truncation (rolling back rejected drafted tokens)
# ---------------------------------------------------------------------------
def test_truncate_releases_whole_blocks_and_appends_reuse_the_slots():
    m = BlockAllocatorModel(16, 16)
    assert m.add_seq(0, 100) == OK                  # blocks 0..6, the last holds 4 tokens
    assert m.truncate(0, 40) == OK
    assert m.block_table(0) == [0, 1, 2] and m.num_tokens(0) == 40
    assert m.num_free() == 13
    # position 40 is block 2, offset 8 again
    assert m.append_slot(0) == (OK, 2 * 16 + 8, -1, -1)
    # fill block 2 (positions 41..47); blocks 3..6 went back in table order, so the
    # next fresh block is 6
    for _ in range(7):
        assert m.append_slot(0)[0] == OK
    assert m.append_slot(0) == (OK, 6 * 16, -1, -1)
    assert m.truncate(0, 0) == OK and m.block_table(0) == [] and m.num_free() == 16
    # blocks 0, 1, 2, 6 went back in table order: block 6 is handed out next
    assert m.append_slot(0) == (OK, 6 * 16, -1, -1)


def test_truncate_into_a_shared_block_copies_it_on_the_next_append():
    m = BlockAllocatorModel(16, 16)
    m.add_seq(0, 40)                                # blocks 0, 1, 2 (2 holds 8 tokens)
    m.fork(0, 1)
    assert m.truncate(1, 20) == OK                  # keeps 0, 1; block 1 now partial for seq 1
    assert m.refcount(2) == 1 and m.refcount(1) == 2
    st, slot, src, dst = m.append_slot(1)           # position 20 lands in shared block 1: copy
    assert st == OK and src == 1 and dst not in (0, 1, 2) and slot == dst * 16 + 4
    assert m.append_slot(0) == (OK, 2 * 16 + 8, -1, -1)  # seq 0 alone holds block 2


def test_truncate_unregisters_a_cached_block_it_will_write_and_parks_dropped_ones():
    m = BlockAllocatorModel(8, 16)
    prompt = list(range(100, 148))                  # 3 full blocks, all registered
    assert m.add_seq_cached(0, prompt) == (OK, 0)
    assert m.cache_stats()["cached_blocks"] == 3
    assert m.truncate(0, 20) == OK                  # keeps blocks 0, 1 (1 now partial)
    stats = m.cache_stats()
    # block 1 (partial, sole holder) unregistered; block 2 dropped but still registered
    assert stats["cached_blocks"] == 2 and stats["evictable_blocks"] == 1
    assert m.num_free() == 8 - 2
    # a new prompt with the same tokens finds only block 0 (its chain stops at block 1)
    assert m.add_seq_cached(1, prompt) == (OK, 16)


def test_truncate_rejects_bad_arguments_and_changes_nothing():
    m = BlockAllocatorModel(8, 16)
    m.add_seq(0, 30)
    before = (m.block_table(0), m.num_tokens(0), m.num_free())
    assert m.truncate(0, 31) == ERR_INVALID
    assert m.truncate(0, -1) == ERR_INVALID
    assert m.truncate(7, 0) == ERR_INVALID
    assert (m.block_table(0), m.num_tokens(0), m.num_free()) == before


def test_extend_equals_single_appends_and_is_all_or_nothing():
    a = BlockAllocatorModel(16, 16)
    b = BlockAllocatorModel(16, 16)
    for m in (a, b):
        m.add_seq(0, 40)
        m.fork(0, 1)                                # block 2 (8 tokens) shared
    st, slots, src, dst = a.extend(1, 30)           # positions 40..69 of seq 1
    singles = [b.append_slot(1) for _ in range(30)]
    assert st == OK and slots == [x[1] for x in singles]
    # the shared partial block is copied once, at the first token
    assert (src, dst) == (singles[0][2], singles[0][3]) and src == 2
    assert a.block_table(1) == b.block_table(1) and a.num_free() == b.num_free()
    # not enough blocks: nothing changes
    before = (a.block_table(1), a.num_tokens(1), a.num_free())
    assert a.extend(1, 16 * 16)[0] == ERR_OOM
    assert (a.block_table(1), a.num_tokens(1), a.num_free()) == before
    assert a.extend(1, 0) == (OK, [], -1, -1) and a.extend(1, -1)[0] == ERR_INVALID
