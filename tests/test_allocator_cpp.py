"""The library's C++ allocator against the oracle's allocator model,
operation by operation (statuses, slots, copy pairs, tables, refcounts,
free counts and waste must all be identical)."""
import random

import numpy as np
import pytest

import paged_kv_cache_279_gb300 as pkv
from oracle import BlockAllocatorModel


def assert_same_state(c, m, seqs):
    assert c.num_free() == m.num_free()
    for b in range(m.num_blocks):
        assert c.refcount(b) == m.refcount(b)
    for s in seqs:
        assert c.block_table(s) == m.block_table(s)
        assert c.num_tokens(s) == m.num_tokens(s)
    assert c.waste() == m.waste()


def run_ops(ops, num_blocks, block_size):
    c = pkv.BlockAllocator(num_blocks, block_size)
    m = BlockAllocatorModel(num_blocks, block_size)
    for op in ops:
        kind = op[0]
        if kind == "add":
            assert c.add_seq(op[1], op[2]) == m.add_seq(op[1], op[2])
        elif kind == "append":
            assert c.append_slot(op[1]) == m.append_slot(op[1])
        elif kind == "fork":
            assert c.fork(op[1], op[2]) == m.fork(op[1], op[2])
        elif kind == "free":
            assert c.free_seq(op[1]) == m.free_seq(op[1])
        elif kind == "cached":
            assert c.add_seq_cached(op[1], op[2]) == m.add_seq_cached(op[1], op[2])
        elif kind == "clear":
            assert c.cache_clear() == m.cache_clear()
        elif kind == "truncate":
            assert c.truncate(op[1], op[2]) == m.truncate(op[1], op[2])
        elif kind == "extend":
            cs, cslots, csrc, cdst = c.extend(op[1], op[2])
            assert (cs, cslots.tolist(), csrc, cdst) == m.extend(op[1], op[2])
        assert_same_state(c, m, m.sequences())
        assert c.cache_stats() == m.cache_stats()
    return c, m


def random_ops(rnd, n, block_size):
    ops, ids = [], []
    for _ in range(n):
        r = rnd.random()
        if r < 0.2 or not ids:
            ids.append(len(ids) + rnd.randint(0, 2))  # occasionally a duplicate id
            ops.append(("add", ids[-1], rnd.randint(0, 3 * block_size)))
        elif r < 0.65:
            ops.append(("append", rnd.choice(ids + [999])))
        elif r < 0.8:
            child = len(ids) + 100
            ops.append(("fork", rnd.choice(ids), child))
            ids.append(child)
        elif r < 0.85:
            ops.append(("truncate", rnd.choice(ids), rnd.randint(-1, 3 * block_size)))
        elif r < 0.9:
            ops.append(("extend", rnd.choice(ids + [999]), rnd.randint(-1, 2 * block_size + 3)))
        else:
            ops.append(("free", rnd.choice(ids)))
    return ops


@pytest.mark.parametrize("seed", range(12))
def test_random_sequences_match_model(seed):
    rnd = random.Random(seed)
    B = rnd.choice([1, 4, 8, 16, 32])
    run_ops(random_ops(rnd, 250, B), rnd.randint(1, 48), B)


def test_hypothesis_sequences_match_model():
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    op = st.one_of(
        st.tuples(st.just("add"), st.integers(0, 6), st.integers(0, 40)),
        st.tuples(st.just("append"), st.integers(0, 6)),
        st.tuples(st.just("fork"), st.integers(0, 6), st.integers(0, 6)),
        st.tuples(st.just("free"), st.integers(0, 6)),
    )

    @hyp.settings(max_examples=150, deadline=None, derandomize=True)
    @hyp.given(st.lists(op, max_size=60), st.integers(1, 20), st.sampled_from([1, 2, 4, 16]))
    def prop(ops, nb, bs):
        run_ops(ops, nb, bs)

    prop()


def test_beam_fork_copy_pairs_and_dense_tables():
    c = pkv.BlockAllocator(400, 16)
    assert c.add_seq(0, 1032) == 0
    for k in range(1, 8):
        assert c.fork(0, k) == 0
    pairs = []
    for k in range(8):
        st, slot, src, dst = c.append_slot(k)
        assert st == 0
        if src >= 0:
            pairs.append((src, dst))
    assert len(pairs) == 7
    tables, lens = c.block_tables(list(range(8)), cap=70, pad=-5)
    assert tables.shape == (8, 70) and (lens == 1033).all()
    assert (tables[:, 66:] == -5).all()
    assert len(set(tables[:, 64].tolist())) == 8  # every beam now owns its last block
    assert (tables[:, :64] == tables[0, :64]).all()  # full prefix blocks still shared
    slots = c.slots(3, 1030, 3)
    t3 = c.block_table(3)
    assert slots.tolist() == [t3[p // 16] * 16 + p % 16 for p in (1030, 1031, 1032)]
    with pytest.raises(pkv.PkvError):
        c.slots(3, 1030, 10)  # past the end
    with pytest.raises(pkv.PkvError):
        c.block_tables([0, 1], cap=10)  # too narrow


@pytest.mark.parametrize("seed", range(6))
def test_batched_append_matches_sequential_model(seed):
    rnd = random.Random(100 + seed)
    B = rnd.choice([4, 16])
    NB = rnd.randint(8, 60)
    c = pkv.BlockAllocator(NB, B)
    m = BlockAllocatorModel(NB, B)
    live = []
    for sid in range(6):
        n = rnd.randint(0, 2 * B)
        assert c.add_seq(sid, n) == m.add_seq(sid, n)
        if sid in m.sequences():
            live.append(sid)
    for sid in list(live)[:3]:
        child = 100 + sid
        if c.fork(sid, child) == 0:
            m.fork(sid, child)
            live.append(child)
    for step in range(40):
        batch = rnd.sample(live, rnd.randint(1, len(live)))
        st, slots, pairs = c.append_slots(batch)
        # model: all or nothing over the sequential semantics
        need = sum(1 for s in batch
                   if m.num_tokens(s) % B == 0 or m.refcount(m.block_table(s)[-1]) > 1)
        if need > m.num_free():
            assert st == 2
            assert_same_state(c, m, live)
            continue
        assert st == 0
        want_slots, want_pairs = [], []
        for s in batch:
            mst, slot, src, dst = m.append_slot(s)
            assert mst == 0
            want_slots.append(slot)
            if src >= 0:
                want_pairs.append((src, dst))
        assert slots.tolist() == want_slots
        assert [tuple(p) for p in pairs.tolist()] == want_pairs
        assert_same_state(c, m, live)
    st, _, _ = c.append_slots([live[0], live[0]])
    assert st == 1  # repeated id


def test_prefix_groups_follow_forks():
    c = pkv.BlockAllocator(600, 16)
    for p in range(3):
        assert c.add_seq(10 * p, 1032) == 0
        for k in range(1, 4):
            assert c.fork(10 * p, 10 * p + k) == 0
    assert c.add_seq(100, 40) == 0
    order = [0, 1, 2, 3, 10, 11, 12, 13, 100, 20, 21, 22, 23]
    offs, pre = c.prefix_groups(order)
    assert offs.tolist() == [0, 4, 8, 9, 13]
    assert pre.tolist() == [1024, 1024, 0, 1024]  # 64 full shared blocks; singleton 0
    # after every beam appends (copy-on-write of the partial block) the full blocks stay shared
    for s in order:
        assert c.append_slot(s)[0] == 0
    offs2, pre2 = c.prefix_groups(order)
    assert offs2.tolist() == offs.tolist() and pre2.tolist() == [1024, 1024, 0, 1024]
    # block size 8 rounds the shared length down to whole 16-token tiles
    c8 = pkv.BlockAllocator(100, 8)
    c8.add_seq(0, 100)
    c8.fork(0, 1)
    offs8, pre8 = c8.prefix_groups([0, 1])
    assert offs8.tolist() == [0, 2] and pre8.tolist() == [96]


def prompt_ops(rnd, n, block_size, vocab=3):
    """Prompts drawn from a few shared prefixes (prefix caching), mixed with
    appends, forks, frees, plain prompts and cache clears."""
    bases = [[rnd.randrange(vocab) for _ in range(4 * block_size)] for _ in range(3)]
    ops, ids = [], []
    for _ in range(n):
        r = rnd.random()
        if r < 0.35 or not ids:
            base = rnd.choice(bases)
            cut = rnd.randint(0, len(base))
            tail = [rnd.randrange(vocab) for _ in range(rnd.randint(0, block_size + 3))]
            ids.append(len(ids) + 1000 * rnd.randint(0, 1))
            ops.append(("cached", ids[-1], base[:cut] + tail))
        elif r < 0.4:
            ids.append(len(ids) + 5000)
            ops.append(("add", ids[-1], rnd.randint(0, 2 * block_size)))
        elif r < 0.65:
            ops.append(("append", rnd.choice(ids)))
        elif r < 0.75:
            child = len(ids) + 10000
            ops.append(("fork", rnd.choice(ids), child))
            ids.append(child)
        elif r < 0.82:
            ops.append(("truncate", rnd.choice(ids), rnd.randint(0, 5 * block_size)))
        elif r < 0.85:
            ops.append(("extend", rnd.choice(ids), rnd.randint(0, 2 * block_size)))
        elif r < 0.97:
            ops.append(("free", rnd.choice(ids)))
        else:
            ops.append(("clear",))
    return ops


@pytest.mark.parametrize("seed", range(16))
def test_prefix_cache_sequences_match_model(seed):
    """add_seq_cached with hits, misses, evictions under pressure and clears:
    tables, refcounts, free counts and cache counters equal the model's."""
    rnd = random.Random(1000 + seed)
    B = rnd.choice([2, 4, 16])
    run_ops(prompt_ops(rnd, 250, B), num_blocks=rnd.choice([6, 12, 40]), block_size=B)


def test_prefix_cache_reports_cached_tokens_and_shares_blocks():
    c = pkv.BlockAllocator(64, 16)
    system = list(range(1000, 1040))                 # 40 shared tokens: 2 full blocks
    assert c.add_seq_cached(0, system + [1, 2, 3]) == (pkv.PKV_OK, 0)
    assert c.add_seq_cached(1, system + [4, 5]) == (pkv.PKV_OK, 32)
    assert c.block_table(1)[:2] == c.block_table(0)[:2]
    assert c.cache_stats() == {"hits": 2, "misses": 2, "cached_blocks": 2, "evictable_blocks": 0}
    # the shared blocks are prefix groups for the grouped decode
    offs, pre = c.prefix_groups([0, 1])
    assert offs.tolist() == [0, 2] and pre.tolist() == [32]


@pytest.mark.parametrize("seed", range(6))
def test_append_step_keeps_dense_tables_equal_to_a_rebuild(seed):
    """The serving loop's incremental tables: after every step (fresh blocks,
    CoW of shared last blocks after forks, OOM refusals) the tables and lengths
    that append_step updated in place equal a full block_tables rebuild, and the
    slots and copy pairs equal append_slots' on the reference model."""
    rnd = random.Random(300 + seed)
    B = rnd.choice([4, 8, 16])
    NB = rnd.randint(20, 80)
    c = pkv.BlockAllocator(NB, B)
    m = BlockAllocatorModel(NB, B)
    live = []
    for sid in range(5):
        n = rnd.randint(1, 3 * B)
        if c.add_seq(sid, n) == 0:
            assert m.add_seq(sid, n) == 0
            live.append(sid)
    for sid in list(live)[:2]:
        for k in range(2):
            child = 100 * (k + 1) + sid
            if c.fork(sid, child) == 0:
                m.fork(sid, child)
                live.append(child)
    cap = 40
    tables, lens = c.block_tables(live, cap=cap, pad=-1)
    tables, lens = np.ascontiguousarray(tables), np.ascontiguousarray(lens)
    for step in range(30):
        before = tables.copy(), lens.copy()
        st, slots, pairs = c.append_step(live, tables, lens)
        need = sum(1 for s in live if m.num_tokens(s) % B == 0 or m.refcount(m.block_table(s)[-1]) > 1)
        if need > m.num_free():
            assert st == 2
            assert np.array_equal(tables, before[0]) and np.array_equal(lens, before[1])
            break
        assert st == 0
        want_slots, want_pairs = [], []
        for s in live:
            mst, slot, src, dst = m.append_slot(s)
            assert mst == 0
            want_slots.append(slot)
            if src >= 0:
                want_pairs.append((src, dst))
        assert slots.tolist() == want_slots
        assert [tuple(p) for p in pairs.tolist()] == want_pairs
        ref_t, ref_l = c.block_tables(live, cap=cap, pad=-1)
        assert np.array_equal(tables, ref_t) and np.array_equal(lens, ref_l)
        assert_same_state(c, m, live)


def test_append_step_refuses_a_row_too_narrow():
    c = pkv.BlockAllocator(16, 4)
    assert c.add_seq(0, 8) == 0 and c.add_seq(1, 3) == 0
    tables, lens = c.block_tables([0, 1], cap=2, pad=-1)
    tables, lens = np.ascontiguousarray(tables), np.ascontiguousarray(lens)
    st, _, _ = c.append_step([0, 1], tables, lens)  # seq 0's ninth token needs block index 2
    assert st == 1
    assert c.num_tokens(0) == 8 and c.num_tokens(1) == 3 and c.num_free() == 13
    st, slots, _ = c.append_step([1], tables[1:], lens[1:])
    assert st == 0 and lens[1] == 4 and slots[0] == tables[1, 0] * 4 + 3
    with pytest.raises(ValueError):
        c.append_step([0], tables[:, :1], lens[:1])  # not C-contiguous
