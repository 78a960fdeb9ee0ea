"""Pins for the CPU oracle: values the pages print, closed forms, invariants and
an independent library routine.  Each test is chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, a wrong head mapping) fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------
def test_kv_size_worked_example():
    g = _golden("kv_size_example.json")
    total = oracle.kv_cache_bytes(g["layers"], g["tokens"], g["kv_heads"], g["head_dim"],
                                  g["bytes_per_element"])
    # The printed figure matches one of K or V (the formula without its 2).
    per_tensor_gb = total / 2 / 1e9
    assert abs(per_tensor_gb - g["printed_total_gb"]) <= g["printed_precision_gb"]
    # ... and the formula itself, key AND value, is twice the printed total.
    assert abs(total / 1e9 - 2 * g["printed_total_gb"]) <= 2 * g["printed_precision_gb"]


def test_kv_size_matches_real_pool_bytes():
    """The closed form equals the bytes a paged pool really holds for one
    16,000-token sequence: 1000 full blocks per layer, K and V tensors of shape
    [blocks, kv_heads, block_size, head_dim] in a 2-byte type, 32 layers."""
    g = _golden("kv_size_example.json")
    blocks = oracle.blocks_needed(g["tokens"], 16)
    one_k = torch.empty((blocks, g["kv_heads"], 16, g["head_dim"]), dtype=torch.bfloat16, device="meta")
    pool_bytes = g["layers"] * 2 * one_k.numel() * one_k.element_size()
    assert pool_bytes == oracle.kv_cache_bytes(g["layers"], g["tokens"], g["kv_heads"],
                                               g["head_dim"], g["bytes_per_element"])


def test_block_table_example():
    g = _golden("block_table_example.json")
    B = g["block_size"]
    assert oracle.blocks_needed(g["tokens"], B) == g["blocks"]
    assert oracle.blocks_needed(g["tokens"], B) * B == g["slots"]
    assert oracle.blocks_needed(g["reserved_tokens"], B) == g["reserved_blocks"]
    assert math.isclose(oracle.paged_waste_fraction([g["tokens"]], B),
                        (g["slots"] - g["tokens"]) / g["slots"])
    assert math.isclose(oracle.preallocation_waste_fraction([g["tokens"]], g["reserved_tokens"]),
                        1 - g["tokens"] / g["reserved_tokens"])


def test_slot_of_follows_logical_blocks():
    g = _golden("block_table_example.json")
    B = g["block_size"]
    table = [41, 7, 19]
    for (lo, hi), phys in zip(g["logical_blocks_example"], table):
        slots = [oracle.slot_of(table, p, B) for p in range(lo, hi + 1)]
        # every token of logical block i lands in physical block table[i] ...
        assert all(s // B == phys for s in slots)
        # ... in order, one slot per token
        assert slots == list(range(phys * B, phys * B + B))
    all_slots = [oracle.slot_of(table, p, B) for p in range(len(table) * B)]
    assert len(set(all_slots)) == len(all_slots)


# ---------------------------------------------------------------------------
# Decode attention
# ---------------------------------------------------------------------------
def _case(rng, S, Hq, Hkv, D, lens):
    q = _rand(rng, S, Hq, D)
    ks = [_rand(rng, L, Hkv, D) for L in lens]
    vs = [_rand(rng, L, Hkv, D) for L in lens]
    return q, ks, vs


@pytest.mark.parametrize("Hq,Hkv,D,lens", [
    (4, 4, 64, [1, 17, 33, 100]),
    (8, 2, 64, [5, 64, 200]),
    (32, 8, 128, [3, 129, 513]),
    (16, 2, 128, [1000]),
    (8, 1, 64, [2, 40]),
])
def test_decode_matches_library_sdpa(Hq, Hkv, D, lens):
    """torch's scaled_dot_product_attention in float64 (an independent library
    routine), with each KV head repeated for its group of query heads."""
    rng = np.random.default_rng(1234 + Hq + D)
    q, ks, vs = _case(rng, len(lens), Hq, Hkv, D, lens)
    scale = 1.0 / math.sqrt(D)
    out, werr = oracle.decode_attention(q, ks, vs, scale, return_weight_error=True)
    G = Hq // Hkv
    for s, L in enumerate(lens):
        qt = torch.from_numpy(q[s]).reshape(1, Hq, 1, D)
        kt = torch.from_numpy(ks[s]).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        vt = torch.from_numpy(vs[s]).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(out[s], ref.reshape(Hq, D).numpy(), rtol=0, atol=1e-12)
    assert werr.max() < 1e-12


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    q, ks, vs = _case(rng, 3, 8, 2, 64, [1, 1, 1])
    out = oracle.decode_attention(q, ks, vs, 0.125)
    for s in range(3):
        for h in range(8):
            assert np.array_equal(out[s, h], vs[s][0, h // 4])


def test_constant_values_give_the_constant():
    rng = np.random.default_rng(2)
    q, ks, _ = _case(rng, 2, 4, 4, 64, [37, 300])
    vs = [np.full((k.shape[0], 4, 64), 2.5) for k in ks]
    out = oracle.decode_attention(q, ks, vs, 0.3)
    np.testing.assert_allclose(out, 2.5, rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(3)
    _, ks, vs = _case(rng, 2, 8, 4, 64, [10, 77])
    q = np.zeros((2, 8, 64))
    out = oracle.decode_attention(q, ks, vs, 1.0)
    for s in range(2):
        for h in range(8):
            np.testing.assert_allclose(out[s, h], vs[s][:, h // 2].mean(axis=0), rtol=0, atol=1e-13)


def test_two_tokens_closed_form():
    """Softmax of two scores is a logistic function of their difference."""
    rng = np.random.default_rng(4)
    q, ks, vs = _case(rng, 1, 2, 1, 64, [2])
    scale = 0.37
    out = oracle.decode_attention(q, ks, vs, scale)
    for h in range(2):
        d = scale * (q[0, h] @ ks[0][0, 0] - q[0, h] @ ks[0][1, 0])
        w0 = expit(d)
        ref = w0 * vs[0][0, 0] + (1 - w0) * vs[0][1, 0]
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-13)


def test_large_scores_are_stable_and_pick_the_winner():
    rng = np.random.default_rng(5)
    q, ks, vs = _case(rng, 1, 1, 1, 64, [50])
    ks[0][17, 0] = 40.0 * q[0, 0] / np.linalg.norm(q[0, 0])  # dominant key
    out = oracle.decode_attention(q, ks, vs, 1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], vs[0][17, 0], rtol=0, atol=1e-9)


def test_gqa_head_mapping_is_consecutive_groups():
    """Query head h reads KV head h // (Hq / Hkv)."""
    rng = np.random.default_rng(6)
    q, ks, _ = _case(rng, 1, 8, 4, 64, [9])
    vs = [np.broadcast_to(np.arange(4.0).reshape(1, 4, 1), (9, 4, 64)).copy()]
    out = oracle.decode_attention(q, ks, vs, 0.2)
    for h in range(8):
        np.testing.assert_allclose(out[0, h], h // 2, rtol=0, atol=1e-13)


def test_token_order_does_not_matter():
    rng = np.random.default_rng(7)
    q, ks, vs = _case(rng, 1, 4, 2, 64, [61])
    perm = rng.permutation(61)
    a = oracle.decode_attention(q, ks, vs, 0.125)
    b = oracle.decode_attention(q, [ks[0][perm]], [vs[0][perm]], 0.125)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_key_shift_invariance():
    """Adding one vector to every key shifts all scores of a query by the same
    amount, which the softmax removes."""
    rng = np.random.default_rng(8)
    q, ks, vs = _case(rng, 1, 2, 1, 64, [30])
    shift = _rand(rng, 64) * 3
    a = oracle.decode_attention(q, ks, vs, 0.125)
    b = oracle.decode_attention(q, [ks[0] + shift], vs, 0.125)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(9)
    q, ks, vs = _case(rng, 2, 4, 4, 64, [0, 5])
    out = oracle.decode_attention(q, ks, vs, 0.125)
    assert np.array_equal(out[0], np.zeros((4, 64)))
    assert np.all(np.isfinite(out[1]))


# ---------------------------------------------------------------------------
# Cache write and block copy semantics
# ---------------------------------------------------------------------------
def test_cache_write_places_tokens_and_skips_negative_slots():
    B, NB, Hkv, D = 16, 6, 2, 8
    sentinel = -777.0
    kc = np.full((NB, Hkv, B, D), sentinel)
    vc = np.full((NB, Hkv, B, D), sentinel)
    kn = np.arange(3 * Hkv * D, dtype=np.float64).reshape(3, Hkv, D)
    vn = -kn
    slots = [5 * B + 3, -1, 0]
    oracle.kv_cache_write(kc, vc, kn, vn, slots, B)
    assert np.array_equal(kc[5, :, 3, :], kn[0]) and np.array_equal(vc[5, :, 3, :], vn[0])
    assert np.array_equal(kc[0, :, 0, :], kn[2]) and np.array_equal(vc[0, :, 0, :], vn[2])
    touched = np.zeros((NB, B), bool)
    touched[5, 3] = touched[0, 0] = True
    for blk in range(NB):
        for off in range(B):
            if not touched[blk, off]:
                assert np.all(kc[blk, :, off] == sentinel) and np.all(vc[blk, :, off] == sentinel)


def test_block_copy_copies_whole_blocks_in_every_layer():
    rng = np.random.default_rng(10)
    ks = [_rand(rng, 5, 2, 4, 8) for _ in range(3)]
    vs = [_rand(rng, 5, 2, 4, 8) for _ in range(3)]
    before_k = [k.copy() for k in ks]
    oracle.block_copy(ks, vs, [[1, 3], [4, 0]])
    for layer in range(3):
        assert np.array_equal(ks[layer][3], before_k[layer][1])
        assert np.array_equal(ks[layer][0], before_k[layer][4])
        for b in (1, 2, 4):
            assert np.array_equal(ks[layer][b], before_k[layer][b])
        assert np.array_equal(vs[layer][3], vs[layer][1])


# ---------------------------------------------------------------------------
# Waste versus block size on a continuous-batching length mix
# ---------------------------------------------------------------------------
def test_waste_grows_with_block_size_and_stays_small_at_16():
    from paged_kv_cache_279_gb300 import workloads as wl
    lens = wl.draw_lengths(wl.MIXED_BF16, seed=0)
    w8, w16, w32 = (oracle.paged_waste_fraction(lens, b) for b in (8, 16, 32))
    assert w8 < w16 < w32
    assert w16 < 0.05  # "under 4%" is quoted for real traffic; this mix gives ~3%
    # every sequence wastes less than one block
    for L in lens:
        assert oracle.blocks_needed(L, 16) * 16 - L < 16
    assert oracle.preallocation_waste_fraction(lens, 4096) > 0.9
