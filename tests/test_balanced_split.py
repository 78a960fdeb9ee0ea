"""Invariants of the balanced split that the attention kernel's in-kernel merge
relies on, checked on the library's own split arithmetic (the share sizing and
share ownership the kernel runs, exported as host diagnostics) over many
random workloads:

* every context (sequence, kv head) is cut into at most `slots` pieces, the
  partial slots the workspace holds per (sequence, head);
* a share cuts at most its first and its last context (so a warp stores at most
  two partials);
* a split context's first tile lies in exactly one share, and that context is
  the last one of the share (its warp merges it after the share);
* the other pieces' slots j = share - first share are distinct and lie in
  [1, pieces).
Both tile sizes (16 tokens, 32 for the FP8 cache) and grids of one or several
CTAs per SM are covered.  No GPU needed.
"""
import math
import random

import pytest

from paged_kv_cache_279_gb300 import _lib


def lib():
    return _lib.load()


def split(lens, hkv, tile, max_seq_len, warps):
    """Laid-out tiles per context (the real ones after the library's lead
    tiles), total T, number of shares `parts` (from the library)."""
    seg = [lib().pkv_balanced_segment_tiles(math.ceil(L / tile)) for L in lens for _ in range(hkv)]
    T = sum(seg)
    slots = lib().pkv_balanced_slots(max_seq_len)
    parts = lib().pkv_balanced_split_parts(T, max(seg) if seg else 0, max_seq_len, warps)
    return seg, T, parts, slots


def share_owner(t, T, parts):
    return lib().pkv_balanced_share_owner(t, T, parts)


def test_slots_and_bad_arguments():
    L = lib()
    lead = L.pkv_balanced_segment_tiles(1) - 1
    assert lead >= 0 and L.pkv_balanced_segment_tiles(0) == 0 and L.pkv_balanced_segment_tiles(-1) == -1
    assert all(L.pkv_balanced_segment_tiles(n) == n + lead for n in (1, 2, 17, 1000))
    assert L.pkv_balanced_slots(0) == 1 and L.pkv_balanced_slots(256) == 2 and L.pkv_balanced_slots(257) == 3
    assert L.pkv_balanced_slots(-1) == -1
    assert L.pkv_balanced_split_parts(0, 0, 100, 8) == 0
    assert L.pkv_balanced_split_parts(-1, 0, 100, 8) == -1
    assert L.pkv_balanced_split_parts(10, 10, 100, 0) == -1
    assert L.pkv_balanced_share_owner(5, 5, 1) == -1
    # one share: every tile belongs to share 0; T shares: tile t to share t
    assert all(L.pkv_balanced_share_owner(t, 7, 1) == 0 for t in range(7))
    assert all(L.pkv_balanced_share_owner(t, 7, 7) == t for t in range(7))


@pytest.mark.parametrize("seed", range(40))
def test_split_invariants(seed):
    rnd = random.Random(seed)
    tile = rnd.choice([16, 32])
    hkv = rnd.choice([1, 2, 4, 8])
    S = rnd.choice([1, 2, 5, 64, 256, 700])
    max_len = rnd.choice([64, 300, 2048, 16000])
    lens = [rnd.choice([0, 1, rnd.randint(1, max_len)]) if rnd.random() < 0.2 else rnd.randint(1, max_len)
            for _ in range(S)]
    warps = rnd.choice([152 * 3 * 4, 152 * 4, 16, 1])
    seg, T, parts, slots = split(lens, hkv, tile, max_len, warps)
    if T == 0:
        assert parts == 0
        return
    assert 1 <= parts <= warps
    bounds = [(g * T // parts, (g + 1) * T // parts) for g in range(parts)]
    assert all(hi > lo for lo, hi in bounds)                        # no empty share
    assert all(share_owner(t, T, parts) == g for g, (lo, hi) in enumerate(bounds) for t in (lo, hi - 1))
    starts = [0]
    for n in seg:
        starts.append(starts[-1] + n)
    partial_per_share = [0] * parts
    for c, n in enumerate(seg):
        if n == 0:
            continue
        a, b = starts[c], starts[c] + n
        w0, w1 = share_owner(a, T, parts), share_owner(b - 1, T, parts)
        pieces = w1 - w0 + 1
        assert pieces <= slots
        if pieces == 1:
            continue
        for w in range(w0, w1 + 1):
            partial_per_share[w] += 1
        # the merger's share ends inside the context: it is that share's last segment
        assert bounds[w0][1] < b and bounds[w0][0] <= a
        slots_used = [w - w0 for w in range(w0 + 1, w1 + 1)]
        assert sorted(set(slots_used)) == slots_used and all(1 <= j < pieces for j in slots_used)
    assert max(partial_per_share) <= 2


def test_gqa_workload_shape():
    """The GQA decode workload (64 contexts of U[64, 2048] tokens, 8 kv heads,
    456 CTAs x 4 warps): shares of ~18 tiles, at most 9 pieces per context."""
    rnd = random.Random(0)
    lens = [rnd.randint(64, 2048) for _ in range(64)]
    seg, T, parts, slots = split(lens, 8, 16, 2048 + 64, 152 * 3 * 4)
    assert parts == 152 * 3 * 4 and 15 <= T / parts <= 22
    worst = max(share_owner(s + n - 1, T, parts) - share_owner(s, T, parts) + 1
                for s, n in zip([sum(seg[:i]) for i in range(len(seg))], seg))
    assert worst <= slots
