"""Split edge cases of the two kernels that cut a tile list into equal shares.

Both kernels charge each context a few tiles of fixed cost in that list (empty
lead tiles in the balanced decode kernel, virtual tiles in the rows kernel), so
a share can start or end inside a context's charge.  The cases below are found
on the host with the library's own split arithmetic (its diagnostic exports)
and then run on the GPU against the fp64 oracle:

* balanced decode: a share ends inside a split segment's lead tiles, so the
  warp that merges the segment (the one holding its first laid-out tile) holds
  none of its real tiles and merges an empty piece of its own;
* rows kernel (multi-token): a share ends inside a split context's virtual
  tiles, so that share publishes no piece for it and the merge falls to the
  share holding its first real tile.

Few enough tiles that the share count (total / minimum share) stays below any
grid the launch could use, so the host knows the split without the device.
"""
import math

import numpy as np
import pytest
import torch

from oracle.multi_token import multi_token_attention
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import _lib, workloads as wl
from harness import assert_bf16_close, make_decode_case, oracle_out, place_paged, run_decode


def lib():
    return _lib.load()


def _boundaries(T, parts):
    return [w * T // parts for w in range(1, parts)]


def _edge(seg, parts, lead):
    """Index of a context (laid-out sizes `seg`) split between shares, with a
    share starting inside its first `lead` tiles; None if there is none."""
    T = sum(seg)
    bounds = _boundaries(T, parts)
    start = 0
    for c, n in enumerate(seg):
        if n > 0:
            inside = any(start < b <= start + lead for b in bounds)  # a share starts in its charge
            split = any(start < b < start + n for b in bounds)
            if inside and split:
                return c
        start += n
    return None


def balanced_edge_case():
    """(lens, context index) for the balanced decode kernel, 16-token tiles, 8 kv heads."""
    L = lib()
    lead = L.pkv_balanced_segment_tiles(1) - 1
    for seed in range(5000):
        rng = np.random.default_rng(seed)
        lens = [int(x) for x in rng.integers(1, 1200, int(rng.integers(3, 9)))]
        seg = [L.pkv_balanced_segment_tiles(math.ceil(x / 16)) for x in lens for _ in range(8)]
        parts = L.pkv_balanced_split_parts(sum(seg), max(seg), max(lens), 10 ** 6)
        if not 2 <= parts < 600:  # below any grid's warp count: the split is the host's
            continue
        c = _edge(seg, parts, lead)
        if c is not None:
            return lens, c
    return None


def rows_edge_case():
    """(lens, qlens, context index) for the rows kernel's multi-token calls:
    4 query heads per kv head (32 queries per context), 8 kv heads, 64-key tiles."""
    L = lib()
    lead = L.pkv_rows_context_tiles(1) - 1
    for seed in range(5000):
        rng = np.random.default_rng(10_000 + seed)
        S = int(rng.integers(2, 6))
        qlens = [int(x) for x in rng.integers(1, 33, S)]
        lens = [int(max(q, x)) for q, x in zip(qlens, rng.integers(1, 500, S))]
        seg = [L.pkv_rows_context_tiles(math.ceil(x / 64)) for x in lens for _ in range(8)]
        parts = L.pkv_rows_split_parts(sum(seg), 10 ** 6)
        if not 2 <= parts < 100:  # below any GPU's SM count: the split is the host's
            continue
        c = _edge(seg, parts, lead)
        if c is not None:
            return lens, qlens, c
    return None


def test_edge_cases_exist():
    """The host finds both edge cases (no GPU needed)."""
    assert balanced_edge_case() is not None
    assert rows_edge_case() is not None


@pytest.mark.gpu
def test_balanced_merge_of_a_segment_whose_merger_holds_only_lead_tiles():
    lens, _ = balanced_edge_case()
    shape = wl.DecodeShape("edge", len(lens), 32, 8, 128, 16, torch.bfloat16)
    case = make_decode_case(shape, lens, seed=31)
    pkv.read_device_errors(clear=True)
    out = run_decode(case, shape, partition_size=0, max_seq_len=max(lens))
    assert_bf16_close(out.cpu(), oracle_out(case, shape), "balanced split, merger on lead tiles only")
    assert pkv.read_device_errors() == 0


@pytest.mark.gpu
def test_rows_context_whose_share_ends_in_its_virtual_tiles():
    lens, qlens, _ = rows_edge_case()
    Hq, Hkv, D, B = 32, 8, 128, 16
    shape = wl.DecodeShape("edge_mt", len(lens), Hq, Hkv, D, B, torch.bfloat16)
    counts = [-(-x // B) for x in lens]
    NB = sum(counts) + 3
    tables = wl.random_block_tables(counts, NB, max(counts), 41)
    ks, vs = zip(*[wl.draw_seq_kv(shape, 40, s, x) for s, x in enumerate(lens)])
    kc, vc = place_paged(ks, vs, tables, NB, B, torch.bfloat16)
    T = sum(qlens)
    q = wl.draw_normal((T, Hq, D), torch.bfloat16, wl.sub_seed(40, 20))
    starts = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    dev = "cuda"
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    pkv.read_device_errors(clear=True)
    pkv.paged_attention_multi_token(out, q.to(dev), kc.to(dev), vc.to(dev), torch.from_numpy(tables).to(dev),
                                    torch.tensor(lens, dtype=torch.int32, device=dev),
                                    torch.from_numpy(starts).to(dev), shape.scale, max(qlens), max(lens))
    torch.cuda.synchronize()
    qs = [q[starts[s]:starts[s + 1]].float().numpy() for s in range(len(lens))]
    ref = multi_token_attention(qs, [k.float().numpy() for k in ks], [v.float().numpy() for v in vs], shape.scale)
    assert_bf16_close(out.cpu(), np.concatenate(ref, axis=0), "rows split, share ending in virtual tiles")
    assert pkv.read_device_errors() == 0
