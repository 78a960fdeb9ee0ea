"""Prefix caching on the GPU: requests whose prompts start with the same
tokens share the pool blocks of that prefix (block_allocator_add_seq_cached),
only the uncached tail of each prompt is written, and the decode (plain and
grouped) equals the fp64 oracle on every request's full context.

Synthetic K/V: the K and V of position p depend on the token prefix up to p
(as a causal model's would), so a cached block holds exactly what the new
request would have computed."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import assert_bf16_close

pytestmark = pytest.mark.gpu


def kv_at(tokens, p, Hkv, D):
    seed = zlib.crc32(np.asarray(tokens[:p + 1], dtype=np.int32).tobytes())
    x = np.random.default_rng(seed).standard_normal((2, Hkv, D)).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def test_prefix_cached_pool_decodes_like_the_oracle():
    B, Hq, Hkv, D = 16, 32, 8, 128
    shape = wl.DecodeShape("prefix_cache", 0, Hq, Hkv, D, B, torch.bfloat16)
    rng = np.random.default_rng(7)
    systems = [rng.integers(0, 50, n).tolist() for n in (100, 256, 40)]
    reqs = []
    for r in range(12):
        base = systems[r % 3]
        reqs.append(base + rng.integers(0, 50, int(rng.integers(0, 80))).tolist())
    NB = 200
    alloc = pkv.BlockAllocator(NB, B)
    model = oracle.BlockAllocatorModel(NB, B)
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    full_kv = {}

    def admit(r, toks):
        st, cached = alloc.add_seq_cached(r, toks)
        assert (st, cached) == model.add_seq_cached(r, toks)
        kv = torch.stack([kv_at(toks, p, Hkv, D) for p in range(len(toks))])  # [n, 2, Hkv, D]
        full_kv[r] = kv
        if len(toks) > cached:  # only the uncached tail is written
            slots = torch.from_numpy(alloc.slots(r, cached, len(toks) - cached)).cuda()
            pkv.kv_cache_write(kv[cached:, 0].cuda(), kv[cached:, 1].cuda(), kc, vc, slots)
        return cached

    cached = [admit(r, t) for r, t in enumerate(reqs)]
    assert sum(cached) > 0 and alloc.cache_stats()["hits"] > 0

    def check(seqs, grouped):
        order = sorted(seqs, key=lambda r: (reqs_all[r][:B], r))  # requests of one prompt side by side
        cap = max(len(alloc.block_table(r)) for r in order)
        tables, lens = alloc.block_tables(order, cap=cap)
        q = wl.draw_query(shape, 3, num_seqs=len(order)).cuda()
        out = torch.full_like(q, float("nan"))
        if grouped:
            offs, pre = alloc.prefix_groups(order)
            pkv.paged_attention_decode_grouped(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                                               torch.from_numpy(lens).cuda(), torch.from_numpy(offs).cuda(),
                                               torch.from_numpy(pre).cuda(), shape.scale, int(lens.max()))
        else:
            pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                                       torch.from_numpy(lens).cuda(), shape.scale, int(lens.max()))
        torch.cuda.synchronize()
        ks = [full_kv[r][:, 0].float().numpy() for r in order]
        vs = [full_kv[r][:, 1].float().numpy() for r in order]
        ref = oracle.decode_attention(q.float().cpu().numpy(), ks, vs, shape.scale)
        assert_bf16_close(out, ref, f"prefix cache grouped={grouped}")

    reqs_all = dict(enumerate(reqs))
    pkv.read_device_errors(clear=True)
    check(list(range(12)), grouped=False)
    check(list(range(12)), grouped=True)
    # free half the requests: their cached blocks stay (evictable) and are found again
    for r in range(0, 12, 2):
        assert alloc.free_seq(r) == model.free_seq(r)
    assert alloc.cache_stats()["evictable_blocks"] == model.cache_stats()["evictable_blocks"]
    more = {}
    for r in range(12, 18):
        toks = systems[r % 3] + rng.integers(0, 50, int(rng.integers(1, 40))).tolist()
        reqs_all[r] = toks
        more[r] = admit(r, toks)
    assert sum(more.values()) > 0
    live = [r for r in reqs_all if r % 2 == 1 or r >= 12]
    check(live, grouped=False)
    check(live, grouped=True)
    assert pkv.read_device_errors() == 0
