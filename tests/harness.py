"""Test-side helpers: place contiguous per-sequence K/V into a paged pool on
the host, move things to the GPU, and compare GPU results with the oracle under
the stated tolerances.  Nothing here is used by the library."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl

BF16_MAX_ABS = 1e-2
BF16_MEAN_ABS = 1e-3
F32_MAX_ABS = 1e-5


def token_slots(table_row, length, block_size):
    """Slots of positions 0..length-1: logical block p // B of the table, offset p % B."""
    pos = np.arange(length, dtype=np.int64)
    return np.asarray(table_row, dtype=np.int64)[pos // block_size] * block_size + pos % block_size


def place_paged(k_seqs, v_seqs, tables, num_blocks, block_size, dtype, fill=float("nan")):
    """Host pools [NB, Hkv, B, D] holding each sequence's tokens at the slots its
    table names; every other slot holds ``fill``."""
    Hkv, D = k_seqs[0].shape[1], k_seqs[0].shape[2]
    kc = torch.full((num_blocks, Hkv, block_size, D), fill, dtype=dtype)
    vc = torch.full_like(kc, fill)
    for s, (k, v) in enumerate(zip(k_seqs, v_seqs)):
        L = k.shape[0]
        if L == 0:
            continue
        slots = torch.from_numpy(token_slots(tables[s], L, block_size))
        kc[slots // block_size, :, slots % block_size, :] = k
        vc[slots // block_size, :, slots % block_size, :] = v
    return kc, vc


def make_decode_case(shape: wl.DecodeShape, lens, seed=0, num_blocks=None, fill=float("nan"),
                     table_seed=None, extra_blocks=0):
    """Contiguous data (for the oracle) and a randomly placed paged pool (for the GPU)."""
    lens = [int(x) for x in lens]
    B = shape.block_size
    counts = [-(-L // B) for L in lens]
    NB = num_blocks or max(1, sum(counts) + extra_blocks)
    maxB = max(1, max(counts) if counts else 1)
    tables = wl.random_block_tables(counts, NB, maxB, seed if table_seed is None else table_seed)
    ks, vs = zip(*[wl.draw_seq_kv(shape, seed, s, L) for s, L in enumerate(lens)])
    q = wl.draw_query(shape, seed, num_seqs=len(lens))
    kc, vc = place_paged(ks, vs, tables, NB, B, shape.dtype, fill)
    return dict(q=q, ks=list(ks), vs=list(vs), tables=tables, lens=lens, kc=kc, vc=vc, NB=NB,
                maxB=maxB)


def run_decode(case, shape, partition_size=0, max_seq_len=None, device="cuda"):
    q = case["q"].to(device)
    out = torch.empty_like(q)
    maxL = max_seq_len if max_seq_len is not None else max(1, max(case["lens"]))
    pkv.paged_attention_decode(
        out, q, case["kc_dev"] if "kc_dev" in case else case["kc"].to(device),
        case["vc_dev"] if "vc_dev" in case else case["vc"].to(device),
        torch.from_numpy(case["tables"]).to(device),
        torch.tensor(case["lens"], dtype=torch.int32, device=device), shape.scale, maxL,
        partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def oracle_out(case, shape, seqs=None):
    idx = range(len(case["lens"])) if seqs is None else seqs
    q = case["q"].float().numpy()[list(idx)]
    ks = [case["ks"][s].float().numpy() for s in idx]
    vs = [case["vs"][s].float().numpy() for s in idx]
    return oracle.decode_attention(q, ks, vs, shape.scale)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def assert_bf16_close(got: torch.Tensor, ref: np.ndarray, what=""):
    """max-abs 1e-2 and mean-abs 1e-3 against the fp64 oracle; where |ref| >= 4
    one bf16 rounding alone can exceed 1e-2, so there the bound is one bf16 ulp."""
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    big = np.abs(ref) >= 4.0
    small_err = err[~big]
    assert small_err.size == 0 or small_err.max() <= BF16_MAX_ABS, f"{what}: max abs err {small_err.max():.3e}"
    if big.any():
        assert np.all(err[big] <= bf16_ulp(ref[big])), f"{what}: large-value error above one ulp"
    assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def assert_f32_close(got: torch.Tensor, ref: np.ndarray, what=""):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    assert err.max() <= F32_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    return float(err.max()), float(err.mean())


def bits(t: torch.Tensor) -> torch.Tensor:
    """Integer view for bit-exact comparisons (NaN payloads included)."""
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def build_beam_pool(shape, shared, num_prompts, width, divergent, seed=2, append_last=False):
    """Beam search through the library's allocator: `num_prompts` prompts of
    `shared` tokens, each forked into `width` beams; beam b then produces
    divergent[b] tokens (copy-on-write pairs executed with block_copy, tokens
    stored with kv_cache_write).  With append_last, every beam's last token is
    left unwritten (for a decode-and-append call) and returned as k_new/v_new.
    Returns a dict with the pool, allocator, tables, lengths and the contiguous
    K/V of every beam (prompt followed by its own tokens)."""
    B, Hkv, D = shape.block_size, shape.num_kv_heads, shape.head_dim
    div = [int(d) for d in divergent]
    nbeams = num_prompts * width
    NB = num_prompts * (-(-shared // B) + 1) + sum(-(-d // B) + 1 for d in div) + 64
    alloc = pkv.BlockAllocator(NB, B)
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=shape.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    prefix = [wl.draw_seq_kv(shape, seed, p, shared) for p in range(num_prompts)]
    own = [wl.draw_seq_kv(shape, seed + 1, b, div[b]) for b in range(nbeams)]
    for p in range(num_prompts):
        assert alloc.add_seq(p * width, shared) == 0
        slots = torch.from_numpy(alloc.slots(p * width, 0, shared)).cuda()
        pkv.kv_cache_write(prefix[p][0].cuda(), prefix[p][1].cuda(), kc, vc, slots)
        for c in range(1, width):
            assert alloc.fork(p * width, p * width + c) == 0
    copies = 0
    for t in range(max(div) if div else 0):
        beams = [b for b in range(nbeams) if div[b] > t]
        st, slots, pairs = alloc.append_slots(beams)
        assert st == 0
        if len(pairs):
            copies += len(pairs)
            pkv.block_copy([kc], [vc], torch.from_numpy(np.ascontiguousarray(pairs)).cuda())
        keep = [i for i, b in enumerate(beams) if not (append_last and t == div[b] - 1)]
        if keep:
            kn = torch.stack([own[beams[i]][0][t] for i in keep]).cuda()
            vn = torch.stack([own[beams[i]][1][t] for i in keep]).cuda()
            pkv.kv_cache_write(kn, vn, kc, vc, torch.from_numpy(slots[keep]).cuda())
    seqs = list(range(nbeams))
    cap = max(len(alloc.block_table(s)) for s in seqs)
    tables, lens = alloc.block_tables(seqs, cap=cap)
    ks = [torch.cat([prefix[b // width][0], own[b][0]]) for b in seqs]
    vs = [torch.cat([prefix[b // width][1], own[b][1]]) for b in seqs]
    k_new = torch.stack([own[b][0][div[b] - 1] if div[b] else torch.zeros(Hkv, D, dtype=shape.dtype)
                         for b in seqs])
    v_new = torch.stack([own[b][1][div[b] - 1] if div[b] else torch.zeros(Hkv, D, dtype=shape.dtype)
                         for b in seqs])
    return dict(kc=kc, vc=vc, alloc=alloc, tables=tables, lens=lens, ks=ks, vs=vs, copies=copies,
                seqs=seqs, k_new=k_new, v_new=v_new)
