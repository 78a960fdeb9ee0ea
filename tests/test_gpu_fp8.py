"""GPU parity of the FP8 (E4M3) KV cache against the oracle.

kv_cache_write_fp8 must produce the oracle's codes bit for bit (the rounding
decision is taken in float32 on both sides: the IEEE quotient x / scale, then
nearest-even E4M3 with saturation).  paged_attention_decode_fp8 must match the
fp64 oracle's attention over the dequantised cache (code value x scale)
within the bf16 output tolerance.  Slots that no sequence owns hold NaN codes,
so any read of a masked token shows up as a non-finite output.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_e4m3 as f8
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import assert_bf16_close, token_slots

pytestmark = pytest.mark.gpu

D = 128
K_SCALE, V_SCALE = 1.0 / 32, 1.0 / 40


def _pool_with_codes(lens, Hkv, B, seed, extra_blocks=3, fill=0x7F):
    """Random E4M3 codes per sequence placed at random physical blocks: K rows
    at [blk, h, off, :], V columns at [blk, h, :, off]; unowned slots = fill."""
    counts = [-(-L // B) for L in lens]
    NB = max(1, sum(counts) + extra_blocks)
    maxB = max(1, max(counts))
    tables = wl.random_block_tables(counts, NB, maxB, seed + 1)
    kc = np.full((NB, Hkv, B, D), fill, dtype=np.uint8)
    vc = np.full((NB, Hkv, D, B), fill, dtype=np.uint8)
    kq, vq = [], []
    for s, L in enumerate(lens):
        k = wl.draw_e4m3_codes((L, Hkv, D), wl.sub_seed(seed, 10, s))
        v = wl.draw_e4m3_codes((L, Hkv, D), wl.sub_seed(seed, 11, s))
        kq.append(k)
        vq.append(v)
        if L:
            slots = token_slots(tables[s], L, B)
            kc[slots // B, :, slots % B, :] = k
            vc[slots // B, :, :, slots % B] = v  # advanced indices first: [L, Hkv, D]
    return dict(kc=kc, vc=vc, kq=kq, vq=vq, tables=tables, NB=NB)


def _run(pool, q, lens, scale, max_seq_len=None):
    dev = "cuda"
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    pkv.paged_attention_decode_fp8(
        out, q.to(dev), torch.from_numpy(pool["kc"]).to(dev), torch.from_numpy(pool["vc"]).to(dev),
        torch.from_numpy(pool["tables"]).to(dev), torch.tensor(lens, dtype=torch.int32, device=dev),
        scale, K_SCALE, V_SCALE, max_seq_len or max(1, max(lens)))
    torch.cuda.synchronize()
    return out.cpu()


def _oracle(pool, q, scale):
    ks = [f8.dequantize(k, K_SCALE) for k in pool["kq"]]
    vs = [f8.dequantize(v, V_SCALE) for v in pool["vq"]]
    return oracle.decode_attention(q.float().numpy(), ks, vs, scale)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (64, 8), (12, 4)])
@pytest.mark.parametrize("B", [16, 32])
def test_decode_fp8_matches_oracle(Hq, Hkv, B):
    lens = [1, 17, 100, 0, 16, 2048, 513, 33, 255, 1000]
    shape = wl.DecodeShape("fp8", len(lens), Hq, Hkv, D, B, torch.bfloat16)
    pool = _pool_with_codes(lens, Hkv, B, seed=Hq * 7 + B)
    q = wl.draw_query(shape, seed=B + Hq)
    got = _run(pool, q, lens, shape.scale)
    assert_bf16_close(got, _oracle(pool, q, shape.scale), f"fp8 decode Hq={Hq} Hkv={Hkv} B={B}")
    assert torch.all(got[3] == 0)  # empty context: zero rows
    assert pkv.read_device_errors() == 0


def test_decode_fp8_full_gqa_workload():
    """The GQA decode workload (64 sequences, lengths uniform in [64, 2048],
    32 query / 8 KV heads, block 16) on an FP8 cache, every output checked."""
    shape = wl.GQA_BF16
    lens = wl.draw_lengths(shape, seed=3).tolist()
    pool = _pool_with_codes(lens, shape.num_kv_heads, shape.block_size, seed=3,
                            extra_blocks=sum(-(-L // 16) for L in lens) // 10)
    q = wl.draw_query(shape, seed=3)
    got = _run(pool, q, lens, shape.scale)
    assert_bf16_close(got, _oracle(pool, q, shape.scale), "fp8 GQA workload")


def test_decode_fp8_long_contexts_and_permutation_invariance():
    lens = [16000, 12345, 7]
    Hkv, B = 8, 16
    shape = wl.DecodeShape("fp8_long", len(lens), 32, Hkv, D, B, torch.bfloat16)
    pool = _pool_with_codes(lens, Hkv, B, seed=21)
    q = wl.draw_query(shape, seed=21)
    got = _run(pool, q, lens, shape.scale)
    assert_bf16_close(got, _oracle(pool, q, shape.scale), "fp8 long contexts")
    # move every block to another physical id: bit-identical output
    perm = np.random.default_rng(5).permutation(pool["NB"])
    moved = dict(pool)
    moved["kc"] = np.empty_like(pool["kc"])
    moved["vc"] = np.empty_like(pool["vc"])
    moved["kc"][perm] = pool["kc"]
    moved["vc"][perm] = pool["vc"]
    t = pool["tables"]
    moved["tables"] = np.where(t >= 0, perm[np.maximum(t, 0)], t).astype(np.int32)
    assert torch.equal(_run(moved, q, lens, shape.scale).view(torch.int16), got.view(torch.int16))


def test_decode_fp8_single_token_returns_its_value():
    lens = [1, 1]
    Hkv, B = 2, 16
    shape = wl.DecodeShape("fp8_one", 2, 8, Hkv, D, B, torch.bfloat16)
    pool = _pool_with_codes(lens, Hkv, B, seed=4)
    q = wl.draw_query(shape, seed=4)
    got = _run(pool, q, lens, shape.scale).double().numpy()
    for s in range(2):
        v = f8.dequantize(pool["vq"][s][0], V_SCALE)  # [Hkv, D]
        want = np.repeat(v, 4, axis=0)
        assert np.all(np.abs(got[s] - want) <= np.maximum(np.abs(want) * 2.0 ** -8, 1e-6))


def _bf16_tokens(T, Hkv, seed):
    k = wl.draw_normal((T, Hkv, D), torch.bfloat16, seed)
    v = wl.draw_normal((T, Hkv, D), torch.bfloat16, seed + 1)
    return k, v


@pytest.mark.parametrize("B", [16, 32])
def test_write_fp8_bit_exact(B):
    T, Hkv, NB = 300, 8, 40
    k, v = _bf16_tokens(T, Hkv, 31 + B)
    # specials: ties, subnormal-range values, saturation, zeros of both signs
    specials = torch.tensor([1.0625, 1.1875, 2.0 ** -10 / 32, -0.0, 0.0, 432.0 / 32, 1e4, -1e4,
                             float("inf"), float("-inf"), 1.5 * 2.0 ** -9 / 32, 7.5 * 2.0 ** -9 / 32],
                            dtype=torch.bfloat16)
    k[0, 0, :specials.numel()] = specials
    v[1, 3, -specials.numel():] = specials
    rng = np.random.default_rng(B)
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[::17] = -1  # padding tokens
    kc0 = wl.draw_e4m3_codes((NB, Hkv, B, D), 91)
    vc0 = wl.draw_e4m3_codes((NB, Hkv, D, B), 92)
    kc, vc = torch.from_numpy(kc0).cuda(), torch.from_numpy(vc0).cuda()
    pkv.kv_cache_write_fp8(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda(), K_SCALE, V_SCALE)
    torch.cuda.synchronize()
    want_k, want_v = kc0.copy(), vc0.copy()
    f8.kv_cache_write_fp8(want_k, want_v, k.float().numpy(), v.float().numpy(), slots, B, K_SCALE, V_SCALE)
    assert np.array_equal(kc.cpu().numpy(), want_k)
    assert np.array_equal(vc.cpu().numpy(), want_v)
    assert pkv.read_device_errors() == 0


def test_write_fp8_nan_gives_a_nan_code_and_bad_slots_are_flagged():
    Hkv, B, NB = 2, 16, 4
    k, v = _bf16_tokens(3, Hkv, 7)
    k[0, 1, 5] = float("nan")
    kc = torch.zeros((NB, Hkv, B, D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros((NB, Hkv, D, B), dtype=torch.uint8, device="cuda")
    pkv.read_device_errors()
    slots = torch.tensor([3, NB * B + 5, 40], dtype=torch.int64, device="cuda")
    pkv.kv_cache_write_fp8(k.cuda(), v.cuda(), kc, vc, slots, 0.5, 0.5)
    torch.cuda.synchronize()
    assert (int(kc[0, 1, 3, 5]) & 0x7F) == 0x7F
    assert pkv.read_device_errors() & 4  # PKV_DEVERR_SLOT
    # the out-of-range token wrote nothing: only tokens 0 and 2 are present
    assert int((kc != 0).sum()) <= 2 * Hkv * D


def test_write_then_decode_end_to_end():
    """bf16 K/V written through kv_cache_write_fp8, attended by
    paged_attention_decode_fp8; the oracle quantises the same bf16 values
    itself.  Also reports the quantisation error against bf16 attention."""
    lens = [300, 64, 1, 1777]
    Hq, Hkv, B = 32, 8, 16
    shape = wl.DecodeShape("fp8_e2e", len(lens), Hq, Hkv, D, B, torch.bfloat16)
    counts = [-(-L // B) for L in lens]
    NB = sum(counts) + 5
    tables = wl.random_block_tables(counts, NB, max(counts), 77)
    ks, vs = zip(*[wl.draw_seq_kv(shape, 77, s, L) for s, L in enumerate(lens)])
    slots = np.concatenate([token_slots(tables[s], L, B) for s, L in enumerate(lens)])
    kc = torch.full((NB, Hkv, B, D), 0x7F, dtype=torch.uint8, device="cuda")
    vc = torch.full((NB, Hkv, D, B), 0x7F, dtype=torch.uint8, device="cuda")
    pkv.kv_cache_write_fp8(torch.cat(ks).cuda(), torch.cat(vs).cuda(), kc, vc,
                           torch.from_numpy(slots).cuda(), K_SCALE, V_SCALE)
    q = wl.draw_query(shape, 77)
    out = torch.empty((len(lens), Hq, D), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_decode_fp8(out, q.cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                                   torch.tensor(lens, dtype=torch.int32, device="cuda"), shape.scale,
                                   K_SCALE, V_SCALE, max(lens))
    torch.cuda.synchronize()
    kd = [f8.dequantize(f8.quantize(k.float().numpy(), K_SCALE), K_SCALE) for k in ks]
    vd = [f8.dequantize(f8.quantize(v.float().numpy(), V_SCALE), V_SCALE) for v in vs]
    ref = oracle.decode_attention(q.float().numpy(), kd, vd, shape.scale)
    assert_bf16_close(out.cpu(), ref, "fp8 write + decode")
    # the price of the 8-bit cache (not a parity bound): distance to bf16 attention
    exact = oracle.decode_attention(q.float().numpy(), [k.float().numpy() for k in ks],
                                    [v.float().numpy() for v in vs], shape.scale)
    qerr = np.abs(out.cpu().double().numpy() - exact)
    print(f"fp8 cache vs bf16 cache: max abs {qerr.max():.3e}, mean abs {qerr.mean():.3e}")
    assert qerr.mean() < 0.05


def test_decode_fp8_graph_replays():
    """Split contexts are merged inside the attention kernel: each partial has a
    ready flag set to the call's tag and cleared by the merging warp; graph
    replays reuse one tag and must still merge."""
    lens = [2048, 700, 0, 1, 1500, 3000]
    Hkv, B = 8, 32
    shape = wl.DecodeShape("fp8_graph", len(lens), 32, Hkv, D, B, torch.bfloat16)
    pool = _pool_with_codes(lens, Hkv, B, seed=12)
    dev = "cuda"
    kc, vc = torch.from_numpy(pool["kc"]).to(dev), torch.from_numpy(pool["vc"]).to(dev)
    tables = torch.from_numpy(pool["tables"]).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    qs = [wl.draw_query(shape, seed=300 + r) for r in range(3)]
    q = qs[0].to(dev)
    out = torch.empty_like(q)
    ws = torch.randint(0, 256, (pkv.paged_attention_workspace_size(len(lens), 32, D, 3000, 0),),
                       dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        pkv.paged_attention_decode_fp8(out, q, kc, vc, tables, sl, shape.scale, K_SCALE, V_SCALE, 3000, ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            pkv.paged_attention_decode_fp8(out, q, kc, vc, tables, sl, shape.scale, K_SCALE, V_SCALE, 3000, ws)
    for r in range(3):
        q.copy_(qs[r].to(dev))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_bf16_close(out.cpu(), _oracle(pool, qs[r], shape.scale), f"fp8 replay {r}")
        assert torch.all(out[2] == 0)


@pytest.mark.parametrize("B", [16, 32])
def test_decode_append_fp8_equals_write_then_decode(B):
    """The fused step (quantise and store each new token inside the attention
    kernel) must leave the same cache bytes and give the same output bits as
    kv_cache_write_fp8 at position len - 1 followed by paged_attention_decode_fp8,
    and match the oracle."""
    lens = [1, 2, 17, 300, 1024, 2049, 0, 33]
    Hq, Hkv = 32, 8
    shape = wl.DecodeShape("fp8_append", len(lens), Hq, Hkv, D, B, torch.bfloat16)
    pool = _pool_with_codes(lens, Hkv, B, seed=40 + B)
    q = wl.draw_query(shape, seed=41)
    k_new, v_new = _bf16_tokens(len(lens), Hkv, 42)
    dev = "cuda"
    tables = torch.from_numpy(pool["tables"]).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    maxL = max(lens)
    # path A: separate write (slots of position len - 1), then decode
    slots = np.array([token_slots(pool["tables"][s], L, B)[-1] if L else -1 for s, L in enumerate(lens)],
                     dtype=np.int64)
    kcA, vcA = torch.from_numpy(pool["kc"]).to(dev), torch.from_numpy(pool["vc"]).to(dev)
    pkv.kv_cache_write_fp8(k_new.to(dev), v_new.to(dev), kcA, vcA, torch.from_numpy(slots).to(dev),
                           K_SCALE, V_SCALE)
    outA = torch.empty((len(lens), Hq, D), dtype=torch.bfloat16, device=dev)
    pkv.paged_attention_decode_fp8(outA, q.to(dev), kcA, vcA, tables, sl, shape.scale, K_SCALE, V_SCALE, maxL)
    # path B: one call
    kcB, vcB = torch.from_numpy(pool["kc"]).to(dev), torch.from_numpy(pool["vc"]).to(dev)
    outB = torch.empty_like(outA)
    pkv.paged_attention_decode_append_fp8(outB, q.to(dev), k_new.to(dev), v_new.to(dev), kcB, vcB, tables, sl,
                                          shape.scale, K_SCALE, V_SCALE, maxL)
    torch.cuda.synchronize()
    assert torch.equal(kcA, kcB) and torch.equal(vcA, vcB)
    assert torch.equal(outA.view(torch.int16), outB.view(torch.int16))
    # oracle: the new token quantised by the oracle replaces position len - 1
    kq = [k.copy() for k in pool["kq"]]
    vq = [v.copy() for v in pool["vq"]]
    for s, L in enumerate(lens):
        if L:
            kq[s][L - 1] = f8.quantize(k_new[s].float().numpy(), K_SCALE)
            vq[s][L - 1] = f8.quantize(v_new[s].float().numpy(), V_SCALE)
    ref = oracle.decode_attention(q.float().numpy(), [f8.dequantize(k, K_SCALE) for k in kq],
                                  [f8.dequantize(v, V_SCALE) for v in vq], shape.scale)
    assert_bf16_close(outB.cpu(), ref, f"fp8 append B={B}")
    assert torch.all(outB[6] == 0)
    assert pkv.read_device_errors() == 0


@pytest.mark.parametrize("B", [16, 32])
def test_decode_append_fp8_graph_replays_advance_one_token_each(B):
    """The serving loop over an E4M3 cache: one paged_attention_decode_append_fp8
    call captured in a CUDA graph and replayed, the lengths and new bf16 tokens
    refreshed in place before each replay.  Each replay must quantise and store
    its tokens at the new position (the oracle's codes, bit for bit), attend over
    the grown context (oracle over the dequantised codes, the new token's own
    codes included), and leave later positions untouched."""
    lens0 = [1, 31, 32, 33, 300, 2047, 64]
    steps = 4
    full = [L + steps for L in lens0]
    Hq, Hkv = 32, 8
    shape = wl.DecodeShape("fp8_replay", len(lens0), Hq, Hkv, D, B, torch.bfloat16)
    pool = _pool_with_codes(full, Hkv, B, seed=70 + B)
    kc, vc = pool["kc"].copy(), pool["vc"].copy()
    for s, L in enumerate(lens0):  # positions L-1 .. are not in the pool yet: NaN codes there
        slots = token_slots(pool["tables"][s], full[s], B)[L - 1:]
        kc[slots // B, :, slots % B, :] = 0x7F
        vc[slots // B, :, :, slots % B] = 0x7F
    dev = "cuda"
    dkc, dvc = torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev)
    tables = torch.from_numpy(pool["tables"]).to(dev)
    q = wl.draw_query(shape, seed=71).to(dev)
    out = torch.empty((len(lens0), Hq, D), dtype=torch.bfloat16, device=dev)
    sl = torch.tensor(lens0, dtype=torch.int32, device=dev)
    toks = [_bf16_tokens(len(lens0), Hkv, 80 + r) for r in range(steps + 1)]
    k_new = torch.empty((len(lens0), Hkv, D), dtype=torch.bfloat16, device=dev)
    v_new = torch.empty_like(k_new)

    def refresh(rep):
        sl.copy_(torch.tensor([L + rep for L in lens0], dtype=torch.int32))
        k_new.copy_(toks[rep][0])
        v_new.copy_(toks[rep][1])

    call = lambda: pkv.paged_attention_decode_append_fp8(out, q, k_new, v_new, dkc, dvc, tables, sl, shape.scale,
                                                         K_SCALE, V_SCALE, max(full))
    refresh(0)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        call()  # warm; stores replay 0's tokens
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
    kq = [k.copy() for k in pool["kq"]]
    vq = [v.copy() for v in pool["vq"]]
    for rep in range(steps + 1):
        refresh(rep)
        g.replay()
        torch.cuda.synchronize()
        lens = [L + rep for L in lens0]
        for s, L in enumerate(lens):
            kq[s][L - 1] = f8.quantize(toks[rep][0][s].float().numpy(), K_SCALE)
            vq[s][L - 1] = f8.quantize(toks[rep][1][s].float().numpy(), V_SCALE)
        hk, hv = dkc.cpu().numpy(), dvc.cpu().numpy()
        for s, L in enumerate(lens):
            slots = token_slots(pool["tables"][s], full[s], B)
            assert np.array_equal(hk[slots[:L] // B, :, slots[:L] % B, :], kq[s][:L]), f"K codes, replay {rep}"
            assert np.array_equal(hv[slots[:L] // B, :, :, slots[:L] % B], vq[s][:L]), f"V codes, replay {rep}"
            assert (hk[slots[L:] // B, :, slots[L:] % B, :] == 0x7F).all()
        ref = oracle.decode_attention(q.cpu().float().numpy(), [f8.dequantize(k[:L], K_SCALE) for k, L in zip(kq, lens)],
                                      [f8.dequantize(v[:L], V_SCALE) for v, L in zip(vq, lens)], shape.scale)
        assert_bf16_close(out.cpu(), ref, f"fp8 append replay {rep} B={B}")
    assert pkv.read_device_errors() == 0
