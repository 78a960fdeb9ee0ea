"""GPU parity of multi-token paged attention (chunked prefill, verification of
drafted tokens) against the fp64 oracle: each sequence's last Q_s positions
attend causally over its paged context.  Calls whose queries span more than one
128-row block run as paired contexts (two blocks per context, one per softmax
group); shorter ones (verification) in the alternating form.  Unowned slots of the pool hold NaN,
so a read of a masked token would show as a non-finite output."""
import numpy as np
import pytest
import torch

from oracle.multi_token import multi_token_attention
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import assert_bf16_close, place_paged

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_errors():
    pkv.read_device_errors(clear=True)
    yield


def _case(Hq, Hkv, D, B, lens, qlens, seed, extra_blocks=5):
    shape = wl.DecodeShape(f"mt{Hq}_{Hkv}_{D}_{B}", len(lens), Hq, Hkv, D, B, torch.bfloat16)
    counts = [-(-L // B) for L in lens]
    NB = max(1, sum(counts) + extra_blocks)
    tables = wl.random_block_tables(counts, NB, max(1, max(counts)), seed + 1)
    ks, vs = zip(*[wl.draw_seq_kv(shape, seed, s, L) for s, L in enumerate(lens)])
    kc, vc = place_paged(ks, vs, tables, NB, B, torch.bfloat16)
    T = sum(qlens)
    q = wl.draw_normal((max(T, 1), Hq, D), torch.bfloat16, wl.sub_seed(seed, 20))[:T]
    starts = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    return dict(shape=shape, ks=ks, vs=vs, kc=kc, vc=vc, tables=tables, q=q, starts=starts, lens=lens,
                qlens=qlens, NB=NB)


def _run(c, max_q_len=None, max_seq_len=None, kc=None, vc=None, tables=None):
    dev = "cuda"
    q = c["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_multi_token(
        out, q, (c["kc"] if kc is None else kc).to(dev), (c["vc"] if vc is None else vc).to(dev),
        torch.from_numpy(c["tables"] if tables is None else tables).to(dev),
        torch.tensor(c["lens"], dtype=torch.int32, device=dev), torch.from_numpy(c["starts"]).to(dev),
        c["shape"].scale, max_q_len or max(1, max(c["qlens"])), max_seq_len or max(1, max(c["lens"])))
    torch.cuda.synchronize()
    return out.cpu()


def _oracle(c):
    st = c["starts"]
    qs = [c["q"][st[s]:st[s + 1]].float().numpy() for s in range(len(c["lens"]))]
    outs = multi_token_attention(qs, [k.float().numpy() for k in c["ks"]], [v.float().numpy() for v in c["vs"]],
                                 c["shape"].scale)
    return np.concatenate([o for o in outs if o.shape[0]], axis=0)


@pytest.mark.parametrize("Hq,Hkv,D,B,lens,qlens", [
    (32, 8, 128, 16, [5, 64, 700, 2000, 17, 1025], [5, 5, 5, 5, 5, 5]),       # verification of 4 drafts
    (32, 8, 128, 16, [3000, 1500], [512, 300]),                              # prefill chunks, 3 partitions
    (32, 8, 128, 16, [40, 1, 200, 33], [40, 1, 0, 17]),                       # whole prompt, decode, none
    (8, 8, 64, 8, [129, 1100], [16, 9]),                                      # MHA, head_dim 64, block 8
    (64, 8, 128, 32, [2500, 31], [24, 31]),                                   # 8 heads per KV head, block 32
    (12, 4, 64, 32, [1024, 1025, 2049], [8, 8, 8]),                           # partition edges
    (16, 4, 64, 8, [600, 333, 100], [200, 45, 33]),                           # paired blocks, head_dim 64, block 8
    (32, 8, 128, 16, [100, 65, 4000], [33, 65, 129]),                         # a pair's second block of 1 query
])
def test_multi_token_matches_oracle(Hq, Hkv, D, B, lens, qlens):
    c = _case(Hq, Hkv, D, B, lens, qlens, seed=Hq + D + B + len(lens))
    out = _run(c)
    assert_bf16_close(out, _oracle(c), f"multi-token {Hq}/{Hkv} D{D} B{B}")
    assert pkv.read_device_errors() == 0


def test_one_query_per_sequence_agrees_with_decode():
    lens = [1, 100, 1500, 2048]
    c = _case(32, 8, 128, 16, lens, [1, 1, 1, 1], seed=9)
    out = _run(c)
    dec = torch.empty_like(c["q"]).cuda()
    pkv.paged_attention_decode(dec, c["q"].cuda(), c["kc"].cuda(), c["vc"].cuda(),
                               torch.from_numpy(c["tables"]).cuda(),
                               torch.tensor(lens, dtype=torch.int32, device="cuda"), c["shape"].scale, 2048)
    torch.cuda.synchronize()
    err = (out.float() - dec.cpu().float()).abs()
    assert err.max() <= 2e-2 and err.mean() <= 1e-3


def test_placement_is_irrelevant_bit_identical():
    c = _case(32, 8, 128, 16, [1800, 400], [64, 7], seed=11)
    a = _run(c)
    perm = np.random.default_rng(3).permutation(c["NB"])
    kc2, vc2 = torch.empty_like(c["kc"]), torch.empty_like(c["vc"])
    kc2[torch.from_numpy(perm)] = c["kc"]
    vc2[torch.from_numpy(perm)] = c["vc"]
    t = c["tables"]
    t2 = np.where(t >= 0, perm[np.maximum(t, 0)], t).astype(np.int32)
    b = _run(c, kc=kc2, vc=vc2, tables=t2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_more_queries_than_context_is_flagged_and_zeroed():
    c = _case(16, 4, 128, 16, [3, 50], [3, 4], seed=12)
    # claim 5 query tokens for a 3-token context: positions -2, -1 see nothing
    c["starts"] = np.array([0, 5, 7], dtype=np.int32)
    c["q"] = wl.draw_normal((7, 16, 128), torch.bfloat16, 77)
    c["qlens"] = [5, 2]
    out = _run(c, max_q_len=5)
    assert pkv.read_device_errors() & pkv.DEVERR_SEQ_LEN
    assert torch.all(out[0:2].float() == 0)
    assert torch.isfinite(out.float()).all()


def test_workspace_too_small_is_rejected():
    c = _case(32, 8, 128, 16, [3000], [64], seed=13)
    need = pkv.paged_attention_multi_token_workspace_size(64, 32, 128, 3000)
    assert need > 0
    q = c["q"].cuda()
    with pytest.raises(pkv.PkvError):
        pkv.paged_attention_multi_token(torch.empty_like(q), q, c["kc"].cuda(), c["vc"].cuda(),
                                        torch.from_numpy(c["tables"]).cuda(),
                                        torch.tensor([3000], dtype=torch.int32, device="cuda"),
                                        torch.from_numpy(c["starts"]).cuda(), c["shape"].scale, 64, 3000,
                                        workspace=torch.empty(need - 256, dtype=torch.uint8, device="cuda"))


def test_graph_replays_over_a_random_workspace():
    """Prefill chunks long enough to be split between CTAs, merged inside the
    kernel: a CUDA graph replays one call several times over a workspace that
    starts as random bytes, with new queries each time."""
    c = _case(32, 8, 128, 16, [3000, 2500, 900, 4000], [512, 300, 64, 700], seed=14)
    dev = "cuda"
    q = c["q"].to(dev)
    out = torch.empty_like(q)
    kc, vc = c["kc"].to(dev), c["vc"].to(dev)
    tables = torch.from_numpy(c["tables"]).to(dev)
    lens = torch.tensor(c["lens"], dtype=torch.int32, device=dev)
    starts = torch.from_numpy(c["starts"]).to(dev)
    need = pkv.paged_attention_multi_token_workspace_size(q.shape[0], 32, 128, 4000)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device=dev)
    qs = [wl.draw_normal(tuple(q.shape), torch.bfloat16, 300 + r) for r in range(3)]

    def call():
        pkv.paged_attention_multi_token(out, q, kc, vc, tables, lens, starts, c["shape"].scale, 700, 4000,
                                        workspace=ws)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
    for r in range(3):
        q.copy_(qs[r].to(dev))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_bf16_close(out.cpu(), _oracle(dict(c, q=qs[r])), f"multi-token replay {r}")
    assert pkv.read_device_errors() == 0


@pytest.mark.parametrize("qlens", [[64, 7], [300, 200]])  # alternating and paired contexts
def test_output_at_a_16_byte_offset_gives_the_same_bits(qlens):
    """The output is promised 16-byte alignment only: rows are written in whole
    32-byte sectors where the address allows, else in 16-byte halves; both
    forms give the same bits."""
    c = _case(32, 8, 128, 16, [1800, 400], qlens, seed=15)
    a = _run(c)
    dev = "cuda"
    q = c["q"].to(dev)
    buf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=dev)
    out = buf[8:].view(q.shape)  # 16 bytes past a 256-byte aligned allocation
    assert out.data_ptr() % 32 == 16
    pkv.paged_attention_multi_token(out, q, c["kc"].to(dev), c["vc"].to(dev), torch.from_numpy(c["tables"]).to(dev),
                                    torch.tensor(c["lens"], dtype=torch.int32, device=dev),
                                    torch.from_numpy(c["starts"]).to(dev), c["shape"].scale, max(c["qlens"]),
                                    max(c["lens"]))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), out.cpu().view(torch.int16))
    assert pkv.read_device_errors() == 0
