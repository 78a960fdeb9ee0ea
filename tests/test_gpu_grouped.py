"""Grouped decode (shared prefixes read once per group) against the fp64
oracle and against the plain decode: beam search with 1024 and 1032 shared
tokens, decode-and-append, members with nothing of their own, singleton
groups, and a bad group description (flagged, no fault)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import assert_bf16_close, bits, build_beam_pool, make_decode_case, oracle_out, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_errors():
    pkv.read_device_errors(clear=True)
    yield


def grouped(case, shape, q, offs, pre, max_seq_len, k_new=None, v_new=None):
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_grouped(
        out, q, case["kc"], case["vc"], torch.from_numpy(case["tables"]).cuda(),
        torch.from_numpy(np.asarray(case["lens"], dtype=np.int32)).cuda(),
        torch.from_numpy(offs).cuda(), torch.from_numpy(pre).cuda(), shape.scale, max_seq_len,
        k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("shared", [wl.BEAM_SHARED, wl.BEAM_SHARED_PARTIAL])
def test_beam_search_grouped_matches_oracle(shared):
    shape = wl.BEAM_BF16
    div = wl.draw_divergent_lengths(wl.BEAM_PROMPTS * wl.BEAM_WIDTH, seed=1)
    case = build_beam_pool(shape, shared, wl.BEAM_PROMPTS, wl.BEAM_WIDTH, div)
    offs, pre = case["alloc"].prefix_groups(case["seqs"])
    assert len(pre) == wl.BEAM_PROMPTS and (pre == 1024).all()
    q = wl.draw_query(shape, 4).cuda()
    maxL = int(case["lens"].max())
    out = grouped(case, shape, q, offs, pre, maxL)
    ref = oracle.decode_attention(q.float().cpu().numpy(), [k.float().numpy() for k in case["ks"]],
                                  [v.float().numpy() for v in case["vs"]], shape.scale)
    assert_bf16_close(out, ref, f"grouped beam shared={shared}")
    assert pkv.read_device_errors() == 0


def test_grouped_append_matches_oracle_and_stores_tokens():
    shape = wl.DecodeShape("beam_small", 0, 64, 8, 128, 16, torch.bfloat16)
    div = np.array([1, 40, 17, 3, 90, 16, 5, 200] * 4)  # every beam has a new token
    case = build_beam_pool(shape, 512, 4, 8, div, seed=8, append_last=True)
    offs, pre = case["alloc"].prefix_groups(case["seqs"])
    q = wl.draw_query(shape, 9, num_seqs=len(case["seqs"])).cuda()
    out = grouped(case, shape, q, offs, pre, int(case["lens"].max()),
                  case["k_new"].cuda(), case["v_new"].cuda())
    ref = oracle.decode_attention(q.float().cpu().numpy(), [k.float().numpy() for k in case["ks"]],
                                  [v.float().numpy() for v in case["vs"]], shape.scale)
    assert_bf16_close(out, ref, "grouped append")
    # the new tokens were stored where the allocator put them
    for s in (0, 7, 13):
        L = int(case["lens"][s])
        slot = int(case["alloc"].slots(s, L - 1, 1)[0])
        got = case["kc"][slot // 16, :, slot % 16].cpu()
        assert torch.equal(bits(got), bits(case["k_new"][s]))
    assert pkv.read_device_errors() == 0


def test_members_with_nothing_of_their_own_and_singletons():
    shape = wl.DecodeShape("beam_edge", 0, 32, 8, 128, 16, torch.bfloat16)
    div = np.array([0, 0, 33, 0,  5, 0, 0, 0])  # 2 prompts x 4 beams, most beams empty
    case = build_beam_pool(shape, 256, 2, 4, div, seed=11)
    q = wl.draw_query(shape, 12, num_seqs=8).cuda()
    ref = oracle.decode_attention(q.float().cpu().numpy(), [k.float().numpy() for k in case["ks"]],
                                  [v.float().numpy() for v in case["vs"]], shape.scale)
    offs, pre = case["alloc"].prefix_groups(case["seqs"])
    assert (pre == 256).all()
    assert_bf16_close(grouped(case, shape, q, offs, pre, int(case["lens"].max())), ref, "grouped edges")
    # the same batch described as singleton groups (no sharing) gives the same result
    single = np.arange(9, dtype=np.int32)
    out = grouped(case, shape, q, single, np.zeros(8, dtype=np.int32), int(case["lens"].max()))
    assert_bf16_close(out, ref, "singletons")
    assert pkv.read_device_errors() == 0


def test_bad_group_description_is_flagged_not_faulted():
    shape = wl.DecodeShape("beam_bad", 0, 32, 8, 128, 16, torch.bfloat16)
    case = build_beam_pool(shape, 256, 2, 4, np.array([3, 3, 3, 3, 3, 3, 3, 3]), seed=13)
    q = wl.draw_query(shape, 14, num_seqs=8).cuda()
    offs = np.array([0, 8], dtype=np.int32)          # two prompts claimed as one group
    pre = np.array([256], dtype=np.int32)
    out = grouped(case, shape, q, offs, pre, int(case["lens"].max()))
    assert pkv.read_device_errors() & pkv.DEVERR_PREFIX
    assert torch.isfinite(out.float()).all()
    offs = np.array([0, 3, 8], dtype=np.int32)
    pre = np.array([250, 256], dtype=np.int32)        # not a whole number of tiles
    grouped(case, shape, q, offs, pre, int(case["lens"].max()))
    assert pkv.read_device_errors() & pkv.DEVERR_PREFIX


@pytest.mark.parametrize("D,B,Hq,Hkv,prompts,width,shared", [
    (64, 8, 16, 4, 3, 5, 256),     # head_dim 64, 8-token blocks (8 TMA boxes per 64-token tile)
    (128, 32, 8, 8, 2, 40, 320),   # one query head per kv head, 32-token blocks
    (128, 16, 32, 4, 1, 20, 200),  # 20 members x 8 heads = 160 rows: two row chunks
    (128, 8, 8, 8, 1, 150, 128),   # 150 members x 1 head: chunks of 128 and 22 rows
])
def test_grouped_shapes_match_oracle(D, B, Hq, Hkv, prompts, width, shared):
    shape = wl.DecodeShape("grouped_shape", 0, Hq, Hkv, D, B, torch.bfloat16)
    div = np.random.default_rng(D + B + width).integers(0, 41, prompts * width)
    case = build_beam_pool(shape, shared, prompts, width, div, seed=17)
    offs, pre = case["alloc"].prefix_groups(case["seqs"])
    assert len(pre) == prompts and (pre > 0).all()
    q = wl.draw_query(shape, 18, num_seqs=prompts * width).cuda()
    out = grouped(case, shape, q, offs, pre, int(case["lens"].max()))
    ref = oracle.decode_attention(q.float().cpu().numpy(), [k.float().numpy() for k in case["ks"]],
                                  [v.float().numpy() for v in case["vs"]], shape.scale)
    assert_bf16_close(out, ref, f"grouped D={D} B={B} {Hq}/{Hkv} {prompts}x{width}")
    assert pkv.read_device_errors() == 0


def test_more_groups_than_one_launch_scans():
    """2100 groups (one launch scans at most 1024): the call runs the groups in
    three launches over the same workspace."""
    shape = wl.DecodeShape("beam_many", 0, 8, 2, 64, 16, torch.bfloat16)
    prompts, width = 2100, 2
    div = np.random.default_rng(7).integers(0, 21, prompts * width)
    case = build_beam_pool(shape, 64, prompts, width, div, seed=21)
    offs, pre = case["alloc"].prefix_groups(case["seqs"])
    assert len(pre) == prompts and (pre == 64).all()
    q = wl.draw_query(shape, 22, num_seqs=prompts * width).cuda()
    out = grouped(case, shape, q, offs, pre, int(case["lens"].max()))
    ref = oracle.decode_attention(q.float().cpu().numpy(), [k.float().numpy() for k in case["ks"]],
                                  [v.float().numpy() for v in case["vs"]], shape.scale)
    assert_bf16_close(out, ref, "2100 groups")
    assert pkv.read_device_errors() == 0


def test_grouped_graph_replays_over_a_random_workspace():
    """Contexts split between CTAs are merged inside the kernel through ready
    flags carrying the call's tag, cleared by the merging CTA: a CUDA graph
    replays one call (one tag) several times over a workspace that starts as
    random bytes, with new queries before each replay."""
    shape = wl.BEAM_BF16
    div = wl.draw_divergent_lengths(wl.BEAM_PROMPTS * wl.BEAM_WIDTH, seed=3)
    case = build_beam_pool(shape, wl.BEAM_SHARED_PARTIAL, wl.BEAM_PROMPTS, wl.BEAM_WIDTH, div, seed=5)
    offs, pre = case["alloc"].prefix_groups(case["seqs"])
    S = len(case["seqs"])
    maxL = int(case["lens"].max())
    need = pkv.paged_attention_grouped_workspace_size(S, shape.num_heads, shape.head_dim, maxL)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    tables = torch.from_numpy(case["tables"]).cuda()
    lens = torch.from_numpy(np.asarray(case["lens"], dtype=np.int32)).cuda()
    d_offs, d_pre = torch.from_numpy(offs).cuda(), torch.from_numpy(pre).cuda()
    q = torch.empty((S, shape.num_heads, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    qs = [wl.draw_query(shape, 40 + r, num_seqs=S) for r in range(3)]

    def call():
        pkv.paged_attention_decode_grouped(out, q, case["kc"], case["vc"], tables, lens, d_offs, d_pre,
                                           shape.scale, maxL, workspace=ws)
    q.copy_(qs[0].cuda())
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
    ks = [k.float().numpy() for k in case["ks"]]
    vs = [v.float().numpy() for v in case["vs"]]
    for r in range(3):
        q.copy_(qs[r].cuda())
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.decode_attention(qs[r].float().numpy(), ks, vs, shape.scale)
        assert_bf16_close(out, ref, f"grouped replay {r}")
    assert pkv.read_device_errors() == 0
