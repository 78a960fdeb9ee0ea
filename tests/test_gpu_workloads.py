"""The five workloads at their full sizes, in the launch configuration the
benchmark times (partition_size 0: balanced split; the fused store where the
benchmark uses it), against the fp64 oracle.

* GQA decode: 64 sequences, lengths U[64, 2048], 32/8 heads -- every output.
* long context: 8 x 16,000 tokens, 512-token partitions and the balanced split
  -- two whole sequences (all heads) compared.
* beam search: 32 prompts x 8 beams, 1024 or 1032 shared tokens, 0-256 own
  tokens per beam, built through the C++ allocator (fork, append, copy-on-write
  pairs executed with block_copy) -- every beam against the oracle on its own
  token sequence, and the allocator checked step by step against its model.
* continuous-batching mix: 256 lognormal lengths at block sizes 8, 16, 32,
  built through the allocator -- sampled sequences, and the allocator's waste
  equal to the closed form.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import assert_bf16_close, bits, make_decode_case, oracle_out, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_errors():
    pkv.read_device_errors(clear=True)
    yield
    assert pkv.read_device_errors(clear=True) == 0


def test_gqa_decode_full_size_every_output():
    shape = wl.GQA_BF16
    lens = wl.draw_lengths(shape, seed=0).tolist()
    need = sum(-(-L // 16) for L in lens)
    case = make_decode_case(shape, lens, seed=0, num_blocks=int(np.ceil(1.1 * need)))
    # the benchmark's call: the newest token stored by the attention kernel itself
    kc, vc = case["kc"].clone(), case["vc"].clone()
    k_new = torch.stack([case["ks"][s][L - 1] for s, L in enumerate(lens)])
    v_new = torch.stack([case["vs"][s][L - 1] for s, L in enumerate(lens)])
    for s, L in enumerate(lens):
        slot = int(case["tables"][s][(L - 1) // 16]) * 16 + (L - 1) % 16
        kc[slot // 16, :, slot % 16] = float("nan")
        vc[slot // 16, :, slot % 16] = float("nan")
    dkc, dvc, q = kc.cuda(), vc.cuda(), case["q"].cuda()
    out = torch.empty_like(q)
    pkv.paged_attention_decode_append(out, q, k_new.cuda(), v_new.cuda(), dkc, dvc,
                                      torch.from_numpy(case["tables"]).cuda(),
                                      torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                      shape.scale, max(lens) + 64, partition_size=0)
    torch.cuda.synchronize()
    assert torch.equal(bits(dkc.cpu()), bits(case["kc"]))
    assert_bf16_close(out, oracle_out(case, shape), "GQA full size")


@pytest.mark.parametrize("P", [512, 0])
def test_long_context_full_size_sampled(P):
    shape = wl.LONG_BF16
    lens = wl.draw_lengths(shape, seed=0).tolist()
    case = make_decode_case(shape, lens, seed=0, extra_blocks=800)
    out = run_decode(case, shape, partition_size=P, max_seq_len=16000)
    pick = [0, 5]
    assert_bf16_close(out[pick], oracle_out(case, shape, seqs=pick), f"long context P={P}")


@pytest.mark.parametrize("shared", [wl.BEAM_SHARED, wl.BEAM_SHARED_PARTIAL])
def test_beam_search_with_copy_on_write(shared):
    shape = wl.BEAM_BF16
    B, Hkv, D = shape.block_size, shape.num_kv_heads, shape.head_dim
    P_, W = wl.BEAM_PROMPTS, wl.BEAM_WIDTH
    div = wl.draw_divergent_lengths(P_ * W, seed=1)
    NB = P_ * (-(-shared // B) + 1) + sum(-(-int(d) // B) + 1 for d in div) + 64
    alloc = pkv.BlockAllocator(NB, B)
    model = oracle.BlockAllocatorModel(NB, B)
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=shape.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    prefix = [wl.draw_seq_kv(shape, 2, p, shared) for p in range(P_)]
    own = [wl.draw_seq_kv(shape, 3, b, int(div[b])) for b in range(P_ * W)]
    for p in range(P_):
        assert alloc.add_seq(p * W, shared) == 0 and model.add_seq(p * W, shared) == 0
        slots = torch.from_numpy(alloc.slots(p * W, 0, shared)).cuda()
        pkv.kv_cache_write(prefix[p][0].cuda(), prefix[p][1].cuda(), kc, vc, slots)
        for c in range(1, W):
            assert alloc.fork(p * W, p * W + c) == 0 and model.fork(p * W, p * W + c) == 0
    copies = 0
    for t in range(int(div.max())):
        beams = [b for b in range(P_ * W) if div[b] > t]
        st, slots, pairs = alloc.append_slots(beams)
        assert st == 0
        want = [model.append_slot(b) for b in beams]
        assert slots.tolist() == [w[1] for w in want]
        assert [tuple(x) for x in pairs.tolist()] == [(w[2], w[3]) for w in want if w[2] >= 0]
        if len(pairs):
            copies += len(pairs)
            pkv.block_copy([kc], [vc], torch.from_numpy(np.ascontiguousarray(pairs)).cuda())
        kn = torch.stack([own[b][0][t] for b in beams]).cuda()
        vn = torch.stack([own[b][1][t] for b in beams]).cuda()
        pkv.kv_cache_write(kn, vn, kc, vc, torch.from_numpy(slots).cuda())
    # copy-on-write: only a partially filled shared block is ever copied, by every
    # diverging beam but the last holder
    if shared % B == 0:
        assert copies == 0
    else:
        expect = sum(min(W - 1, int((div[p * W:(p + 1) * W] > 0).sum())) for p in range(P_))
        assert copies == expect and copies > 0
    seqs = list(range(P_ * W))
    lens = [shared + int(d) for d in div]
    tables, seq_lens = alloc.block_tables(seqs, cap=max(len(alloc.block_table(s)) for s in seqs))
    assert seq_lens.tolist() == lens
    q = wl.draw_query(shape, 4).cuda()
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(seq_lens).cuda(), shape.scale, max(lens))
    torch.cuda.synchronize()
    # each beam sees its prompt followed by its own tokens, nothing of its siblings
    ks = [torch.cat([prefix[b // W][0], own[b][0]]).float().numpy() for b in seqs]
    vs = [torch.cat([prefix[b // W][1], own[b][1]]).float().numpy() for b in seqs]
    ref = oracle.decode_attention(q.float().cpu().numpy(), ks, vs, shape.scale)
    assert_bf16_close(out, ref, f"beam search shared={shared}")
    used, allocated = alloc.waste()
    assert (used, allocated) == model.waste()


@pytest.mark.parametrize("B", [8, 16, 32])
def test_mixed_batch_block_sizes_and_waste(B):
    base = wl.MIXED_BF16
    shape = wl.DecodeShape(base.name, base.num_seqs, base.num_heads, base.num_kv_heads,
                           base.head_dim, B, base.dtype, base.num_layers)
    lens = wl.draw_lengths(shape, seed=0).tolist()
    Hkv, D, S = shape.num_kv_heads, shape.head_dim, len(lens)
    NB = int(np.ceil(1.1 * sum(-(-L // B) for L in lens)))
    alloc = pkv.BlockAllocator(NB, B)
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=shape.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    ks, vs, slots = [], [], []
    for s, L in enumerate(lens):
        assert alloc.add_seq(s, L) == 0
        k, v = wl.draw_seq_kv(shape, 5, s, L)
        ks.append(k)
        vs.append(v)
        slots.append(alloc.slots(s, 0, L))
    pkv.kv_cache_write(torch.cat(ks).cuda(), torch.cat(vs).cuda(), kc, vc,
                       torch.from_numpy(np.concatenate(slots)).cuda())
    used, allocated = alloc.waste()
    assert used == sum(lens)
    assert allocated == sum(oracle.blocks_needed(L, B) * B for L in lens)
    assert np.isclose(1 - used / allocated, oracle.paged_waste_fraction(lens, B))
    cap = max(-(-L // B) for L in lens)
    tables, seq_lens = alloc.block_tables(range(S), cap=cap)
    q = wl.draw_query(shape, 6).cuda()
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(seq_lens).cuda(), shape.scale, max(lens))
    torch.cuda.synchronize()
    rng = np.random.default_rng(B)
    pick = sorted(set([int(np.argmax(lens)), int(np.argmin(lens))] + rng.choice(S, 22, replace=False).tolist()))
    ref = oracle.decode_attention(q.float().cpu().numpy()[pick], [ks[s].float().numpy() for s in pick],
                                  [vs[s].float().numpy() for s in pick], shape.scale)
    assert_bf16_close(out[pick], ref, f"mixed B={B}")
