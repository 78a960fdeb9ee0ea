"""Paged decode attention on the GPU against the fp64 oracle, on sizes that
span several tiles, partitions and ragged tails, plus the properties the
method fixes: physical placement does not matter (bit-identical), a single
token returns its value, constant values come back unchanged, the split into
partitions does not change the result beyond rounding, empty contexts give
zeros, and bad indices are reported without a fault."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import workloads as wl
from harness import (assert_bf16_close, assert_f32_close, bits, make_decode_case, oracle_out, token_slots,
                     run_decode)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_errors():
    pkv.read_device_errors(clear=True)
    yield


def shape_of(Hq, Hkv, D, B, dtype=torch.bfloat16):
    return wl.DecodeShape(f"t{Hq}_{Hkv}_{D}_{B}", 0, Hq, Hkv, D, B, dtype)


def test_tiny_fp32_workload_with_cache_write():
    """4 sequences {1, 17, 33, 100}, 4/4 heads, head_dim 64, block 16, pool of 64
    blocks assigned by a seeded permutation; the newest token of each sequence
    is written with kv_cache_write before the decode."""
    shape = wl.TINY_FP32
    lens = wl.draw_lengths(shape, seed=0).tolist()
    case = make_decode_case(shape, lens, seed=0, num_blocks=64)
    kc, vc = case["kc"].clone(), case["vc"].clone()
    # remove the newest token from the pool, then write it through the library
    slots = []
    for s, L in enumerate(lens):
        slot = int(case["tables"][s][(L - 1) // 16]) * 16 + (L - 1) % 16
        slots.append(slot)
        kc[slot // 16, :, slot % 16] = float("nan")
        vc[slot // 16, :, slot % 16] = float("nan")
    case["kc_dev"], case["vc_dev"] = kc.cuda(), vc.cuda()
    k_new = torch.stack([case["ks"][s][L - 1] for s, L in enumerate(lens)]).cuda()
    v_new = torch.stack([case["vs"][s][L - 1] for s, L in enumerate(lens)]).cuda()
    pkv.kv_cache_write(k_new, v_new, case["kc_dev"], case["vc_dev"],
                       torch.tensor(slots, dtype=torch.int64, device="cuda"))
    assert torch.equal(bits(case["kc_dev"].cpu()), bits(case["kc"]))
    out = run_decode(case, shape)
    assert_f32_close(out, oracle_out(case, shape), "tiny fp32")
    assert pkv.read_device_errors() == 0


@pytest.mark.parametrize("Hq,Hkv,D,B,lens,P", [
    (32, 8, 128, 16, [1, 15, 16, 17, 100, 513, 1000], 0),
    (32, 8, 128, 16, [1, 15, 16, 17, 100, 513, 1000], 64),
    (64, 8, 128, 16, [3, 700, 1100], 128),
    (8, 8, 128, 16, [5, 47, 300], 0),      # MHA
    (16, 8, 128, 16, [33, 257], 48),       # 2 query heads per KV head
    (32, 8, 64, 16, [9, 160, 999], 256),
    (32, 4, 128, 8, [1, 8, 9, 95, 600], 96),
    (32, 4, 128, 32, [1, 31, 32, 33, 700], 64),
    (24, 4, 64, 32, [2, 2000], 512),
    (8, 1, 128, 16, [4096], 0),            # one KV head, 8 partitions
    (32, 4, 128, 8, [1, 8, 9, 95, 600], 0),    # balanced split, block 8
    (32, 4, 128, 32, [1, 31, 32, 33, 700], 0),  # balanced split, block 32
    (32, 8, 64, 16, [9, 160, 999], 0),
    # balanced split with contexts merged inside the attention kernel, every
    # lane layout of the merge: head_dim 64 and 128, 1, 2, 3, 7 and 8 query
    # heads per KV head
    (8, 8, 64, 16, [5, 47, 300, 2000], 0),
    (16, 8, 64, 16, [33, 1257, 2600], 0),
    (12, 4, 64, 16, [700, 1500], 0),
    (64, 8, 64, 32, [3000, 17], 0),
    (56, 8, 128, 16, [900, 1800], 0),
    (12, 4, 128, 16, [2500, 64, 1], 0),
])
def test_bf16_decode_matches_oracle(Hq, Hkv, D, B, lens, P):
    shape = shape_of(Hq, Hkv, D, B)
    case = make_decode_case(shape, lens, seed=Hq + D + B + P, extra_blocks=7)
    out = run_decode(case, shape, partition_size=P)
    assert_bf16_close(out, oracle_out(case, shape), f"{shape.name} P={P}")
    assert pkv.read_device_errors() == 0


@pytest.mark.parametrize("Hq,Hkv,D,B", [(4, 4, 64, 16), (8, 2, 128, 8), (16, 2, 64, 32)])
@pytest.mark.parametrize("P", [0, 32])
def test_fp32_decode_matches_oracle(Hq, Hkv, D, B, P):
    shape = shape_of(Hq, Hkv, D, B, torch.float32)
    case = make_decode_case(shape, [1, 30, 77, 130], seed=3 + Hq + B)
    out = run_decode(case, shape, partition_size=P)
    assert_f32_close(out, oracle_out(case, shape), f"fp32 {shape.name} P={P}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_physical_placement_is_irrelevant_bit_identical(dtype):
    shape = shape_of(32, 8, 128, 16, dtype)
    lens = [1, 37, 300, 1024]
    a = make_decode_case(shape, lens, seed=11, table_seed=1, extra_blocks=40)
    b = make_decode_case(shape, lens, seed=11, table_seed=2, extra_blocks=40)
    assert not np.array_equal(a["tables"], b["tables"])
    for P in (0, 64):
        oa = run_decode(a, shape, partition_size=P)
        ob = run_decode(b, shape, partition_size=P)
        assert torch.equal(bits(oa.cpu()), bits(ob.cpu()))


def test_single_token_context_returns_its_value_exactly():
    shape = shape_of(64, 8, 128, 16)
    case = make_decode_case(shape, [1] * 9, seed=4)
    out = run_decode(case, shape).cpu()
    for s in range(9):
        want = case["vs"][s][0].repeat_interleave(8, dim=0)  # [Hq, D]
        assert torch.equal(bits(out[s]), bits(want))


def test_constant_values_come_back_unchanged():
    shape = shape_of(32, 8, 128, 16)
    case = make_decode_case(shape, [5, 200, 1500], seed=5)
    for s, v in enumerate(case["vs"]):
        v.fill_(1.5)
    case["vc"] = torch.where(torch.isnan(case["vc"]), case["vc"], torch.full_like(case["vc"], 1.5))
    out = run_decode(case, shape, partition_size=64).float().cpu()
    assert torch.all(out == 1.5)


def test_partition_sizes_agree():
    shape = shape_of(32, 8, 128, 16)
    lens = [700, 2048, 16, 1]
    case = make_decode_case(shape, lens, seed=6)
    ref = oracle_out(case, shape)
    outs = {}
    for P in (16, 64, 512, 4096, 0):
        outs[P] = run_decode(case, shape, partition_size=P)
        assert_bf16_close(outs[P], ref, f"P={P}")
    # one partition covering everything is the plain single pass
    assert torch.equal(bits(run_decode(case, shape, partition_size=2048).cpu()),
                       bits(run_decode(case, shape, partition_size=4096).cpu()))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_empty_context_gives_zeros(dtype):
    shape = shape_of(8, 2, 64, 16, dtype)
    case = make_decode_case(shape, [0, 20, 0, 600], seed=7)
    out = run_decode(case, shape, partition_size=64).float().cpu()
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.isfinite(out).all()
    ref = oracle_out(case, shape)
    if dtype == torch.bfloat16:
        assert_bf16_close(out.to(torch.bfloat16), ref)
    else:
        assert_f32_close(out, ref)


def test_bad_block_id_and_length_are_flagged_not_faulted():
    shape = shape_of(32, 8, 128, 16)
    case = make_decode_case(shape, [40, 40], seed=8)
    case["tables"] = case["tables"].copy()
    case["tables"][0, 1] = case["NB"] + 5          # out of the pool
    case["tables"][1, 0] = -3
    out = run_decode(case, shape)
    assert pkv.read_device_errors() & pkv.DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    # a length beyond max_seq_len is clamped and reported
    case2 = make_decode_case(shape, [40, 64], seed=9)
    run_decode(case2, shape, max_seq_len=48)
    assert pkv.read_device_errors() & pkv.DEVERR_SEQ_LEN


def test_workspace_too_small_is_rejected():
    shape = shape_of(32, 8, 128, 16)
    case = make_decode_case(shape, [1000], seed=10)
    q = case["q"].cuda()
    need = pkv.paged_attention_workspace_size(1, 32, 128, 1000, 64)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode(torch.empty_like(q), q, case["kc"].cuda(), case["vc"].cuda(),
                                   torch.from_numpy(case["tables"]).cuda(),
                                   torch.tensor([1000], dtype=torch.int32, device="cuda"),
                                   shape.scale, 1000, partition_size=64, workspace=ws)
    assert e.value.status == pkv.PKV_ERR_INVALID


@pytest.mark.parametrize("S,maxlen,Hq,Hkv", [(300, 3000, 32, 8), (8, 16000, 32, 8), (77, 700, 64, 8)])
def test_balanced_split_many_sequences(S, maxlen, Hq, Hkv):
    """partition_size 0: all (sequence, kv head) contexts cut into equal shares,
    with empty contexts, contexts inside one share and contexts cut into many
    pieces in the same call."""
    shape = shape_of(Hq, Hkv, 128, 16)
    rng = np.random.default_rng(S + maxlen)
    lens = rng.integers(0, maxlen, size=S, endpoint=True)
    lens[:3] = [0, 1, maxlen]
    case = make_decode_case(shape, lens.tolist(), seed=S)
    out = run_decode(case, shape, partition_size=0, max_seq_len=maxlen)
    pick = sorted(set([0, 1, 2] + rng.choice(S, size=min(S, 12), replace=False).tolist()))
    ref = oracle_out(case, shape, seqs=pick)
    assert_bf16_close(out[pick], ref, f"balanced S={S}")
    assert torch.all(out[0].float() == 0)
    assert pkv.read_device_errors() == 0


def test_balanced_workspace_reused_across_calls():
    """One workspace, never cleared, serves many balanced calls in a row
    (different lengths, different splits): nothing left over from an earlier
    call may leak into a later one."""
    shape = shape_of(32, 8, 128, 16)
    need = pkv.paged_attention_workspace_size(40, 32, 128, 3000, 0)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN-like garbage
    rng = np.random.default_rng(99)
    for call in range(4):
        lens = rng.integers(0, 3000, size=40, endpoint=True).tolist()
        case = make_decode_case(shape, lens, seed=100 + call)
        q = case["q"].cuda()
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, case["kc"].cuda(), case["vc"].cuda(),
                                   torch.from_numpy(case["tables"]).cuda(),
                                   torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                   shape.scale, 3000, partition_size=0, workspace=ws)
        torch.cuda.synchronize()
        assert_bf16_close(out, oracle_out(case, shape), f"call {call}")
    assert pkv.read_device_errors() == 0


@pytest.mark.parametrize("P,dtype,B,nseq,D", [
    (0, torch.bfloat16, 16, 7, 128), (0, torch.bfloat16, 8, 7, 128), (0, torch.bfloat16, 32, 7, 128),
    (0, torch.bfloat16, 16, 7, 64), (0, torch.bfloat16, 8, 150, 64),
    (64, torch.bfloat16, 16, 7, 128),     # fixed partitions: the separate store kernel, then decode
    (64, torch.bfloat16, 16, 150, 128),
    (0, torch.float32, 16, 7, 128),       # fp32: the separate store kernel, then decode
    (0, torch.bfloat16, 16, 150, 128)])   # 150 x 8 segments: new rows patched into landed tiles
def test_decode_append_equals_write_then_decode(P, dtype, B, nseq, D):
    """paged_attention_decode_append = store the newest token of every
    sequence at position len - 1, then attend (fused into the balanced bf16
    kernel: the new row replaces the stale slot in the landed tile and is
    stored to the pool; a separate store kernel on the fixed-partition and fp32
    paths)."""
    shape = shape_of(32, 8, D, B, dtype)
    base = [1, 16, 17, 300, 0, 1500, 33]
    lens = (base * (nseq // len(base) + 1))[:nseq] if nseq != len(base) else base
    case = make_decode_case(shape, lens, seed=31 + B + P + D)
    kc, vc = case["kc"].clone(), case["vc"].clone()
    k_new = torch.zeros((len(lens), 8, D), dtype=dtype)
    v_new = torch.zeros_like(k_new)
    for s, L in enumerate(lens):
        if L == 0:
            continue
        slot = int(case["tables"][s][(L - 1) // B]) * B + (L - 1) % B
        kc[slot // B, :, slot % B] = float("nan")   # the newest token is not in the pool yet
        vc[slot // B, :, slot % B] = float("nan")
        k_new[s] = case["ks"][s][L - 1]
        v_new[s] = case["vs"][s][L - 1]
    dkc, dvc = kc.cuda(), vc.cuda()
    q = case["q"].cuda()
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_append(out, q, k_new.cuda(), v_new.cuda(), dkc, dvc,
                                      torch.from_numpy(case["tables"]).cuda(),
                                      torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                      shape.scale, max(lens), partition_size=P)
    torch.cuda.synchronize()
    assert torch.equal(bits(dkc.cpu()), bits(case["kc"])) and torch.equal(bits(dvc.cpu()), bits(case["vc"]))
    ref = oracle_out(case, shape)
    if dtype == torch.bfloat16:
        assert_bf16_close(out, ref, f"append P={P} B={B}")
    else:
        assert_f32_close(out, ref, "append fp32")
    assert torch.all(out[4].float() == 0)
    assert pkv.read_device_errors() == 0


def _replay_checks(call, refresh, check, reps=3):
    """Capture `call` in a CUDA graph on a side stream, then replay it `reps`
    times, refreshing the inputs in place before each replay."""
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        call()  # warm (tensor maps, shared-memory opt-in) outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
    for rep in range(reps):
        refresh(rep)
        g.replay()
        torch.cuda.synchronize()
        check(rep)


def test_balanced_merge_survives_graph_replays_and_random_workspace():
    """The balanced path merges split contexts inside the attention kernel:
    one ready flag per partial slot, carrying the call's tag, cleared by the
    merging warp.  A graph replays one call (same tag, same flags) several
    times, and the workspace starts as random bytes, so every call must both
    ignore stale flags and leave its own ready for a replay."""
    shape = shape_of(32, 8, 128, 16)
    lens = [3000, 1, 0, 2048, 517, 64] * 3
    case = make_decode_case(shape, lens, seed=55)
    dev = "cuda"
    kc, vc = case["kc"].to(dev), case["vc"].to(dev)
    tables = torch.from_numpy(case["tables"]).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    q = case["q"].to(dev)
    out = torch.empty_like(q)
    need = pkv.paged_attention_workspace_size(len(lens), 32, 128, 3000, 0)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device=dev)
    qs = [wl.draw_query(shape, seed=200 + r, num_seqs=len(lens)) for r in range(3)]

    def call():
        pkv.paged_attention_decode(out, q, kc, vc, tables, sl, shape.scale, 3000, 0, ws)

    def refresh(r):
        q.copy_(qs[r].to(dev))
        out.fill_(float("nan"))

    def check(r):
        assert_bf16_close(out, oracle_out(dict(case, q=qs[r]), shape), f"replay {r}")
        assert torch.all(out[2].float() == 0)

    _replay_checks(call, refresh, check)
    assert pkv.read_device_errors() == 0


def test_decode_append_graph_replays_advance_one_token_each():
    """The serving loop: one decode_append call captured in a CUDA graph and
    replayed step after step, the lengths and new tokens refreshed in place
    before each replay.  Every replay must store its token at the new
    position (pool bit-exact), attend over the context including it (oracle),
    and the tokens not yet appended stay NaN in the pool."""
    shape = shape_of(32, 8, 128, 16)
    lens0 = [1, 15, 16, 31, 300, 2047, 64] * 3
    steps = 4
    full = [L + steps for L in lens0]
    case = make_decode_case(shape, full, seed=77, extra_blocks=8)
    kc, vc = case["kc"].clone(), case["vc"].clone()
    B = shape.block_size
    for s, L in enumerate(lens0):  # positions L-1 .. L+steps-1 are not in the pool yet
        slots = torch.from_numpy(token_slots(case["tables"][s], full[s], B)[L - 1:])
        kc[slots // B, :, slots % B] = float("nan")
        vc[slots // B, :, slots % B] = float("nan")
    dkc, dvc = kc.cuda(), vc.cuda()
    tables = torch.from_numpy(case["tables"]).cuda()
    q = case["q"].cuda()
    out = torch.empty_like(q)
    S = len(lens0)
    sl = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    k_new = torch.empty((S, 8, 128), dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)

    def refresh(rep):
        lens = [L + rep for L in lens0]
        sl.copy_(torch.tensor(lens, dtype=torch.int32))
        k_new.copy_(torch.stack([case["ks"][s][L - 1] for s, L in enumerate(lens)]))
        v_new.copy_(torch.stack([case["vs"][s][L - 1] for s, L in enumerate(lens)]))

    refresh(0)
    call = lambda: pkv.paged_attention_decode_append(out, q, k_new, v_new, dkc, dvc, tables, sl, shape.scale,
                                                     max(full))

    def check(rep):
        lens = [L + rep for L in lens0]
        sub = dict(case, ks=[k[:L] for k, L in zip(case["ks"], lens)], vs=[v[:L] for v, L in zip(case["vs"], lens)],
                   lens=lens)
        assert_bf16_close(out, oracle_out(sub, shape), f"replay {rep}")
        hk = dkc.cpu()
        for s, L in enumerate(lens):
            sl_ = torch.from_numpy(token_slots(case["tables"][s], full[s], B))
            assert torch.equal(bits(hk[sl_[:L] // B, :, sl_[:L] % B]), bits(case["kc"][sl_[:L] // B, :, sl_[:L] % B]))
            assert torch.isnan(hk[sl_[L:] // B, :, sl_[L:] % B].float()).all()

    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        call()  # warm (tensor maps, shared-memory opt-in); stores replay 0's tokens
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
    for rep in range(steps + 1):
        refresh(rep)
        g.replay()
        torch.cuda.synchronize()
        check(rep)
    assert pkv.read_device_errors() == 0
