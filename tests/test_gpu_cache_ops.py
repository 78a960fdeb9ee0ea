"""Cache write and block copy on the GPU: bit-exact against the oracle's
array semantics, untouched slots keep their sentinel, bad indices are skipped
and reported through the device error word."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_279_gb300 as pkv
from harness import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_errors():
    pkv.read_device_errors(clear=True)
    yield


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_kv_cache_write_bit_exact(dtype, D, B):
    g = torch.Generator().manual_seed(D * 100 + B)
    NB, Hkv, T = 37, 4, 53
    kc = torch.full((NB, Hkv, B, D), -3.25, dtype=dtype)
    vc = torch.full_like(kc, 7.5)
    kn = torch.randn(T, Hkv, D, generator=g).to(dtype)
    vn = torch.randn(T, Hkv, D, generator=g).to(dtype)
    perm = torch.randperm(NB * B, generator=g)[:T].to(torch.int64)
    perm[5] = -1  # padding token
    perm[11] = -42
    kc_ref, vc_ref = kc.clone(), vc.clone()
    oracle.kv_cache_write(kc_ref, vc_ref, kn, vn, perm.numpy(), B)
    dkc, dvc = kc.cuda(), vc.cuda()
    pkv.kv_cache_write(kn.cuda(), vn.cuda(), dkc, dvc, perm.cuda())
    torch.cuda.synchronize()
    assert torch.equal(bits(dkc.cpu()), bits(kc_ref))
    assert torch.equal(bits(dvc.cpu()), bits(vc_ref))
    assert pkv.read_device_errors() == 0


def test_kv_cache_write_out_of_range_slot_is_skipped_and_flagged():
    NB, Hkv, B, D = 8, 2, 16, 64
    kc = torch.zeros((NB, Hkv, B, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones((3, Hkv, D), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([0, NB * B, NB * B + 1000], dtype=torch.int64, device="cuda")
    pkv.kv_cache_write(kn, kn, kc, vc, slots)
    flags = pkv.read_device_errors()
    assert flags & pkv.DEVERR_SLOT
    assert kc[0, :, 0].eq(1).all() and kc.sum().item() == Hkv * D  # only slot 0 written


def test_kv_cache_write_nan_payloads_survive():
    NB, Hkv, B, D = 4, 1, 16, 64
    kc = torch.zeros((NB, Hkv, B, D), dtype=torch.bfloat16, device="cuda")
    raw = torch.arange(D, dtype=torch.int16).view(1, 1, D) | 0x7F80  # NaN/Inf patterns
    kn = raw.view(torch.bfloat16).cuda()
    pkv.kv_cache_write(kn, kn, kc, kc.clone(), torch.tensor([17], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(bits(kc[1, 0, 1].cpu()), raw.view(-1))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_block_copy_bit_exact_every_layer(dtype):
    g = torch.Generator().manual_seed(5)
    L, NB, Hkv, B, D = 5, 30, 8, 16, 128
    ks = [torch.randn(NB, Hkv, B, D, generator=g).to(dtype) for _ in range(L)]
    vs = [torch.randn(NB, Hkv, B, D, generator=g).to(dtype) for _ in range(L)]
    pairs = np.array([[3, 17], [4, 9], [29, 0], [12, 13]], dtype=np.int64)
    ks_ref = [k.clone() for k in ks]
    vs_ref = [v.clone() for v in vs]
    oracle.block_copy(ks_ref, vs_ref, pairs)
    dks = [k.cuda() for k in ks]
    dvs = [v.cuda() for v in vs]
    pkv.block_copy(dks, dvs, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    for l in range(L):
        assert torch.equal(bits(dks[l].cpu()), bits(ks_ref[l]))
        assert torch.equal(bits(dvs[l].cpu()), bits(vs_ref[l]))
    assert pkv.read_device_errors() == 0


def test_block_copy_many_layers_and_bad_pairs():
    L, NB, Hkv, B, D = 70, 6, 2, 8, 64  # more layers than one launch carries
    ks = [torch.full((NB, Hkv, B, D), float(l), dtype=torch.bfloat16, device="cuda") for l in range(L)]
    vs = [torch.full((NB, Hkv, B, D), float(-l), dtype=torch.bfloat16, device="cuda") for l in range(L)]
    for l in range(L):
        ks[l][1] = 100 + l
        vs[l][1] = -100 - l
    pairs = torch.tensor([[1, 4], [2, 2], [-1, 3], [5, 6]], dtype=torch.int64, device="cuda")
    pkv.block_copy(ks, vs, pairs)
    flags = pkv.read_device_errors()
    assert flags & pkv.DEVERR_COPY_PAIR
    for l in (0, 63, 64, 69):
        assert ks[l][4].eq(100 + l).all() and vs[l][4].eq(-100 - l).all()
        assert ks[l][3].eq(l).all() and ks[l][2].eq(l).all()
