"""The decode entry point for callers that cannot allocate device memory.

Such callers (a runtime that owns all device memory in its own pool, a plugin
host that only passes input and output buffers, a decode path where
allocation is forbidden) call paged_attention_decode_noalloc, which keeps
its split-K partials in an array built into the library instead of a
caller-provided workspace.  These tests call it through the C ABI and check
it against the fp64 oracle and against paged_attention_decode (same inputs,
workspace from PyTorch) on two calls in a row, so the second call runs over
the first call's leftovers in the shared array, and check that a problem too
large for the array is refused before any launch.

The file is named to be collected last: it must pass alone in a fresh
process and after every other test.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import _lib
from paged_kv_cache_279_gb300 import workloads as wl
from harness import (BF16_MAX_ABS, BF16_MEAN_ABS, F32_MAX_ABS, assert_bf16_close, assert_f32_close,
                     make_decode_case, oracle_out, run_decode)

pytestmark = pytest.mark.gpu


def call_noalloc(case, shape, partition_size=0, max_seq_len=None):
    """paged_attention_decode_noalloc through the C ABI; returns (status, out)."""
    lib = _lib.load()
    q = case["q"].cuda()
    out = torch.full_like(q, float("nan"))
    kc, vc = case["kc"].cuda(), case["vc"].cuda()
    tables = torch.from_numpy(case["tables"]).cuda()
    lens = torch.tensor(case["lens"], dtype=torch.int32, device="cuda")
    maxL = max_seq_len if max_seq_len is not None else max(1, max(case["lens"]))
    S, Hq, D = q.shape
    NB, Hkv, B, _ = kc.shape
    dtype = pkv.PKV_BF16 if q.dtype == torch.bfloat16 else pkv.PKV_F32
    st = lib.paged_attention_decode_noalloc(
        out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(),
        lens.data_ptr(), S, Hq, Hkv, D, B, tables.shape[1], NB, maxL, ctypes.c_float(shape.scale),
        partition_size, dtype, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, out


def assert_matches(got, want, dtype):
    err = (got.double() - want.double()).abs()
    assert torch.isfinite(got.float()).all()
    if dtype == torch.bfloat16:
        assert err.max().item() <= BF16_MAX_ABS and err.mean().item() <= BF16_MEAN_ABS
    else:
        assert err.max().item() <= F32_MAX_ABS


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_decode_on_two_calls(dtype):
    pkv.read_device_errors(clear=True)
    shape = wl.DecodeShape("noalloc", 0, 32, 8, 128, 16, dtype)
    # first call: long contexts split into many partitions
    first = make_decode_case(shape, [1, 700, 2048, 33, 1500], seed=21)
    close = assert_bf16_close if dtype == torch.bfloat16 else assert_f32_close
    st, out1 = call_noalloc(first, shape, partition_size=0)
    assert st == pkv.PKV_OK
    close(out1.cpu(), oracle_out(first, shape), "noalloc, first call")
    assert_matches(out1, run_decode(first, shape, partition_size=512), dtype)
    # second call in a row: other data and another split over the same array
    second = make_decode_case(shape, [900, 5, 1200], seed=22)
    st, out2 = call_noalloc(second, shape, partition_size=64)
    assert st == pkv.PKV_OK
    close(out2.cpu(), oracle_out(second, shape), "noalloc, second call")
    assert_matches(out2, run_decode(second, shape, partition_size=64), dtype)
    assert pkv.read_device_errors() == 0


def test_noalloc_refuses_problems_larger_than_its_array():
    shape = wl.DecodeShape("noalloc_big", 0, 32, 8, 128, 16, torch.bfloat16)
    case = make_decode_case(shape, [64, 64], seed=23)
    # 2 sequences x 32 heads x 4096 partitions of 16 tokens need far more than 16 MiB
    need = pkv.paged_attention_workspace_size(2, 32, 128, 65536, 16)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    st, out = call_noalloc(case, shape, partition_size=16, max_seq_len=65536)
    assert st == pkv.PKV_ERR_TOO_LARGE
    assert torch.isnan(out.float()).all()  # nothing was launched
