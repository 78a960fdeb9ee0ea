"""The C-ABI library loads without a GPU, exports every function that
include/pkv.h declares, and rejects bad arguments on the host before any
device work (these calls return before touching CUDA)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_279_gb300 as pkv
from paged_kv_cache_279_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    # every declaration is marked PKV_EXPORT: take the identifier before "("
    names = re.findall(r"^PKV_EXPORT [^;(]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    lib = _lib.load()
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), f"libpkv.so does not export {n}"
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_status_strings_and_version():
    lib = _lib.load()
    assert lib.pkv_abi_version() == 1
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(2) == b"out of KV blocks"
    assert lib.pkv_status_string(99) == b"unknown status"


def test_host_validation_rejects_before_launch():
    lib = _lib.load()
    # unsupported head_dim / block size / dtype: rejected on the host
    assert lib.kv_cache_write(None, None, None, None, None, 4, 8, 96, 16, 64, 1, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.kv_cache_write(None, None, None, None, None, 4, 8, 128, 12, 64, 1, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.kv_cache_write(None, None, None, None, None, 4, 8, 128, 16, 64, 7, None) == pkv.PKV_ERR_UNSUPPORTED
    # null pointers with work to do
    assert lib.kv_cache_write(None, None, None, None, None, 4, 8, 128, 16, 64, 1, None) == pkv.PKV_ERR_INVALID
    # nothing to do is fine
    assert lib.kv_cache_write(None, None, None, None, None, 0, 8, 128, 16, 64, 1, None) == pkv.PKV_OK
    dec = lib.paged_attention_decode
    common = dict(S=2, Hq=32, Hkv=8, D=128, B=16, maxB=4, NB=16, maxL=64)

    def call(S=2, Hq=32, Hkv=8, D=128, B=16, maxB=4, NB=16, maxL=64, P=0, dt=1, scale=0.1):
        return dec(None, None, None, None, None, None, S, Hq, Hkv, D, B, maxB, NB, maxL, scale, P,
                   None, 0, dt, None)
    assert call(Hq=30) == pkv.PKV_ERR_INVALID          # Hq not a multiple of Hkv
    assert call(Hq=72) == pkv.PKV_ERR_UNSUPPORTED      # 9 query heads per KV head
    assert call(D=96) == pkv.PKV_ERR_UNSUPPORTED
    assert call(P=24) == pkv.PKV_ERR_INVALID           # partition not a multiple of 16
    assert call(scale=float("nan")) == pkv.PKV_ERR_INVALID
    assert call(S=0) == pkv.PKV_OK
    assert call() == pkv.PKV_ERR_INVALID               # null pointers
    assert lib.block_copy(None, None, 0, None, 5, 16, 4096, None) == pkv.PKV_OK
    assert lib.block_copy(None, None, 2, None, 5, 16, 4096, None) == pkv.PKV_ERR_INVALID
    assert lib.block_copy(None, None, 2, None, 5, 16, 4000, None) == pkv.PKV_ERR_INVALID
    flags = ctypes.c_uint32()
    assert lib.pkv_read_device_errors(None, 0, None) == pkv.PKV_ERR_INVALID
    del flags
    # the bounded-wait check: bad arguments never reach the device
    assert lib.pkv_bounded_wait_check(None, 4, 7, 1, 100, None) == pkv.PKV_ERR_INVALID
    assert lib.pkv_bounded_wait_check(None, -1, 7, 1, 100, None) == pkv.PKV_ERR_INVALID
    assert lib.pkv_bounded_wait_check(None, 0, 7, 1, 0, None) == pkv.PKV_ERR_INVALID


def test_fp8_host_validation_rejects_before_launch():
    lib = _lib.load()
    w = lib.kv_cache_write_fp8
    assert w(None, None, None, None, None, 4, 8, 64, 16, 64, 0.1, 0.1, None) == pkv.PKV_ERR_UNSUPPORTED   # D 64
    assert w(None, None, None, None, None, 4, 8, 128, 8, 64, 0.1, 0.1, None) == pkv.PKV_ERR_UNSUPPORTED   # B 8
    assert w(None, None, None, None, None, 4, 8, 128, 16, 64, 0.0, 0.1, None) == pkv.PKV_ERR_INVALID      # scale 0
    assert w(None, None, None, None, None, 4, 8, 128, 16, 64, 0.1, float("inf"), None) == pkv.PKV_ERR_INVALID
    assert w(None, None, None, None, None, 4, 8, 128, 16, 64, 0.1, 0.1, None) == pkv.PKV_ERR_INVALID      # null
    assert w(None, None, None, None, None, 0, 8, 128, 32, 64, 0.1, 0.1, None) == pkv.PKV_OK

    def dec(S=2, Hq=32, Hkv=8, D=128, B=16, maxB=4, NB=16, maxL=64, scale=0.1, ks=0.05, vs=0.05):
        return lib.paged_attention_decode_fp8(None, None, None, None, None, None, S, Hq, Hkv, D, B, maxB,
                                              NB, maxL, scale, ks, vs, None, 0, None)
    assert dec(D=64) == pkv.PKV_ERR_UNSUPPORTED
    assert dec(B=8) == pkv.PKV_ERR_UNSUPPORTED
    assert dec(Hq=72) == pkv.PKV_ERR_UNSUPPORTED       # 9 query heads per KV head
    assert dec(S=9000) == pkv.PKV_ERR_UNSUPPORTED      # more sequences than the balanced scan holds
    assert dec(Hq=30) == pkv.PKV_ERR_INVALID
    assert dec(ks=-1.0) == pkv.PKV_ERR_INVALID
    assert dec(vs=float("nan")) == pkv.PKV_ERR_INVALID
    assert dec(scale=float("inf")) == pkv.PKV_ERR_INVALID
    assert dec(S=0) == pkv.PKV_OK
    assert dec() == pkv.PKV_ERR_INVALID                # null pointers


def test_multi_token_host_validation_and_workspace():
    lib = _lib.load()
    f = lib.paged_attention_multi_token

    def call(S=2, T=10, Hq=32, Hkv=8, D=128, B=16, maxB=8, NB=64, maxQ=5, maxL=128, scale=0.1):
        return f(None, None, None, None, None, None, None, S, T, Hq, Hkv, D, B, maxB, NB, maxQ, maxL, scale,
                 None, 0, None)
    assert call(D=96) == pkv.PKV_ERR_UNSUPPORTED
    assert call(B=12) == pkv.PKV_ERR_UNSUPPORTED
    assert call(Hq=72) == pkv.PKV_ERR_UNSUPPORTED        # 9 query heads per KV head
    assert call(Hq=30) == pkv.PKV_ERR_INVALID
    assert call(scale=float("nan")) == pkv.PKV_ERR_INVALID
    assert call(T=-1) == pkv.PKV_ERR_INVALID
    assert call(S=0) == pkv.PKV_OK and call(T=0) == pkv.PKV_OK
    assert call(maxQ=0) == pkv.PKV_ERR_INVALID
    assert call() == pkv.PKV_ERR_INVALID                 # null pointers
    # the tiles of a launch's sequences (every query block of every KV head) are
    # counted in 32-bit integers: checked on the host after the pointers (dummy,
    # 16-byte aligned, never dereferenced: the call is rejected before any launch)
    p = ctypes.c_void_p(256)
    assert f(p, p, p, p, p, p, p, 4000, 10, 32, 8, 128, 16, 8, 64, 32768, 1 << 20, 0.1, p, 1 << 30,
             None) == pkv.PKV_ERR_UNSUPPORTED
    ws = lib.paged_attention_multi_token_workspace_size
    # one slot per CTA (at most 256): 256 rows (a paired context) of a partial
    # (o, max, sum) fp32 and a ready flag, whatever the number of query tokens or
    # the context length
    r = lambda x: (x + 255) // 256 * 256
    fixed = 256 * 256 * 128 * 4 + r(256 * 256 * 2 * 4) + r(256 * 8)
    assert ws(10, 32, 128, 1024) == ws(10, 32, 128, 3000) == ws(5000, 8, 128, 100000) == fixed
    assert ws(10, 32, 64, 3000) == 256 * 256 * 64 * 4 + r(256 * 256 * 2 * 4) + r(256 * 8)
    assert ws(0, 32, 128, 3000) == 0 and ws(10, 32, 96, 3000) == 0
    # grouped calls: 128 rows per slot
    assert lib.paged_attention_grouped_workspace_size(256, 64, 128, 1300) == \
        256 * 128 * 128 * 4 + r(256 * 128 * 2 * 4) + r(256 * 8)


def test_decode_append_fp8_host_validation():
    lib = _lib.load()
    f = lib.paged_attention_decode_append_fp8

    def call(S=2, D=128, B=16, knew=True, maxL=64, ks=0.1):
        k = ctypes.c_void_p(16) if knew else None
        return f(None, None, k, k, None, None, None, None, S, 32, 8, D, B, 4, 16, maxL, 0.1, ks, 0.1, None, 0, None)
    assert call(knew=False) == pkv.PKV_ERR_INVALID        # no new tokens to store
    assert call(maxL=0) == pkv.PKV_ERR_INVALID            # every context holds its new token
    assert call(D=64) == pkv.PKV_ERR_UNSUPPORTED
    assert call(ks=0.0) == pkv.PKV_ERR_INVALID
    assert call(S=0) == pkv.PKV_OK
    assert call() == pkv.PKV_ERR_INVALID                  # null q / out / caches


def test_workspace_size_formula():
    lib = _lib.load()
    # a single partition needs no scratch
    assert lib.paged_attention_workspace_size(64, 32, 128, 512, 512) == 0
    # 8 sequences x 32 heads x 32 partitions: o (fp32, 128 wide) + max + sum
    n = 8 * 32 * 32
    want = n * 128 * 4 + ((n * 4 + 255) // 256) * 256 * 2
    assert lib.paged_attention_workspace_size(8, 32, 128, 16000, 512) == want
    # partition_size 0: the balanced split, ceil(16000 / 256) + 1 = 64 slots per
    # (sequence, head) and an 8-byte ready flag per slot
    n0 = 8 * 32 * 64
    r = lambda x: (x + 255) // 256 * 256
    assert lib.paged_attention_workspace_size(8, 32, 128, 16000, 0) == \
        n0 * 128 * 4 + 2 * r(n0 * 4) + r(n0 * 8)
    assert lib.paged_attention_workspace_size(8, 32, 128, 300, 0) > 0  # may split anywhere
    assert lib.paged_attention_workspace_size(8, 32, 128, 16000, 24) == 0    # invalid partition
