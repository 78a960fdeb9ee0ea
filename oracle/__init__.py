"""CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library never imports, links or calls it, and it imports nothing from the CUDA
library.  Inputs reach both sides from the seeded generators in
``paged_kv_cache_279_gb300.workloads`` (data only, no arithmetic of the method).

Contents and the passages they follow (page titles as given at each address):

* ``decode_attention`` -- fp64 decode attention over contiguous per-sequence
  K/V (C code in ``pkv_oracle.c``).  "KV cache & PagedAttention -- vi sao
  chatbot AI ton bo nho" (aiwiki.vn), second and third paragraphs (query vs
  the keys of visible positions, weights combine the values; K/V come from the
  cache).  "PagedAttention (vLLM) -- Virtual memory cho AI", section "Y tuong
  cot loi": physical placement is irrelevant, so no block table appears here.
* ``kv_cache_write`` / ``slot_of`` -- store one new token's K/V at
  ``slot = physical_block * block_size + offset``.  Same troisinh page,
  section "Co che Block Table" (block granularity, logical -> physical map,
  allocation when a token is produced).
* ``block_copy`` -- copy whole physical blocks (copy-on-write).  Same page,
  section "Copy-on-Write cho Beam Search".
* ``kv_cache_bytes`` -- the KV-memory closed form, aiwiki.vn page, fourth
  paragraph (2 x layers x tokens x kv_heads x head_dim x bytes).
* ``blocks_needed``, ``paged_waste_fraction``, ``preallocation_waste_fraction``
  -- troisinh page, sections "Co che Block Table" (100 tokens -> 7 blocks of
  16 = 112 slots, versus 256 blocks reserved for 4096) and "Y nghia thuc te"
  (waste remains only in each sequence's last block).
* ``BlockAllocatorModel`` (``block_allocator_model.py``) -- the allocator's
  host semantics.
* ``multi_token`` -- causal attention of several new tokens per sequence
  (chunked prefill, verification of drafted tokens).  hada.io page, list of
  advanced features; the causal reading is in that module.
* ``fp8_e4m3`` -- the FP8 (E4M3) KV cache: quantiser, dequantiser and cache
  write.  aiwiki.vn page, paragraph on quantisation and offloading (K/V kept
  in a lower-precision representation to cut bytes, at a conversion cost and
  an error risk); the format and scaling readings are in that module.

Every function is pinned by ``tests/test_oracle_pins.py`` to values the pages
print, closed forms, invariants or an independent library routine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .block_allocator_model import (  # noqa: F401
    BlockAllocatorModel, OK, ERR_INVALID, ERR_OOM,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_pkv.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP when available); return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_decode_attention.restype = ctypes.c_int
            lib.oracle_decode_attention.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def decode_attention(q, k_seqs, v_seqs, scale, return_weight_error=False):
    """Decode attention, fp64, over contiguous per-sequence K/V.

    q: [S, Hq, D]; k_seqs[s], v_seqs[s]: [L_s, Hkv, D] (any float dtype; values
    are widened exactly to fp64).  Returns out [S, Hq, D] float64 (and, if
    asked, |sum of softmax weights - 1| per (s, h)).
    """
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    S, Hq, D = q.shape
    if len(k_seqs) != S or len(v_seqs) != S:
        raise ValueError("one K and one V array per sequence")
    lens = np.array([int(np.shape(k)[0]) for k in k_seqs], dtype=np.int64)
    Hkv = int(np.shape(k_seqs[0])[1]) if S else 1
    starts = np.zeros(S, dtype=np.int64)
    if S > 1:
        starts[1:] = np.cumsum(lens)[:-1]
    total = int(lens.sum())
    k = np.zeros((max(total, 1), Hkv, D), dtype=np.float64)
    v = np.zeros((max(total, 1), Hkv, D), dtype=np.float64)
    for s in range(S):
        if lens[s]:
            if tuple(np.shape(k_seqs[s])) != (lens[s], Hkv, D) or \
                    tuple(np.shape(v_seqs[s])) != (lens[s], Hkv, D):
                raise ValueError("K/V of a sequence must be [L, Hkv, D]")
            k[starts[s]:starts[s] + lens[s]] = np.asarray(k_seqs[s], dtype=np.float64)
            v[starts[s]:starts[s] + lens[s]] = np.asarray(v_seqs[s], dtype=np.float64)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    err = np.zeros((S, Hq), dtype=np.float64)
    rc = _load().oracle_decode_attention(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, starts.ctypes.data,
        lens.ctypes.data, S, Hq, Hkv, D, float(scale), out.ctypes.data, err.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_decode_attention rejected its arguments")
    return (out, err) if return_weight_error else out


# --------------------------------------------------------------------------
# Cache write, block copy: plain array semantics.
# --------------------------------------------------------------------------
def slot_of(block_table_row, position, block_size):
    """Physical slot of a logical token position: the logical block
    ``position // block_size`` is looked up in the sequence's block table and the
    token keeps its offset inside the block."""
    return int(block_table_row[position // block_size]) * block_size + position % block_size


def kv_cache_write(k_cache, v_cache, k_new, v_new, slot_mapping, block_size):
    """In place: token t's K/V rows go to physical block slot//B, offset slot%B.

    Caches are [num_blocks, Hkv, block_size, D]; k_new/v_new are [T, Hkv, D].
    A negative slot means "no token here" and writes nothing.
    """
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        k_cache[blk, :, off, :] = k_new[t]
        v_cache[blk, :, off, :] = v_new[t]


def block_copy(k_caches, v_caches, pairs):
    """In place: for every layer and for K and V, block ``dst`` becomes a byte
    copy of block ``src`` for each (src, dst) pair."""
    for layer in range(len(k_caches)):
        for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
            k_caches[layer][dst] = k_caches[layer][src]
            v_caches[layer][dst] = v_caches[layer][src]


# --------------------------------------------------------------------------
# Closed forms from the pages.
# --------------------------------------------------------------------------
def kv_cache_bytes(layers, tokens, kv_heads, head_dim, elem_bytes):
    """KV memory = 2 (key and value) x layers x tokens x kv_heads x head_dim x bytes."""
    return 2 * layers * tokens * kv_heads * head_dim * elem_bytes


def blocks_needed(tokens, block_size):
    """Blocks a sequence of ``tokens`` occupies when blocks are handed out only
    as tokens are produced: the smallest count whose capacity holds them."""
    return -(-int(tokens) // int(block_size))


def paged_waste_fraction(lengths, block_size):
    """Fraction of allocated slots left empty when every sequence holds
    ceil(L / B) blocks (no sharing)."""
    lengths = [int(x) for x in lengths]
    alloc = sum(blocks_needed(x, block_size) * block_size for x in lengths)
    return 0.0 if alloc == 0 else 1.0 - sum(lengths) / alloc


def preallocation_waste_fraction(lengths, max_seq_len):
    """Fraction of reserved slots left empty when every request reserves a
    contiguous region for max_seq_len tokens up front."""
    lengths = [int(x) for x in lengths]
    alloc = len(lengths) * int(max_seq_len)
    return 0.0 if alloc == 0 else 1.0 - sum(lengths) / alloc
