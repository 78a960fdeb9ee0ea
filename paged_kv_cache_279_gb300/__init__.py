"""Paged KV cache for GB300: Python binding of libpkv (include/pkv.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels or its C++ allocator.  PyTorch supplies device memory and the
current CUDA stream.  If the library has not been built the calls raise; there
is no CPU or PyTorch fallback.

    kv_cache_write(k_new, v_new, k_cache, v_cache, slot_mapping)
    paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens,
                           scale, max_seq_len, partition_size=0, workspace=None)
    paged_attention_decode_append(...)    # store the step's new tokens, then attend
    paged_attention_decode_grouped(...)   # beams sharing prefix blocks: each read once
    paged_attention_multi_token(...)      # several causal query tokens per sequence
    kv_cache_write_fp8(...), paged_attention_decode_fp8(...),
    paged_attention_decode_append_fp8(...)  # E4M3 cache, per-tensor scales
    block_copy(k_caches, v_caches, block_pairs)
    BlockAllocator(num_blocks, block_size)   # host allocator: CoW, prefix cache, truncation
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from . import _lib

(PKV_OK, PKV_ERR_INVALID, PKV_ERR_OOM, PKV_ERR_CUDA, PKV_ERR_UNSUPPORTED, PKV_ERR_TIMEOUT,
 PKV_ERR_TOO_LARGE) = range(7)
NOALLOC_SCRATCH_BYTES = 16 << 20
PKV_F32, PKV_BF16 = 0, 1
DEVERR_BLOCK_ID, DEVERR_SEQ_LEN, DEVERR_SLOT, DEVERR_COPY_PAIR, DEVERR_TIMEOUT, DEVERR_PREFIX = (
    1, 2, 4, 8, 16, 32)

__all__ = [
    "PkvError", "kv_cache_write", "kv_cache_write_fp8", "paged_attention_decode",
    "paged_attention_decode_fp8", "paged_attention_decode_append_fp8", "paged_attention_workspace_size",
    "paged_attention_multi_token", "paged_attention_multi_token_workspace_size",
    "paged_attention_decode_append", "paged_attention_decode_grouped",
    "paged_attention_grouped_workspace_size", "block_copy", "read_device_errors", "BlockAllocator",
    "library_path",
]


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        msg = _lib.load().pkv_status_string(int(status)).decode()
        super().__init__(f"{what}: {msg} (status {status})")


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)


def library_path() -> str:
    return _lib.library_path()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def kv_cache_write(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Scatter new K/V rows [T, Hkv, D] into the caches [NB, Hkv, B, D] at
    slot_mapping[t] (int64; negative = skip)."""
    lib = _lib.load()
    NB, Hkv, B, D = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, Hkv, D) or k_new.shape != v_new.shape or k_cache.shape != v_cache.shape:
        raise ValueError("shape mismatch between new tokens and caches")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping needs one entry per token")
    dt = _dtype_code(k_cache)
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (v_cache, "v_cache")):
        if t.dtype != k_cache.dtype:
            raise TypeError(f"{n} dtype differs from k_cache")
    st = lib.kv_cache_write(_dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
                            _dev(v_cache, "v_cache"), _dev(slot_mapping, "slot_mapping", torch.int64, 1),
                            T, Hkv, D, B, NB, dt, _stream(stream))
    _check(st, "kv_cache_write")


def paged_attention_workspace_size(num_seqs: int, num_heads: int, head_dim: int,
                                   max_seq_len: int, partition_size: int = 0) -> int:
    return int(_lib.load().paged_attention_workspace_size(num_seqs, num_heads, head_dim,
                                                          max_seq_len, partition_size))


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                           max_seq_len: int, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[s, h] = softmax(scale * q[s, h] . K_s^T) V_s over the paged cache.

    q/out [S, Hq, D]; caches [NB, Hkv, B, D]; block_tables int32 [S, maxB];
    seq_lens int32 [S].  ``workspace`` (uint8 CUDA tensor) is allocated from
    PyTorch's caching allocator when not given."""
    lib = _lib.load()
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if Dk != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables must be [S, maxB] and seq_lens [S]")
    dt = _dtype_code(q)
    for t, n in ((out, "out"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if t.dtype != q.dtype:
            raise TypeError(f"{n} dtype differs from q")
    need = paged_attention_workspace_size(S, Hq, D, max_seq_len, partition_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.paged_attention_decode(
        _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32, 2), _dev(seq_lens, "seq_lens", torch.int32, 1),
        S, Hq, Hkv, D, B, block_tables.shape[1], NB, int(max_seq_len), float(scale),
        int(partition_size), ws_ptr, ws_bytes, dt, _stream(stream))
    _check(st, "paged_attention_decode")
    return out


def paged_attention_multi_token_workspace_size(num_q_tokens: int, num_heads: int, head_dim: int,
                                               max_seq_len: int) -> int:
    return int(_lib.load().paged_attention_multi_token_workspace_size(num_q_tokens, num_heads, head_dim,
                                                                      max_seq_len))


def paged_attention_multi_token(out, q, k_cache, v_cache, block_tables, seq_lens, q_starts, scale: float,
                                max_q_len: int, max_seq_len: int, workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """Causal attention of each sequence's last Q_s positions (chunked prefill,
    verification of drafted tokens): q/out bf16 [T, Hq, D] with sequence s
    owning rows q_starts[s] .. q_starts[s+1]-1 (int32 [S+1]); caches
    [NB, Hkv, B, D]; block_tables int32 [S, maxB]; seq_lens int32 [S] (the
    contexts including the query tokens)."""
    lib = _lib.load()
    T, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    S = seq_lens.shape[0]
    if Dk != D or tuple(out.shape) != (T, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or q_starts.shape[0] != S + 1:
        raise ValueError("block_tables must be [S, maxB] and q_starts [S + 1]")
    need = paged_attention_multi_token_workspace_size(T, Hq, D, max_seq_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.paged_attention_multi_token(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache", torch.bfloat16),
        _dev(v_cache, "v_cache", torch.bfloat16), _dev(block_tables, "block_tables", torch.int32, 2),
        _dev(seq_lens, "seq_lens", torch.int32, 1), _dev(q_starts, "q_starts", torch.int32, 1), S, T, Hq, Hkv,
        D, B, block_tables.shape[1], NB, int(max_q_len), int(max_seq_len), float(scale), ws_ptr, ws_bytes,
        _stream(stream))
    _check(st, "paged_attention_multi_token")
    return out


def kv_cache_write_fp8(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float,
                       stream=None) -> None:
    """Quantise bf16 K/V rows [T, Hkv, D] to E4M3 codes and store them: K in
    k_cache uint8 [NB, Hkv, B, D], V transposed in v_cache uint8 [NB, Hkv, D, B]
    (code = e4m3(x / scale), nearest even, saturating)."""
    lib = _lib.load()
    NB, Hkv, B, D = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, Hkv, D) or k_new.shape != v_new.shape or \
            tuple(v_cache.shape) != (NB, Hkv, D, B):
        raise ValueError("shape mismatch between new tokens and FP8 caches")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping needs one entry per token")
    st = lib.kv_cache_write_fp8(
        _dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16),
        _dev(k_cache, "k_cache", torch.uint8), _dev(v_cache, "v_cache", torch.uint8),
        _dev(slot_mapping, "slot_mapping", torch.int64, 1), T, Hkv, D, B, NB,
        float(k_scale), float(v_scale), _stream(stream))
    _check(st, "kv_cache_write_fp8")


def paged_attention_decode_fp8(out, q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                               k_scale: float, v_scale: float, max_seq_len: int,
                               workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention over an FP8 (E4M3) cache: K codes [NB, Hkv, B, D], V
    codes transposed [NB, Hkv, D, B], values code * k_scale / code * v_scale.
    q/out bf16 [S, Hq, D]; block_tables int32 [S, maxB]; seq_lens int32 [S]."""
    lib = _lib.load()
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if Dk != D or tuple(out.shape) != (S, Hq, D) or tuple(v_cache.shape) != (NB, Hkv, D, B):
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables must be [S, maxB] and seq_lens [S]")
    need = paged_attention_workspace_size(S, Hq, D, max_seq_len, 0)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.paged_attention_decode_fp8(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache", torch.uint8),
        _dev(v_cache, "v_cache", torch.uint8), _dev(block_tables, "block_tables", torch.int32, 2),
        _dev(seq_lens, "seq_lens", torch.int32, 1), S, Hq, Hkv, D, B, block_tables.shape[1], NB,
        int(max_seq_len), float(scale), float(k_scale), float(v_scale), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "paged_attention_decode_fp8")
    return out


def paged_attention_decode_append_fp8(out, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                      scale: float, k_scale: float, v_scale: float, max_seq_len: int,
                                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One FP8 decode step: quantise and store each sequence's new token (bf16
    k_new/v_new [S, Hkv, D]) at position seq_lens[s] - 1, then attend; the
    store happens inside the attention kernel."""
    lib = _lib.load()
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if Dk != D or tuple(out.shape) != (S, Hq, D) or tuple(v_cache.shape) != (NB, Hkv, D, B):
        raise ValueError("shape mismatch")
    if tuple(k_new.shape) != (S, Hkv, D) or k_new.shape != v_new.shape:
        raise ValueError("k_new / v_new must be [S, Hkv, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables must be [S, maxB] and seq_lens [S]")
    need = paged_attention_workspace_size(S, Hq, D, max_seq_len, 0)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.paged_attention_decode_append_fp8(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_new, "k_new", torch.bfloat16),
        _dev(v_new, "v_new", torch.bfloat16), _dev(k_cache, "k_cache", torch.uint8),
        _dev(v_cache, "v_cache", torch.uint8), _dev(block_tables, "block_tables", torch.int32, 2),
        _dev(seq_lens, "seq_lens", torch.int32, 1), S, Hq, Hkv, D, B, block_tables.shape[1], NB,
        int(max_seq_len), float(scale), float(k_scale), float(v_scale), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "paged_attention_decode_append_fp8")
    return out


def paged_attention_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                  scale: float, max_seq_len: int, partition_size: int = 0,
                                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step: store k_new[s] / v_new[s] ([S, Hkv, D]) at position
    seq_lens[s] - 1 of each sequence, then attend as paged_attention_decode."""
    lib = _lib.load()
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if Dk != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if tuple(k_new.shape) != (S, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [S, Hkv, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables must be [S, maxB] and seq_lens [S]")
    dt = _dtype_code(q)
    for t, n in ((out, "out"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        if t.dtype != q.dtype:
            raise TypeError(f"{n} dtype differs from q")
    need = paged_attention_workspace_size(S, Hq, D, max_seq_len, partition_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.paged_attention_decode_append(
        _dev(out, "out"), _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32, 2), _dev(seq_lens, "seq_lens", torch.int32, 1),
        S, Hq, Hkv, D, B, block_tables.shape[1], NB, int(max_seq_len), float(scale),
        int(partition_size), ws_ptr, ws_bytes, dt, _stream(stream))
    _check(st, "paged_attention_decode_append")
    return out


def paged_attention_grouped_workspace_size(num_seqs: int, num_heads: int, head_dim: int,
                                           max_seq_len: int) -> int:
    return int(_lib.load().paged_attention_grouped_workspace_size(num_seqs, num_heads, head_dim,
                                                                  max_seq_len))


def paged_attention_decode_grouped(out, q, k_cache, v_cache, block_tables, seq_lens, group_offsets,
                                   prefix_lens, scale: float, max_seq_len: int, k_new=None, v_new=None,
                                   workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode where the sequences of group g (group_offsets[g] .. [g+1]-1,
    int32 on the device) share the blocks of their first prefix_lens[g]
    tokens; each shared block is read once for the whole group.  With k_new /
    v_new the new tokens are stored first, as in paged_attention_decode_append."""
    lib = _lib.load()
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if Dk != D or tuple(out.shape) != (S, Hq, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables must be [S, maxB] and seq_lens [S]")
    G = prefix_lens.shape[0]
    if group_offsets.shape[0] != G + 1:
        raise ValueError("group_offsets needs num_groups + 1 entries")
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new, or neither")
    if k_new is not None and (tuple(k_new.shape) != (S, Hkv, D) or v_new.shape != k_new.shape):
        raise ValueError("k_new/v_new must be [S, Hkv, D]")
    need = paged_attention_grouped_workspace_size(S, Hq, D, max_seq_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.paged_attention_decode_grouped(
        _dev(out, "out"), _dev(q, "q"),
        _dev(k_new, "k_new") if k_new is not None else None,
        _dev(v_new, "v_new") if v_new is not None else None,
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32, 2), _dev(seq_lens, "seq_lens", torch.int32, 1),
        _dev(group_offsets, "group_offsets", torch.int32, 1), _dev(prefix_lens, "prefix_lens", torch.int32, 1),
        G, S, Hq, Hkv, D, B, block_tables.shape[1], NB, int(max_seq_len), float(scale), ws_ptr, ws_bytes,
        _dtype_code(q), _stream(stream))
    _check(st, "paged_attention_decode_grouped")
    return out


def block_copy(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
               block_pairs: torch.Tensor, stream=None) -> None:
    """For every layer, K and V: block dst := block src for each (src, dst)
    row of block_pairs (int64 [N, 2] on the device)."""
    lib = _lib.load()
    L = len(k_caches)
    if len(v_caches) != L:
        raise ValueError("one V cache per K cache")
    if L == 0:
        return
    NB = k_caches[0].shape[0]
    block_bytes = k_caches[0][0].numel() * k_caches[0].element_size()
    for t in list(k_caches) + list(v_caches):
        if t.shape != k_caches[0].shape or t.dtype != k_caches[0].dtype:
            raise ValueError("all caches must share shape and dtype")
    if block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be [N, 2]")
    kp = (ctypes.c_void_p * L)(*[_dev(t, "k_cache") for t in k_caches])
    vp = (ctypes.c_void_p * L)(*[_dev(t, "v_cache") for t in v_caches])
    st = lib.block_copy(kp, vp, L, _dev(block_pairs, "block_pairs", torch.int64, 2),
                        block_pairs.shape[0], NB, block_bytes, _stream(stream))
    _check(st, "block_copy")


def read_device_errors(clear: bool = True, stream=None) -> int:
    """PKV_DEVERR_* bits raised by kernels since the last clear (waits for the stream)."""
    flags = ctypes.c_uint32(0)
    _check(_lib.load().pkv_read_device_errors(ctypes.byref(flags), int(clear), _stream(stream)),
           "pkv_read_device_errors")
    return int(flags.value)


def bounded_wait_check(flags: Optional[torch.Tensor], tag: int, arrive: bool, polls: int,
                       stream=None) -> None:
    """Runs the attention kernels' two bounded waits once with `polls` as the
    limit: the flag wait on the int64 words of `flags` (None: skipped) for
    `tag`, then an mbarrier wait that completes only with `arrive`.  A wait
    that runs out sets DEVERR_TIMEOUT (read_device_errors)."""
    ptr, n = 0, 0
    if flags is not None:
        ptr, n = _dev(flags, "flags", torch.int64, 1), flags.numel()
    _check(_lib.load().pkv_bounded_wait_check(ptr, n, int(tag), int(bool(arrive)), int(polls), _stream(stream)),
           "pkv_bounded_wait_check")


class BlockAllocator:
    """Host block allocator (C++): free stack, block tables, refcounts, CoW."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _lib.load()
        self._h = self._lib.block_allocator_create(int(num_blocks), int(block_size))
        if not self._h:
            raise PkvError(PKV_ERR_INVALID, "block_allocator_create")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.block_allocator_destroy(h)
            self._h = None

    def add_seq(self, seq: int, num_tokens: int) -> int:
        return self._lib.block_allocator_add_seq(self._h, int(seq), int(num_tokens))

    def add_seq_cached(self, seq: int, tokens):
        """A prompt whose leading full blocks may already be in the pool
        (prefix caching).  Returns (status, cached_tokens): the caller writes
        K/V for positions cached_tokens .. len(tokens) - 1 only."""
        ids = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        cached = ctypes.c_int64(0)
        st = self._lib.block_allocator_add_seq_cached(self._h, int(seq), ids.ctypes.data if ids.size else None,
                                                      int(ids.size), ctypes.byref(cached))
        return st, int(cached.value)

    def cache_stats(self) -> dict:
        """Prefix cache counters: hits, misses, cached_blocks, evictable_blocks."""
        h, m = ctypes.c_int64(0), ctypes.c_int64(0)
        c, e = ctypes.c_int(0), ctypes.c_int(0)
        _check(self._lib.block_allocator_cache_stats(self._h, ctypes.byref(h), ctypes.byref(m), ctypes.byref(c),
                                                     ctypes.byref(e)), "cache_stats")
        return {"hits": h.value, "misses": m.value, "cached_blocks": c.value, "evictable_blocks": e.value}

    def cache_clear(self) -> int:
        return self._lib.block_allocator_cache_clear(self._h)

    def append_slot(self, seq: int):
        """(status, slot, cow_src, cow_dst)."""
        slot, src, dst = ctypes.c_int64(-1), ctypes.c_int32(-1), ctypes.c_int32(-1)
        st = self._lib.block_allocator_append_slot(self._h, int(seq), ctypes.byref(slot),
                                                   ctypes.byref(src), ctypes.byref(dst))
        return st, slot.value, src.value, dst.value

    def append_slots(self, seqs):
        """One token for each of the distinct sequences ``seqs``.  Returns
        (status, slots int64 [n], cow_pairs int64 [k, 2])."""
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        slots = np.full(len(ids), -1, dtype=np.int64)
        pairs = np.empty((max(1, len(ids)), 2), dtype=np.int64)
        ncow = ctypes.c_int(0)
        st = self._lib.block_allocator_append_slots(self._h, ids.ctypes.data, len(ids),
                                                    slots.ctypes.data, pairs.ctypes.data,
                                                    ctypes.byref(ncow))
        return st, slots, pairs[:ncow.value]

    def append_step(self, seqs, tables: np.ndarray, lens: np.ndarray):
        """append_slots that also updates the dense tables (int32 [n, cap],
        row i for seqs[i]) and lens (int32 [n]) in place, writing only the
        entry of each new token's block.  Both arrays must be C-contiguous
        (pinned host views are fine).  Returns (status, slots, cow_pairs)."""
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        if (tables.dtype != np.int32 or lens.dtype != np.int32 or tables.ndim != 2 or
                not tables.flags.c_contiguous or not lens.flags.c_contiguous or
                tables.shape[0] != len(ids) or lens.shape[0] != len(ids)):
            raise ValueError("tables must be int32 [n, cap] and lens int32 [n], C-contiguous")
        slots = np.full(len(ids), -1, dtype=np.int64)
        pairs = np.empty((max(1, len(ids)), 2), dtype=np.int64)
        ncow = ctypes.c_int(0)
        st = self._lib.block_allocator_append_step(self._h, ids.ctypes.data, len(ids), tables.ctypes.data,
                                                   tables.shape[1], lens.ctypes.data, slots.ctypes.data,
                                                   pairs.ctypes.data, ctypes.byref(ncow))
        return st, slots, pairs[:ncow.value]

    def extend(self, seq: int, count: int):
        """Slots for ``count`` more tokens of seq (all or nothing).  Returns
        (status, slots int64 [count], cow_src, cow_dst)."""
        slots = np.zeros(max(int(count), 1), dtype=np.int64)
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        st = int(self._lib.block_allocator_extend(self._h, int(seq), int(count),
                                                  slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                                  ctypes.byref(src), ctypes.byref(dst)))
        if st != PKV_OK:
            return st, slots[:0], -1, -1
        return st, slots[:int(count)], int(src.value), int(dst.value)

    def truncate(self, seq: int, num_tokens: int) -> int:
        """Keep the first num_tokens tokens of seq (roll back rejected drafts)."""
        return int(self._lib.block_allocator_truncate(self._h, int(seq), int(num_tokens)))

    def fork(self, parent: int, child: int) -> int:
        return self._lib.block_allocator_fork(self._h, int(parent), int(child))

    def free_seq(self, seq: int) -> int:
        return self._lib.block_allocator_free_seq(self._h, int(seq))

    def num_tokens(self, seq: int) -> int:
        return int(self._lib.block_allocator_num_tokens(self._h, int(seq)))

    def block_table(self, seq: int):
        n = self.num_tokens(seq)
        if n < 0:
            raise PkvError(PKV_ERR_INVALID, "block_table")
        cap = max(1, -(-n // self.block_size) + 1)
        buf = np.empty(cap, dtype=np.int32)
        cnt = ctypes.c_int(0)
        _check(self._lib.block_allocator_block_table(self._h, int(seq), buf.ctypes.data, cap,
                                                     ctypes.byref(cnt)), "block_table")
        return buf[:cnt.value].tolist()

    def block_tables(self, seqs, cap: int, pad: int = -1):
        """(tables int32 [n, cap], seq_lens int32 [n]) as numpy arrays."""
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        tables = np.empty((len(ids), max(1, cap)), dtype=np.int32)
        lens = np.empty(len(ids), dtype=np.int32)
        _check(self._lib.block_allocator_block_tables(self._h, ids.ctypes.data, len(ids),
                                                      tables.ctypes.data, tables.shape[1],
                                                      int(pad), lens.ctypes.data), "block_tables")
        return tables, lens

    def prefix_groups(self, seqs):
        """(group_offsets int32 [G + 1], prefix_lens int32 [G]) for the
        sequences in the given order (runs that start with the same blocks)."""
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        offs = np.zeros(len(ids) + 1, dtype=np.int32)
        pre = np.zeros(max(1, len(ids)), dtype=np.int32)
        ng = ctypes.c_int(0)
        _check(self._lib.block_allocator_prefix_groups(self._h, ids.ctypes.data, len(ids), offs.ctypes.data,
                                                       pre.ctypes.data, ctypes.byref(ng)), "prefix_groups")
        return offs[:ng.value + 1].copy(), pre[:ng.value].copy()

    def slots(self, seq: int, start: int, count: int) -> np.ndarray:
        out = np.empty(max(0, count), dtype=np.int64)
        _check(self._lib.block_allocator_slots(self._h, int(seq), int(start), int(count),
                                               out.ctypes.data), "slots")
        return out

    def num_free(self) -> int:
        return int(self._lib.block_allocator_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.block_allocator_refcount(self._h, int(block)))

    def waste(self):
        used, alloc = ctypes.c_int64(0), ctypes.c_int64(0)
        _check(self._lib.block_allocator_waste(self._h, ctypes.byref(used), ctypes.byref(alloc)),
               "waste")
        return used.value, alloc.value
