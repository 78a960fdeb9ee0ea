"""ctypes declarations of the C ABI in include/pkv.h."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_int, c_int32, c_int64, c_size_t, c_float = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_size_t, ctypes.c_float)
c_void_p, c_uint32 = ctypes.c_void_p, ctypes.c_uint32
P = ctypes.POINTER

# name -> (restype, argtypes); every function the header declares.
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [c_int]),
    "pkv_abi_version": (c_int, []),
    "kv_cache_write": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                               c_int, c_int, c_int, c_int, c_void_p]),
    "kv_cache_write_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                   c_int, c_int, c_int, c_float, c_float, c_void_p]),
    "paged_attention_decode_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                           c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                           c_float, c_float, c_float, c_void_p, c_size_t, c_void_p]),
    "paged_attention_decode_append_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                  c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                                  c_int, c_int, c_int, c_int, c_int, c_float, c_float,
                                                  c_float, c_void_p, c_size_t, c_void_p]),
    "paged_attention_multi_token_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "paged_attention_multi_token": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                            c_int, c_int, c_int, c_float, c_void_p, c_size_t, c_void_p]),
    "paged_attention_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "paged_attention_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                       c_float, c_int, c_void_p, c_size_t, c_int, c_void_p]),
    "paged_attention_decode_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                              c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                              c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                              c_void_p, c_size_t, c_int, c_void_p]),
    "paged_attention_grouped_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "paged_attention_decode_grouped": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                               c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                               c_int, c_int, c_float, c_void_p, c_size_t, c_int,
                                               c_void_p]),
    "block_allocator_prefix_groups": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, P(c_int)]),
    "paged_attention_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                               c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                               c_int, c_int, c_float, c_int, c_int, c_void_p]),
    "block_copy": (c_int, [P(c_void_p), P(c_void_p), c_int, c_void_p, c_int, c_int, c_size_t,
                           c_void_p]),
    "pkv_read_device_errors": (c_int, [P(c_uint32), c_int, c_void_p]),
    "pkv_bounded_wait_check": (c_int, [c_void_p, c_int, ctypes.c_uint64, c_int, c_uint32, c_void_p]),
    "block_allocator_create": (c_void_p, [c_int, c_int]),
    "block_allocator_destroy": (None, [c_void_p]),
    "block_allocator_add_seq": (c_int, [c_void_p, c_int64, c_int64]),
    "block_allocator_extend": (c_int, [c_void_p, c_int64, c_int64, P(c_int64), P(c_int32), P(c_int32)]),
    "block_allocator_truncate": (c_int, [c_void_p, c_int64, c_int64]),
    "block_allocator_add_seq_cached": (c_int, [c_void_p, c_int64, c_void_p, c_int64, P(c_int64)]),
    "block_allocator_cache_stats": (c_int, [c_void_p, P(c_int64), P(c_int64), P(c_int), P(c_int)]),
    "block_allocator_cache_clear": (c_int, [c_void_p]),
    "block_allocator_append_slot": (c_int, [c_void_p, c_int64, P(c_int64), P(c_int32),
                                            P(c_int32)]),
    "block_allocator_append_slots": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, P(c_int)]),
    "block_allocator_append_step": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p,
                                            c_void_p, P(c_int)]),
    "block_allocator_fork": (c_int, [c_void_p, c_int64, c_int64]),
    "block_allocator_free_seq": (c_int, [c_void_p, c_int64]),
    "block_allocator_block_table": (c_int, [c_void_p, c_int64, c_void_p, c_int, P(c_int)]),
    "block_allocator_block_tables": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int32,
                                             c_void_p]),
    "block_allocator_slots": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p]),
    "block_allocator_num_tokens": (c_int64, [c_void_p, c_int64]),
    "block_allocator_num_free": (c_int, [c_void_p]),
    "block_allocator_refcount": (c_int, [c_void_p, c_int32]),
    "block_allocator_waste": (c_int, [c_void_p, P(c_int64), P(c_int64)]),
    "pkv_balanced_segment_tiles": (c_int, [c_int]),
    "pkv_rows_context_tiles": (c_int, [c_int]),
    "pkv_rows_split_parts": (c_int64, [c_int64, c_int64]),
    "pkv_balanced_slots": (c_int, [c_int]),
    "pkv_balanced_split_parts": (c_int64, [c_int64, c_int, c_int, c_int64]),
    "pkv_balanced_share_owner": (c_int64, [c_int64, c_int64, c_int64]),
}


def library_path() -> str:
    return _build.LIB


def load():
    """The loaded libpkv.so.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libpkv.so is not built ({path}); build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
