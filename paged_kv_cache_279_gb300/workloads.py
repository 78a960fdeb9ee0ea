"""Seeded synthetic workloads for the tests and the benchmark.

This module only draws data: context lengths, query/key/value values and
random physical block ids.  It holds none of the method's arithmetic (no slot
computation, no cache placement, no attention), so both the CUDA path and the
CPU oracle can be fed from it without sharing code.

The shapes mirror the serving workloads behind the pages' claims: chat
requests whose answers are mostly 50-200 tokens long, contexts of thousands of
tokens, beam search over a shared prompt, and a continuous-batching mix of
short and long requests.  No dataset is involved; every value is N(0, 1) and
every draw is reproducible from its seed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

_MASK64 = (1 << 64) - 1


def sub_seed(seed: int, *keys: int) -> int:
    """A 63-bit seed derived from ``seed`` and integer keys (SplitMix64 mixing),
    so that any one sequence's data can be regenerated on its own."""
    x = (int(seed) * 0x9E3779B97F4A7C15) & _MASK64
    for k in keys:
        x = (x + 0x9E3779B97F4A7C15 + (int(k) & _MASK64)) & _MASK64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        x = z ^ (z >> 31)
    return x & ((1 << 63) - 1)


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    """One decode workload: S sequences, Hq query heads over Hkv KV heads."""
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    num_layers: int = 1
    partition_size: int = 0  # 0: let the library choose

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The five workloads (tiny fp32, GQA decode, long context, beam search with
# copy-on-write, continuous-batching mix).  Lengths are drawn by draw_lengths.
TINY_FP32 = DecodeShape("tiny_fp32", 4, 4, 4, 64, 16, torch.float32)
GQA_BF16 = DecodeShape("gqa_decode_bf16", 64, 32, 8, 128, 16, torch.bfloat16)
LONG_BF16 = DecodeShape("long_context_bf16", 8, 32, 8, 128, 16, torch.bfloat16,
                        num_layers=32, partition_size=512)
BEAM_BF16 = DecodeShape("beam_cow_bf16", 256, 64, 8, 128, 16, torch.bfloat16)
MIXED_BF16 = DecodeShape("mixed_batch_bf16", 256, 32, 8, 128, 16, torch.bfloat16,
                         num_layers=32)

TINY_LENGTHS = (1, 17, 33, 100)
BEAM_PROMPTS = 32
BEAM_WIDTH = 8
BEAM_SHARED = 1024
BEAM_SHARED_PARTIAL = 1032  # variant whose shared prefix ends inside a block
BEAM_MAX_DIVERGENT = 256


def draw_lengths(shape: DecodeShape, seed: int, num_seqs: Optional[int] = None) -> np.ndarray:
    """Context lengths (after the current token is written) for a workload."""
    n = shape.num_seqs if num_seqs is None else num_seqs
    rng = np.random.default_rng(sub_seed(seed, 1))
    if shape.name == TINY_FP32.name:
        return np.array(TINY_LENGTHS[:n], dtype=np.int64)
    if shape.name == GQA_BF16.name:
        return rng.integers(64, 2048, size=n, endpoint=True).astype(np.int64)
    if shape.name == LONG_BF16.name:
        return np.full(n, 16000, dtype=np.int64)
    if shape.name == MIXED_BF16.name:
        x = np.round(rng.lognormal(mean=math.log(150.0), sigma=1.0, size=n))
        return np.clip(x, 1, 32768).astype(np.int64)
    if shape.name == BEAM_BF16.name:
        return rng.integers(0, BEAM_MAX_DIVERGENT, size=n, endpoint=True).astype(np.int64)
    raise ValueError(f"no length law for {shape.name}")


def draw_divergent_lengths(num_beams_total: int, seed: int) -> np.ndarray:
    """Tokens each beam generated after the shared prompt, uniform in [0, 256]."""
    rng = np.random.default_rng(sub_seed(seed, 2))
    return rng.integers(0, BEAM_MAX_DIVERGENT, size=num_beams_total, endpoint=True).astype(np.int64)


def draw_normal(shape_, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """N(0, 1) values rounded to the storage dtype, on the host."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape_, generator=g, dtype=torch.float32).to(dtype)


def draw_query(shape: DecodeShape, seed: int, num_seqs: Optional[int] = None, layer: int = 0) -> torch.Tensor:
    n = shape.num_seqs if num_seqs is None else num_seqs
    return draw_normal((n, shape.num_heads, shape.head_dim), shape.dtype, sub_seed(seed, 3, layer))


def draw_seq_kv(shape: DecodeShape, seed: int, seq: int, length: int, layer: int = 0):
    """Contiguous K and V of one sequence, each [length, Hkv, D]."""
    k = draw_normal((length, shape.num_kv_heads, shape.head_dim), shape.dtype, sub_seed(seed, 4, layer, seq))
    v = draw_normal((length, shape.num_kv_heads, shape.head_dim), shape.dtype, sub_seed(seed, 5, layer, seq))
    return k, v


def draw_e4m3_codes(shape_, seed: int, exp_center: float = 11.0, exp_sigma: float = 1.5) -> np.ndarray:
    """Random 8-bit E4M3 bit patterns (uint8) for an FP8 cache.

    Drawn field by field -- a fair sign bit, an exponent field from a rounded
    normal clipped to 0..15, a uniform 3-bit mantissa -- with the NaN pattern
    (all exponent and mantissa bits set) replaced by the largest finite one.
    The default centre (field 11, magnitudes around 16-32) matches N(0, 1)
    data quantised with a scale of about 1/32.
    """
    rng = np.random.default_rng(sub_seed(seed, 7))
    n = int(np.prod(shape_))
    sign = rng.integers(0, 2, n, dtype=np.int64)
    e = np.clip(np.rint(rng.normal(exp_center, exp_sigma, n)), 0, 15).astype(np.int64)
    m = rng.integers(0, 8, n, dtype=np.int64)
    m = np.where((e == 15) & (m == 7), 6, m)
    return ((sign << 7) | (e << 3) | m).astype(np.uint8).reshape(shape_)


def draw_block_ids(num_blocks: int, seed: int) -> np.ndarray:
    """A random order of the physical block ids 0..num_blocks-1."""
    rng = np.random.default_rng(sub_seed(seed, 6))
    return rng.permutation(num_blocks).astype(np.int32)


def random_block_tables(block_counts: List[int], num_blocks: int, max_blocks: int,
                        seed: int, pad: int = -1) -> np.ndarray:
    """Block tables [S, max_blocks] int32: sequence s receives block_counts[s]
    distinct physical ids taken in random order from the pool; unused entries
    hold ``pad``."""
    if sum(block_counts) > num_blocks:
        raise ValueError("pool too small for the requested blocks")
    ids = draw_block_ids(num_blocks, seed)
    tables = np.full((len(block_counts), max(1, max_blocks)), pad, dtype=np.int32)
    pos = 0
    for s, n in enumerate(block_counts):
        tables[s, :n] = ids[pos:pos + n]
        pos += n
    return tables
