#!/usr/bin/env python
"""Benchmark of one paged decode step on GB300.

A step is the whole hot path for one batch: the host allocator hands every
running sequence the slot of its new token (copy-on-write pairs, if any, go to
block_copy), kv_cache_write scatters the new K/V into the paged pool, and
paged_attention_decode attends each sequence's query to its whole context
through the block tables (split into partitions plus a merge when long).

Default workload: GQA decode, bf16 -- 64 sequences, context lengths uniform in
[64, 2048], 32 query / 8 KV heads, head_dim 128, block 16, a pool of the
needed blocks + 10% handed out in shuffled order.  Data are synthetic N(0,1).

Prints ONE JSON line (rank 0).  `value` is the unique KV bytes the step's
attention reads divided by the device time of the step, with every input
resident in HBM; `e2e` is the same metric through the public Python API with
host buffers (allocator on the host, H2D of the step's inputs, D2H of the
output, all inside the timed region).  `--impl reference` times the fp64 CPU
oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_cache_279_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-decode attention KV GB/s (% of GB300 HBM peak); decode tokens/s"
WORKLOADS = {
    "gqa": wl.GQA_BF16,
    "tiny": wl.TINY_FP32,
    "long": wl.LONG_BF16,
    "mixed": wl.MIXED_BF16,
    "beam": wl.BEAM_BF16,
    "beam1032": wl.BEAM_BF16,
}
# Multi-token attention (several new tokens per sequence, causal): verification
# of 4 drafted tokens plus one on the GQA shapes (bandwidth-bound, like decode),
# and a 512-token prefill chunk at the end of 4096-token contexts (a dense
# contraction).  (query tokens per sequence, fixed context or None = GQA lengths)
MULTI_TOKEN = {"verify": (5, None, 64), "prefill": (512, 4096, 8)}

# batches rotated so that no step re-reads the previous step's pool from L2
ROTATE = {"gqa": 4, "tiny": 1, "long": 1, "mixed": 4, "beam": 4, "beam1032": 4}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(MULTI_TOKEN), default="gqa")
    p.add_argument("--block-size", type=int, default=0, help="override the block size (mixed sweep)")
    p.add_argument("--partition-size", type=int, default=0)
    p.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                   help="cache element type: bf16, or E4M3 codes with per-tensor scales")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    p.add_argument("--per-workload", choices=["auto", "all", "none"], default="auto",
                   help="also time every other workload (auto: in the default GQA run)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# multi-process plumbing (one process per GPU, independent replicas)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Largest value of x over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device="cpu") -> float:
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        smax = max(r[1] for r in rows)
        loaded = [r for r in rows if r[2] > 250.0] or rows
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(1, 5)
                          if i < len(r[3]) and r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------------------
# workload construction (through the library: allocator + cache write)
# ---------------------------------------------------------------------------
def shape_for(args) -> wl.DecodeShape:
    shape = WORKLOADS[args.workload]
    if args.block_size:
        shape = wl.DecodeShape(shape.name, shape.num_seqs, shape.num_heads, shape.num_kv_heads,
                               shape.head_dim, args.block_size, shape.dtype, shape.num_layers,
                               shape.partition_size)
    return shape


# per-tensor scales of the FP8 cache: N(0, 1) data stays below 448 * scale
FP8_K_SCALE = FP8_V_SCALE = 1.0 / 64

# DRAM bytes (read + write) of one captured launch of the attention kernel and
# that launch's algorithmic bytes, from `ncu --set full` of the same command
# (rotated batch 0); the line reports traffic scaled to the average launch.
# Only valid for the kernel build the capture was taken from.
NCU_TRAFFIC = {
    ("gqa", "bf16"): (269.27e6, 263.95e6, "profiles/decode_balanced_gqa_full.md"),
    ("gqa", "fp8"): (136.92e6, 132.51e6, "profiles/decode_fp8_gqa_full.md"),
}


def kv_bytes(lens, shape, kv_elt=None) -> int:
    """Unique K and V bytes one attention pass reads (every cached token once);
    kv_elt = bytes per cached element (default: the workload's dtype)."""
    elt = kv_elt or torch.tensor([], dtype=shape.dtype).element_size()
    return int(sum(int(x) for x in lens)) * shape.num_kv_heads * shape.head_dim * 2 * elt


def algorithmic_decode_bytes(lens, shape, kv_elt=None) -> int:
    """Bytes one paged_attention_decode call must move: the K/V of every cached
    token, the query and output rows, the block-table entries and lengths."""
    elt = torch.tensor([], dtype=shape.dtype).element_size()
    S = len(lens)
    blocks = sum(-(-int(x) // shape.block_size) for x in lens)
    qo = 2 * S * shape.num_heads * shape.head_dim * elt
    return kv_bytes(lens, shape, kv_elt) + qo + 4 * blocks + 4 * S


class Batch:
    """One resident decode batch: pool, allocator, tables and step inputs."""

    kv = "bf16"

    def __init__(self, pkv, shape, lens, seed, device, partition_size, reserve_tokens=0, kv="bf16"):
        B = shape.block_size
        self.kv = kv
        self.shape = shape
        self.device = device
        self.lens = [int(x) for x in lens]
        S = len(self.lens)
        need = sum(-(-L // B) for L in self.lens)
        # +10% and room for `reserve_tokens` more tokens per sequence; at least 64 blocks
        self.num_blocks = max(64, math.ceil(1.1 * need) + S * (2 + -(-reserve_tokens // B)))
        self.alloc = pkv.BlockAllocator(self.num_blocks, B)
        # hand blocks out in a random order, as after a long run of frees
        order = wl.draw_block_ids(self.num_blocks, seed)
        for i in range(self.num_blocks):
            assert self.alloc.add_seq(-1 - i, B) == 0
        for b in order[::-1]:
            assert self.alloc.free_seq(-1 - int(b)) == 0
        g = torch.Generator(device=device)
        g.manual_seed(int(wl.sub_seed(seed, 9)))
        Hkv, D = shape.num_kv_heads, shape.head_dim
        if kv == "fp8":  # E4M3 codes; V transposed inside each block
            self.k_cache = torch.zeros((self.num_blocks, Hkv, B, D), dtype=torch.uint8, device=device)
            self.v_cache = torch.zeros((self.num_blocks, Hkv, D, B), dtype=torch.uint8, device=device)
        else:
            self.k_cache = torch.zeros((self.num_blocks, Hkv, B, D), dtype=shape.dtype, device=device)
            self.v_cache = torch.zeros_like(self.k_cache)
        # the context before this step: written through the library
        for s, L in enumerate(self.lens):
            assert self.alloc.add_seq(s, L - 1) == 0
            if L > 1:
                slots = torch.from_numpy(self.alloc.slots(s, 0, L - 1)).to(device)
                k = torch.randn((L - 1, Hkv, D), generator=g, device=device).to(shape.dtype)
                v = torch.randn((L - 1, Hkv, D), generator=g, device=device).to(shape.dtype)
                if kv == "fp8":
                    pkv.kv_cache_write_fp8(k, v, self.k_cache, self.v_cache, slots, FP8_K_SCALE, FP8_V_SCALE)
                else:
                    pkv.kv_cache_write(k, v, self.k_cache, self.v_cache, slots)
        self._finish(pkv, g, np.arange(S, dtype=np.int64), partition_size)
        elt = 1 if kv == "fp8" else None
        self.unique_bytes = kv_bytes(self.lens, shape, elt)
        self.alg_bytes = algorithmic_decode_bytes(self.lens, shape, elt)

    def _finish(self, pkv, g, seq_ids, partition_size):
        """This step's new token for every sequence: slots from the allocator
        (copy-on-write pairs executed at once), tables, queries, workspace."""
        shape, device, B = self.shape, self.device, self.shape.block_size
        Hkv, D, S = shape.num_kv_heads, shape.head_dim, len(seq_ids)
        self.seq_ids = seq_ids
        st, slots, pairs = self.alloc.append_slots(self.seq_ids)
        assert st == 0
        self.cow_copies = getattr(self, "cow_copies", 0) + len(pairs)
        if len(pairs):
            pkv.block_copy([self.k_cache], [self.v_cache], torch.from_numpy(np.ascontiguousarray(pairs)).to(device))
        self.max_blocks = max(-(-L // B) for L in self.lens) + 4
        tables, seq_lens = self.alloc.block_tables(self.seq_ids, self.max_blocks)
        self.max_seq_len = self.max_blocks * B
        self.slot_mapping = torch.from_numpy(slots).to(device)
        self.block_tables = torch.from_numpy(tables).to(device)
        self.seq_lens = torch.from_numpy(seq_lens).to(device)
        self.q = torch.randn((S, shape.num_heads, D), generator=g, device=device).to(shape.dtype)
        self.k_new = torch.randn((S, Hkv, D), generator=g, device=device).to(shape.dtype)
        self.v_new = torch.randn((S, Hkv, D), generator=g, device=device).to(shape.dtype)
        self.out = torch.empty_like(self.q)
        self.partition_size = partition_size
        ws = pkv.paged_attention_workspace_size(S, shape.num_heads, D, self.max_seq_len,
                                                partition_size)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)
        self.pkv = pkv

    @classmethod
    def beam(cls, pkv, shape, seed, device, partition_size, shared, reserve_tokens=0):
        """Beam search: prompts of `shared` tokens, each forked into a beam
        group that shares the prompt's blocks; every beam then produced its own
        0-256 tokens (copy-on-write where a shared block was partially filled),
        and this step adds one more token per beam."""
        self = cls.__new__(cls)
        B, Hkv, D = shape.block_size, shape.num_kv_heads, shape.head_dim
        P_, W = wl.BEAM_PROMPTS, wl.BEAM_WIDTH
        div = wl.draw_divergent_lengths(P_ * W, seed)
        self.shape, self.device = shape, device
        self.lens = [shared + int(d) + 1 for d in div]  # after this step's token
        # room for `reserve_tokens` appended tokens per beam (the e2e loop)
        self.num_blocks = (P_ * (-(-shared // B) + 1) + sum(-(-int(d) // B) + 2 for d in div) + 64
                           + P_ * W * -(-reserve_tokens // B))
        self.alloc = pkv.BlockAllocator(self.num_blocks, B)
        order = wl.draw_block_ids(self.num_blocks, seed)
        for i in range(self.num_blocks):
            assert self.alloc.add_seq(-1 - i, B) == 0
        for b in order[::-1]:
            assert self.alloc.free_seq(-1 - int(b)) == 0
        g = torch.Generator(device=device)
        g.manual_seed(int(wl.sub_seed(seed, 9)))
        self.k_cache = torch.zeros((self.num_blocks, Hkv, B, D), dtype=shape.dtype, device=device)
        self.v_cache = torch.zeros_like(self.k_cache)
        for p in range(P_):
            assert self.alloc.add_seq(p * W, shared) == 0
            slots = torch.from_numpy(self.alloc.slots(p * W, 0, shared)).to(device)
            k = torch.randn((shared, Hkv, D), generator=g, device=device).to(shape.dtype)
            pkv.kv_cache_write(k, torch.randn_like(k), self.k_cache, self.v_cache, slots)
            for c in range(1, W):
                assert self.alloc.fork(p * W, p * W + c) == 0
        self.cow_copies = 0
        for t in range(int(div.max())):
            beams = [b for b in range(P_ * W) if div[b] > t]
            st, slots, pairs = self.alloc.append_slots(beams)
            assert st == 0
            self.cow_copies += len(pairs)
            if len(pairs):
                pkv.block_copy([self.k_cache], [self.v_cache],
                               torch.from_numpy(np.ascontiguousarray(pairs)).to(device))
            k = torch.randn((len(beams), Hkv, D), generator=g, device=device).to(shape.dtype)
            pkv.kv_cache_write(k, torch.randn_like(k), self.k_cache, self.v_cache,
                               torch.from_numpy(slots).to(device))
        self._finish(pkv, g, np.arange(P_ * W, dtype=np.int64), partition_size)
        # beams of a prompt share its blocks: one group per prompt
        offs, pre = self.alloc.prefix_groups(self.seq_ids)
        self.group_offsets = torch.from_numpy(offs).to(device)
        self.prefix_lens = torch.from_numpy(pre).to(device)
        ws = pkv.paged_attention_grouped_workspace_size(len(self.lens), shape.num_heads, D, self.max_seq_len)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)
        # bytes a step must read: each prompt once, each beam's own tokens once
        elt = torch.tensor([], dtype=shape.dtype).element_size()
        own = sum(int(d) + 1 for d in div)
        self.unique_bytes = (P_ * shared + own) * Hkv * D * 2 * elt
        blocks = P_ * -(-shared // B) + sum(-(-(int(d) + 1 + shared % B) // B) for d in div)
        self.alg_bytes = (self.unique_bytes + 2 * len(self.lens) * shape.num_heads * D * elt
                          + 4 * blocks + 4 * len(self.lens))
        return self

    group_offsets = None

    def write(self):
        if self.kv == "fp8":
            self.pkv.kv_cache_write_fp8(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slot_mapping,
                                        FP8_K_SCALE, FP8_V_SCALE)
            return
        self.pkv.kv_cache_write(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slot_mapping)

    def decode(self):
        if self.kv == "fp8":
            self.pkv.paged_attention_decode_fp8(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                                self.seq_lens, self.shape.scale, FP8_K_SCALE, FP8_V_SCALE,
                                                self.max_seq_len, self.workspace)
            return
        if self.group_offsets is not None:
            self.pkv.paged_attention_decode_grouped(self.out, self.q, self.k_cache, self.v_cache,
                                                    self.block_tables, self.seq_lens, self.group_offsets,
                                                    self.prefix_lens, self.shape.scale, self.max_seq_len,
                                                    workspace=self.workspace)
            return
        self.pkv.paged_attention_decode(self.out, self.q, self.k_cache, self.v_cache,
                                        self.block_tables, self.seq_lens, self.shape.scale,
                                        self.max_seq_len, self.partition_size, self.workspace)

    def step(self):
        """Store every sequence's new token and attend: one library call
        (grouped by shared prefix for beam search); with an FP8 cache the
        quantising write, then the FP8 decode."""
        if self.kv == "fp8":
            self.pkv.paged_attention_decode_append_fp8(self.out, self.q, self.k_new, self.v_new, self.k_cache,
                                                       self.v_cache, self.block_tables, self.seq_lens,
                                                       self.shape.scale, FP8_K_SCALE, FP8_V_SCALE,
                                                       self.max_seq_len, self.workspace)
            return
        if self.group_offsets is not None:
            self.pkv.paged_attention_decode_grouped(self.out, self.q, self.k_cache, self.v_cache,
                                                    self.block_tables, self.seq_lens, self.group_offsets,
                                                    self.prefix_lens, self.shape.scale, self.max_seq_len,
                                                    k_new=self.k_new, v_new=self.v_new,
                                                    workspace=self.workspace)
            return
        self.pkv.paged_attention_decode_append(self.out, self.q, self.k_new, self.v_new, self.k_cache,
                                               self.v_cache, self.block_tables, self.seq_lens,
                                               self.shape.scale, self.max_seq_len, self.partition_size,
                                               self.workspace)

    def launches_per_step(self) -> int:
        """Kernels one step launches.  Balanced split (bf16, FP8): one -- the
        attention kernel stores the new tokens and merges split contexts itself.
        Fixed partitions: store kernel, attention kernel and the merge kernel
        when contexts are split.  Grouped beam search: the store of the new
        tokens, then one tensor-core kernel (shared prefix, each beam's own
        tokens and the merge of split contexts)."""
        S = len(self.lens)
        if self.group_offsets is not None:
            return 2  # the new tokens' store, then the tensor-core kernel (prefix, own tokens, merge)
        if self.kv == "fp8" or (self.partition_size == 0 and self.shape.dtype == torch.bfloat16):
            return 1
        ws = self.pkv.paged_attention_workspace_size(S, self.shape.num_heads, self.shape.head_dim,
                                                     self.max_seq_len, self.partition_size)
        return 2 + (1 if ws > 0 else 0)


def capture(fns, stream):
    """One CUDA graph that runs the callables in order (one per step)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for fn in fns[:4]:
            fn()  # warm caches (tensor maps, smem opt-in, symbol addresses) outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for fn in fns:
                fn()
    torch.cuda.synchronize()
    return g


def time_graph(graph, stream, repeats=1):
    """Device milliseconds of `repeats` back-to-back replays of `graph`
    (CUDA events on the launch stream, synchronised on both sides)."""
    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(repeats):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1)


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample(shape, seed, budget_s, lens, kv="bf16"):
    """Time the fp64 oracle, as it stands, on one freshly drawn batch of the
    same workload (context lengths `lens`), repeating the call until about
    `budget_s` seconds of work.  With an FP8 cache each call dequantises the
    E4M3 codes first.  Returns (GB/s, cores, description, seconds, calls)."""
    import oracle
    from oracle import fp8_e4m3
    cores = oracle.max_threads()
    q = wl.draw_query(shape, seed + 1, num_seqs=len(lens)).float().numpy()
    ks, vs = [], []
    for i, L in enumerate(lens):
        if kv == "fp8":
            shp = (L, shape.num_kv_heads, shape.head_dim)
            ks.append(wl.draw_e4m3_codes(shp, wl.sub_seed(seed + 1, 10, i)))
            vs.append(wl.draw_e4m3_codes(shp, wl.sub_seed(seed + 1, 11, i)))
        else:
            k, v = wl.draw_seq_kv(shape, seed + 1, i, L)
            ks.append(k.float().numpy())
            vs.append(v.float().numpy())
    done_s, calls = 0.0, 0
    while done_s < budget_s and calls < 1000:
        t0 = time.perf_counter()
        if kv == "fp8":
            oracle.decode_attention(q, [fp8_e4m3.dequantize(k, FP8_K_SCALE) for k in ks],
                                    [fp8_e4m3.dequantize(v, FP8_V_SCALE) for v in vs], shape.scale)
        else:
            oracle.decode_attention(q, ks, vs, shape.scale)
        done_s += time.perf_counter() - t0
        calls += 1
    gbs = calls * kv_bytes(lens, shape, 1 if kv == "fp8" else None) / done_s / 1e9
    desc = (f"fp64 oracle{' (E4M3 codes dequantised per call)' if kv == 'fp8' else ''}, {calls} call(s) "
            f"over one {len(lens)}-sequence batch of the {shape.name} workload, {cores} threads, {done_s:.1f} s")
    return gbs, cores, desc, done_s, calls


# ---------------------------------------------------------------------------
def run_reference_multi_token(args):
    """The fp64 multi-token oracle on a bounded sample of the workload: per step
    one sequence's context and its last min(Q, 16) query tokens."""
    from oracle.multi_token import multi_token_attention
    import oracle
    shape = wl.GQA_BF16
    Q, L_fixed, S = MULTI_TOKEN[args.workload]
    lens = [L_fixed] * S if L_fixed else [max(Q, int(x)) for x in wl.draw_lengths(shape, args.seed + 1).tolist()]
    qn = min(Q, 16)
    times, bytes_ = [], []
    for i in range(args.warmup + args.steps):
        s = i % S
        L = lens[s]
        k, v = wl.draw_seq_kv(shape, args.seed + 1, s, L)
        q = wl.draw_normal((qn, shape.num_heads, shape.head_dim), torch.bfloat16, wl.sub_seed(args.seed, 30, s))
        t0 = time.perf_counter()
        # the sample's queries are the context's last qn positions
        multi_token_attention([q.float().numpy()], [k.float().numpy()], [v.float().numpy()], shape.scale)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            bytes_.append(L * shape.num_kv_heads * shape.head_dim * 2 * 2)
    value = sum(bytes_) / sum(times) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload} (oracle sample: one sequence, last {qn} query tokens per step)"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"one sequence and its last {qn} query tokens per step, numpy fp64"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload in MULTI_TOKEN:
        return run_reference_multi_token(args)
    shape = shape_for(args)
    lens = context_lengths(args, shape, args.seed + 1)
    per_step = max(1, len(lens) // 4)  # a bounded sample per step
    import oracle
    cores = oracle.max_threads()
    times, bytes_ = [], []
    q = wl.draw_query(shape, args.seed + 1, num_seqs=len(lens)).float().numpy()
    fp8 = args.kv == "fp8"
    if fp8:
        from oracle import fp8_e4m3
        shp = lambda L: (L, shape.num_kv_heads, shape.head_dim)  # noqa: E731
        kv = [(wl.draw_e4m3_codes(shp(L), wl.sub_seed(args.seed + 1, 10, s)),
               wl.draw_e4m3_codes(shp(L), wl.sub_seed(args.seed + 1, 11, s))) for s, L in enumerate(lens)]
    else:
        kv = [tuple(t.float().numpy() for t in wl.draw_seq_kv(shape, args.seed + 1, s, L))
              for s, L in enumerate(lens)]
    for i in range(args.warmup + args.steps):
        idx = [((i * per_step) + j) % len(lens) for j in range(per_step)]
        t0 = time.perf_counter()
        if fp8:  # the oracle dequantises the codes, then attends
            oracle.decode_attention(q[idx], [fp8_e4m3.dequantize(kv[s][0], FP8_K_SCALE) for s in idx],
                                    [fp8_e4m3.dequantize(kv[s][1], FP8_V_SCALE) for s in idx], shape.scale)
        else:
            oracle.decode_attention(q[idx], [kv[s][0] for s in idx], [kv[s][1] for s in idx], shape.scale)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            bytes_.append(kv_bytes([lens[s] for s in idx], shape, 1 if fp8 else None))
    total_s = sum(times)
    value = sum(bytes_) / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_s / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(shape, args, len(lens)),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} of {len(lens)} sequences per step, fp64 CPU oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(shape, args, S):
    kv = (f", E4M3 cache (k/v scale {FP8_K_SCALE:g})" if getattr(args, "kv", "bf16") == "fp8" else "")
    return {"workload": f"{shape.name}: {S} seqs, {shape.num_heads}q/{shape.num_kv_heads}kv heads, "
                        f"head_dim {shape.head_dim}, block {shape.block_size}{kv}",
            "num_seqs": S, "num_heads": shape.num_heads, "num_kv_heads": shape.num_kv_heads,
            "head_dim": shape.head_dim, "block_size": shape.block_size,
            "partition_size": args.partition_size or "auto",
            "l2": f"inputs larger than L2: {ROTATE.get(args.workload, 1)} resident batches rotated"}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def timed_replays(graph, stream, min_ms):
    """Replays of `graph` back to back until at least `min_ms` of device time:
    (total device ms, replays).  One replay first sizes the count."""
    one = time_graph(graph, stream, 1)
    reps = max(1, math.ceil(min_ms / max(one, 1e-3)))
    return time_graph(graph, stream, reps), reps


def measure_decode(pkv, shape, args, device, stream, seed, world, steps, warmup, sustained_ms):
    """Device timing of one decode workload: exactly `steps` steps in one CUDA
    graph (the contract's timed region), the same graph replayed for at least
    `sustained_ms`, and the decode call alone (the roofline's kernel) replayed
    as long.  Batches rotate so that no step re-reads the previous step's pool."""
    nrot = ROTATE.get(args.workload, 1)
    batches = [make_batch(pkv, shape, args, seed + r, device) for r in range(nrot)]
    elt = 1 if args.kv == "fp8" else None
    torch.cuda.synchronize()
    warm_graph = capture([batches[i % nrot].step for i in range(warmup)], stream)
    step_graph = capture([batches[i % nrot].step for i in range(steps)], stream)
    decode_graph = capture([batches[i % nrot].decode for i in range(steps)], stream)
    if pkv.read_device_errors() != 0:
        raise RuntimeError(f"{args.workload}: device error bits set while capturing")
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        time_graph(warm_graph, stream)                    # W untimed warm-up steps
        step_ms = time_graph(step_graph, stream)          # exactly `steps` steps
        sus_ms, sus_reps = timed_replays(step_graph, stream, sustained_ms)
        dec_ms, dec_reps = timed_replays(decode_graph, stream, sustained_ms / 2)
    torch.cuda.synchronize()
    barrier(world)
    if pkv.read_device_errors() != 0:
        raise RuntimeError(f"{args.workload}: device error bits set while timing")
    uniq = [b.unique_bytes for b in batches]
    logical = [kv_bytes(b.lens, shape, elt) for b in batches]
    alg = [b.alg_bytes for b in batches]
    step_bytes = sum(uniq[i % nrot] for i in range(steps))
    total_s = max_over_ranks(step_ms / 1e3, world, device)
    sus_s = max_over_ranks(sus_ms / 1e3, world, device)
    total_bytes = sum_over_ranks(step_bytes, world, device)
    peaks = load_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    dec_call_ms = dec_ms / (steps * dec_reps)
    dec_alg = sum(alg[i % nrot] for i in range(steps)) / steps
    achieved = dec_alg / (dec_call_ms / 1e3) / 1e9
    seqs = sum(len(b.lens) for b in batches) / nrot
    res = {
        "value": total_bytes / total_s / 1e9,
        "ms_per_step": 1e3 * total_s / steps,
        "sustained": {"value": round(total_bytes * sus_reps / sus_s / 1e9, 2), "unit": "GB/s",
                      "steps_timed": steps * sus_reps, "timed_ms": round(sus_ms, 2),
                      "ms_per_step": round(sus_ms / (steps * sus_reps), 5)},
        "decode_tokens_per_s": world * seqs / (shape.num_layers * total_s / steps),
        "logical_kv_gbs": sum(logical[i % nrot] for i in range(steps)) / total_s / 1e9 * world,
        "peak": peak, "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "algorithmic_bytes": round(dec_alg),
                     "decode_us": round(dec_call_ms * 1e3, 2), "calls_timed": steps * dec_reps,
                     "timed_ms": round(dec_ms, 2),
                     "peak_source": "measured (hbm_gbs)" if "hbm_gbs" in peaks else "fallback 6800 GB/s"},
        "clocks": clocks.summary(),
        "batches": batches,
    }
    return res


def workload_args(args, workload, kv="bf16", block_size=0):
    a = argparse.Namespace(**vars(args))
    a.workload, a.kv, a.block_size, a.partition_size = workload, kv, block_size, 0
    return a


# Workloads reported beside the headline in the default run (name -> (workload,
# kv, block size)); each is timed for at least SUSTAINED_MS of device time.
EXTRA_WORKLOADS = {
    "long": ("long", "bf16", 0),
    "beam": ("beam", "bf16", 0),
    "beam1032": ("beam1032", "bf16", 0),
    "mixed_b16": ("mixed", "bf16", 16),
    "mixed_b8": ("mixed", "bf16", 8),
    "mixed_b32": ("mixed", "bf16", 32),
    "gqa_fp8": ("gqa", "fp8", 0),
    "long_fp8": ("long", "fp8", 0),
    "mixed_fp8": ("mixed", "fp8", 0),
    "tiny": ("tiny", "bf16", 0),
    "verify": ("verify", "bf16", 0),
    "prefill": ("prefill", "bf16", 0),
}
SUSTAINED_MS = 200.0


def waste_of(batch):
    used, alloc = batch.alloc.waste()
    return 1.0 - used / alloc if alloc else 0.0


def extra_workload(pkv, name, args, device, stream, seed, world):
    """Compact line of one extra workload (device timing only)."""
    wk, kv, bs = EXTRA_WORKLOADS[name]
    a = workload_args(args, wk, kv, bs)
    steps, warmup = args.steps, max(3, args.warmup)
    if wk in MULTI_TOKEN:
        r = measure_multi_token(pkv, a, device, stream, seed, world, steps, warmup, SUSTAINED_MS)
        return {k: r[k] for k in ("value", "unit", "ms_per_step", "query_tokens_per_s", "roofline", "clocks",
                                  "config", "sustained")}
    shape = shape_for(a)
    r = measure_decode(pkv, shape, a, device, stream, seed, world, steps, warmup, SUSTAINED_MS)
    b0 = r["batches"][0]
    line = {"value": round(r["sustained"]["value"], 2), "unit": "GB/s",
            "pct_of_hbm_peak": round(100 * r["sustained"]["value"] / r["peak"], 2),
            "ms_per_step": r["sustained"]["ms_per_step"], "steps_timed": r["sustained"]["steps_timed"],
            "timed_ms": r["sustained"]["timed_ms"], "k_steps_value": round(r["value"], 2),
            "decode_tokens_per_s": round(r["decode_tokens_per_s"], 1),
            "roofline": r["roofline"], "clocks": r["clocks"],
            "config": config_of(shape, a, len(b0.lens))["workload"],
            "dtype": "e4m3" if kv == "fp8" else ("f32" if shape.dtype == torch.float32 else "bf16")}
    if wk.startswith("beam"):
        line["logical_kv_gbs"] = round(r["logical_kv_gbs"] * r["sustained"]["value"] / max(r["value"], 1e-9), 2)
        line["cow_copies_per_batch"] = getattr(b0, "cow_copies", 0)
    if wk == "mixed":
        line["allocator_waste"] = round(waste_of(b0), 5)
    del r
    return line


def run_ours(args):
    rank, world, local = dist_env()
    import paged_kv_cache_279_gb300 as pkv
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    shape = shape_for(args)
    seed = args.seed + 1000 * rank
    stream = torch.cuda.Stream(device)
    steps, warmup = args.steps, max(3, args.warmup)
    r = measure_decode(pkv, shape, args, device, stream, seed, world, steps, warmup, SUSTAINED_MS)
    batches = r.pop("batches")
    nrot = len(batches)
    roofline = r["roofline"]
    traffic, traffic_src = None, None
    cap = NCU_TRAFFIC.get((args.workload, args.kv))
    if cap is not None and not args.block_size and not args.partition_size:
        traffic = round(cap[0] / cap[1] * roofline["algorithmic_bytes"])
        traffic_src = f"{cap[2]}: {cap[0] / 1e6:.2f} MB for {cap[1] / 1e6:.2f} MB algorithmic, scaled to this launch"
    roofline.update({"traffic": traffic, "traffic_unit": "bytes per launch", "traffic_source": traffic_src,
                     "kernel": KERNEL_NAMES.get((args.workload.startswith("beam"), args.kv),
                                                "paged_attention_decode")})
    launches = batches[0].launches_per_step() * steps
    del batches

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(pkv, shape, args, device, stream, seed, world)
    per_workload = None
    if args.per_workload == "all" or (args.per_workload == "auto" and args.workload == "gqa" and
                                      args.kv == "bf16" and not args.block_size and not args.partition_size):
        per_workload = {}
        for name in EXTRA_WORKLOADS:
            try:
                per_workload[name] = extra_workload(pkv, name, args, device, stream, seed, world)
            except Exception as exc:  # reported, never hidden
                per_workload[name] = {"error": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, cores, desc, secs, _ = oracle_sample(shape, seed, args.cpu_budget,
                                                  context_lengths(args, shape, seed + 1), kv=args.kv)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": desc}
    if rank == 0:
        cfg = config_of(shape, args, shape.num_seqs if not args.workload.startswith("beam")
                        else wl.BEAM_PROMPTS * wl.BEAM_WIDTH)
        cfg["l2"] = f"inputs larger than L2: {nrot} resident batches rotated"
        line = {
            "metric": METRIC, "value": round(r["value"], 2), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": round(r["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3" if args.kv == "fp8" else "bf16") if shape.dtype == torch.bfloat16 else "f32",
            "data": "synthetic", "config": cfg,
            "decode_tokens_per_s": round(r["decode_tokens_per_s"], 1),
            "logical_kv_gbs": round(r["logical_kv_gbs"], 2),
            "pct_of_hbm_peak": round(100 * r["value"] / r["peak"], 2),
            "sustained": r["sustained"],
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches,
            "clocks": r["clocks"],
            "per_workload": per_workload,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


KERNEL_NAMES = {
    (False, "bf16"): "paged_attention_decode (one kernel: stores, attention and in-kernel merge)",
    (False, "fp8"): "paged_attention_decode_fp8 (one kernel: stores, attention and in-kernel merge)",
    (True, "bf16"): "paged_attention_decode_grouped",
}


def make_batch(pkv, shape, args, seed, device, reserve_tokens=0):
    if args.kv == "fp8":
        if args.workload not in ("gqa", "long", "mixed") or args.partition_size:
            raise SystemExit("--kv fp8 runs the balanced split on the gqa, long and mixed workloads")
        return Batch(pkv, shape, wl.draw_lengths(shape, seed).tolist(), seed, device, 0, reserve_tokens, kv="fp8")
    if args.workload.startswith("beam"):
        shared = wl.BEAM_SHARED_PARTIAL if args.workload == "beam1032" else wl.BEAM_SHARED
        return Batch.beam(pkv, shape, seed, device, args.partition_size, shared, reserve_tokens)
    return Batch(pkv, shape, wl.draw_lengths(shape, seed).tolist(), seed, device, args.partition_size,
                 reserve_tokens)


def context_lengths(args, shape, seed):
    """Context lengths of one batch of the workload (for the CPU oracle)."""
    if args.workload.startswith("beam"):
        shared = wl.BEAM_SHARED_PARTIAL if args.workload == "beam1032" else wl.BEAM_SHARED
        div = wl.draw_divergent_lengths(wl.BEAM_PROMPTS * wl.BEAM_WIDTH, seed)
        return [shared + int(d) + 1 for d in div]
    return wl.draw_lengths(shape, seed).tolist()


def run_e2e(pkv, shape, args, device, stream, seed, world):
    """The step through the C ABI with host buffers, as a serving loop runs it:
    the host allocator appends a token for every sequence, the host copy of
    the block tables changes only where a sequence took a new block, one H2D
    copy from a pinned buffer carries the step's queries, new K/V, lengths and
    tables (and the groups of a beam batch), the library call stores the new
    tokens and attends, and one D2H copy brings the output back; the host
    waits for it before the next step.  The copy in, the call and the copy out
    are replayed as one CUDA graph.  The allocator's work for the next step
    (which needs only that a token is appended, not which) runs on the host
    while the device runs the current step, into the other of two pinned
    buffers; it is inside the timed region."""
    from paged_kv_cache_279_gb300 import _lib
    lib = _lib.load()
    steps = args.steps
    n_tok = steps + max(1, args.warmup) + 3  # tokens the loop appends per sequence
    b = make_batch(pkv, shape, args, seed + 77, device, reserve_tokens=n_tok + 1)
    S, Hq, Hkv, D, B = len(b.lens), shape.num_heads, shape.num_kv_heads, shape.head_dim, shape.block_size
    cap = b.max_blocks + n_tok // B + 2
    max_seq_len = cap * B
    grouped = b.group_offsets is not None
    fp8 = args.kv == "fp8"
    elt = torch.tensor([], dtype=shape.dtype).element_size()
    # two pinned buffers (steps alternate between them), one device buffer:
    # q | k_new | v_new | lens | tables | groups
    parts = [("q", S * Hq * D * elt), ("k", S * Hkv * D * elt), ("v", S * Hkv * D * elt), ("lens", 4 * S),
             ("tab", 4 * S * cap)]
    if grouped:
        offs, pre = b.alloc.prefix_groups(b.seq_ids)
        parts += [("offs", 4 * len(offs)), ("pre", 4 * len(pre))]
    off, pos = {}, 0
    for name, n in parts:
        off[name] = pos
        pos += (n + 255) // 256 * 256
    h_packs = [torch.zeros(pos, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_pack = torch.zeros(pos, dtype=torch.uint8, device=device)

    def hview(pk, name, dtype, shp):
        n = int(np.prod(shp)) * torch.tensor([], dtype=dtype).element_size()
        return h_packs[pk][off[name]:off[name] + n].view(dtype).view(*shp)
    # the allocator's tables and lengths (host memory the device never reads)
    m_tab, m_lens = b.alloc.block_tables(b.seq_ids, cap)
    m_tab = np.ascontiguousarray(m_tab, dtype=np.int32)
    m_lens = np.ascontiguousarray(m_lens, dtype=np.int32)
    p_lens, p_tab = [], []
    for pk in range(2):
        hview(pk, "q", shape.dtype, (S, Hq, D)).copy_(b.q.cpu())
        hview(pk, "k", shape.dtype, (S, Hkv, D)).copy_(b.k_new.cpu())
        hview(pk, "v", shape.dtype, (S, Hkv, D)).copy_(b.v_new.cpu())
        p_lens.append(hview(pk, "lens", torch.int32, (S,)).numpy())
        p_tab.append(hview(pk, "tab", torch.int32, (S, cap)).numpy())
        p_tab[pk][:] = m_tab
        p_lens[pk][:] = m_lens
        if grouped:
            hview(pk, "offs", torch.int32, (len(offs),)).numpy()[:] = offs
            hview(pk, "pre", torch.int32, (len(pre),)).numpy()[:] = pre
    dptr = d_pack.data_ptr()
    out = torch.empty((S, Hq, D), dtype=shape.dtype, device=device)
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    ws_bytes = (pkv.paged_attention_grouped_workspace_size(S, Hq, D, max_seq_len) if grouped else
                pkv.paged_attention_workspace_size(S, Hq, D, max_seq_len, 0))
    ws = torch.zeros(max(256, ws_bytes), dtype=torch.uint8, device=device)
    st_ptr = ctypes.c_void_p(stream.cuda_stream)
    kc, vc = b.k_cache.data_ptr(), b.v_cache.data_ptr()
    NB = b.num_blocks
    seq_ids = np.ascontiguousarray(b.seq_ids, dtype=np.int64)

    def call():
        if fp8:
            return lib.paged_attention_decode_append_fp8(
                out.data_ptr(), dptr + off["q"], dptr + off["k"], dptr + off["v"], kc, vc, dptr + off["tab"],
                dptr + off["lens"], S, Hq, Hkv, D, B, cap, NB, max_seq_len, shape.scale, FP8_K_SCALE,
                FP8_V_SCALE, ws.data_ptr(), ws.numel(), st_ptr)
        if grouped:
            return lib.paged_attention_decode_grouped(
                out.data_ptr(), dptr + off["q"], dptr + off["k"], dptr + off["v"], kc, vc, dptr + off["tab"],
                dptr + off["lens"], dptr + off["offs"], dptr + off["pre"], len(pre), S, Hq, Hkv, D, B, cap, NB,
                max_seq_len, shape.scale, ws.data_ptr(), ws.numel(), pkv.PKV_BF16, st_ptr)
        return lib.paged_attention_decode_append(
            out.data_ptr(), dptr + off["q"], dptr + off["k"], dptr + off["v"], kc, vc, dptr + off["tab"],
            dptr + off["lens"], S, Hq, Hkv, D, B, cap, NB, max_seq_len, shape.scale, 0, ws.data_ptr(),
            ws.numel(), pkv.PKV_BF16 if shape.dtype == torch.bfloat16 else pkv.PKV_F32, st_ptr)

    h2d = pos
    d2h = h_out.numel() * h_out.element_size()
    ms, byts = [], []
    base_unique, base_lens = b.unique_bytes, list(b.lens)

    def prepare(pk):
        # the next step's bookkeeping: the allocator appends one token per
        # sequence (tables and lengths updated in place, only entries that
        # changed), then pinned buffer pk, two steps behind, takes the new
        # lengths and the table rows whose block count changed
        st, _, pairs = b.alloc.append_step(seq_ids, m_tab, m_lens)
        if st != 0 or len(pairs):
            raise RuntimeError("allocator could not serve the step")
        rows = np.nonzero((p_lens[pk] + B - 1) // B != (m_lens + B - 1) // B)[0]
        if rows.size:
            p_tab[pk][rows] = m_tab[rows]
        p_lens[pk][:] = m_lens

    def device_step(pk):
        d_pack.copy_(h_packs[pk], non_blocking=True)
        rc = call()
        if rc != 0:
            raise RuntimeError(f"library call failed with status {rc}")
        h_out.copy_(out, non_blocking=True)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_eager = max(1, args.warmup)
    with torch.cuda.stream(stream):
        for _ in range(n_eager):  # eager steps: the library's one-time host setup
            prepare(0)
            device_step(0)
            stream.synchronize()  # the next prepare rewrites the buffer this copy reads
        p_tab[1][:] = m_tab
        p_lens[1][:] = m_lens
        bits = pkv.read_device_errors()
        if bits != 0:
            raise RuntimeError(f"e2e: device error bits {bits:#x} set by the eager steps")
        # per pinned buffer, the step's copy in, library call and copy out as
        # one graph; every replay copies the buffer's current contents
        graphs = []
        for pk in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                device_step(pk)
            graphs.append(g)
        cur = 0
        prepare(cur)
        for i in range(steps + 2):
            ev0.record(stream)
            graphs[cur].replay()
            used = p_lens[cur].tolist()  # the lengths this step attends
            # while the device runs this step, the host prepares the next one in
            # the other buffer (the one the previous step read, already done);
            # the step's result is read before the next step starts
            prepare(1 - cur)
            ev1.record(stream)
            ev1.synchronize()  # the host reads the step's result
            if i >= 2:  # the first replay of each graph uploads it
                ms.append(ev0.elapsed_time(ev1))
                # unique bytes: what the batch started with plus the tokens added since
                byts.append(base_unique + kv_bytes(used, shape, 1 if fp8 else None) -
                            kv_bytes(base_lens, shape, 1 if fp8 else None))
            cur = 1 - cur
    bits = pkv.read_device_errors()
    if bits != 0:
        raise RuntimeError(f"e2e: device error bits {bits:#x} set")
    # the allocator's tables after the loop equal the incrementally kept ones,
    # and the last buffer prepared holds them too
    tab, ln = b.alloc.block_tables(b.seq_ids, cap)
    if not (np.array_equal(tab, m_tab) and np.array_equal(ln, m_lens) and
            np.array_equal(p_tab[cur], m_tab) and np.array_equal(p_lens[cur], m_lens)):
        raise RuntimeError("e2e: incremental block tables diverged from the allocator")
    local_s = sum(ms) / 1e3
    total_s = max_over_ranks(local_s, world, device)
    total_b = sum_over_ranks(sum(byts), world, device)
    return {"value": round(total_b / total_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * total_s / steps, 4),
            "copies_per_step": {"h2d": 1, "d2h": 1}, "graph": True}


def multi_token_batch(pkv, args, seed, device):
    """One resident batch of a multi-token workload: pool written through the
    library, the query rows of every sequence's last Q positions."""
    shape = wl.GQA_BF16
    Q, L_fixed, S = MULTI_TOKEN[args.workload]
    B, Hkv, Hq, D = shape.block_size, shape.num_kv_heads, shape.num_heads, shape.head_dim
    lens = [L_fixed] * S if L_fixed else [max(Q, int(x)) for x in wl.draw_lengths(shape, seed).tolist()]
    need = sum(-(-L // B) for L in lens)
    NB = max(64, math.ceil(1.1 * need))
    alloc = pkv.BlockAllocator(NB, B)
    order = wl.draw_block_ids(NB, seed)
    for i in range(NB):
        assert alloc.add_seq(-1 - i, B) == 0
    for b in order[::-1]:
        assert alloc.free_seq(-1 - int(b)) == 0
    g = torch.Generator(device=device)
    g.manual_seed(int(wl.sub_seed(seed, 9)))
    kc = torch.zeros((NB, Hkv, B, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    for s, L in enumerate(lens):
        assert alloc.add_seq(s, L) == 0
        slots = torch.from_numpy(alloc.slots(s, 0, L)).to(device)
        k = torch.randn((L, Hkv, D), generator=g, device=device).to(torch.bfloat16)
        pkv.kv_cache_write(k, torch.randn_like(k), kc, vc, slots)
    maxb = max(-(-L // B) for L in lens)
    tables, seq_lens = alloc.block_tables(np.arange(S), maxb)
    T = Q * S
    b = dict(lens=lens, Q=Q, kc=kc, vc=vc, tables=torch.from_numpy(tables).to(device),
             seq_lens=torch.from_numpy(seq_lens).to(device),
             starts=torch.arange(0, T + 1, Q, dtype=torch.int32, device=device),
             q=torch.randn((T, Hq, D), generator=g, device=device).to(torch.bfloat16),
             max_seq_len=maxb * B)
    b["out"] = torch.empty_like(b["q"])
    ws = pkv.paged_attention_multi_token_workspace_size(T, Hq, D, b["max_seq_len"])
    b["ws"] = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)
    b["kv_bytes"] = sum(lens) * Hkv * D * 2 * 2
    # useful flops: per query at position p, per query head: QK^T and PV over p + 1 tokens
    b["flops"] = sum(4 * D * Hq * (L - Q + i + 1) for L in lens for i in range(Q))
    b["alg_bytes"] = b["kv_bytes"] + 2 * T * Hq * D * 2 + 4 * need + 4 * S + 4 * (S + 1)
    return b


def measure_multi_token(pkv, args, device, stream, seed, world, steps, warmup, sustained_ms):
    """Multi-token attention calls (chunked prefill / verification), timed like
    the decode step: exactly `steps` calls in one CUDA graph over rotated
    resident batches, then the same graph replayed for `sustained_ms`."""
    shape = wl.GQA_BF16
    nrot = 4
    batches = [multi_token_batch(pkv, args, seed + r, device) for r in range(nrot)]

    def call(b):
        return lambda: pkv.paged_attention_multi_token(b["out"], b["q"], b["kc"], b["vc"], b["tables"], b["seq_lens"],
                                                       b["starts"], shape.scale, b["Q"], b["max_seq_len"], b["ws"])
    warm = capture([call(batches[i % nrot]) for i in range(warmup)], stream)
    timed = capture([call(batches[i % nrot]) for i in range(steps)], stream)
    if pkv.read_device_errors() != 0:
        raise RuntimeError(f"{args.workload}: device error bits set while capturing")
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        time_graph(warm, stream)
        total_ms = time_graph(timed, stream)
        sus_ms, sus_reps = timed_replays(timed, stream, sustained_ms)
    torch.cuda.synchronize()
    barrier(world)
    total_s = max_over_ranks(total_ms / 1e3, world, device)
    sus_s = max_over_ranks(sus_ms / 1e3, world, device)
    kvb = sum_over_ranks(sum(batches[i % nrot]["kv_bytes"] for i in range(steps)), world, device)
    flops = sum(batches[i % nrot]["flops"] for i in range(steps)) * world
    alg = sum(batches[i % nrot]["alg_bytes"] for i in range(steps)) / steps
    ms = 1e3 * sus_s / (steps * sus_reps)
    peaks = load_peaks()
    Q, L_fixed, S = MULTI_TOKEN[args.workload]
    if args.workload == "prefill":
        achieved = flops * sus_reps / sus_s / 1e12
        peak = float(peaks.get("bf16_tflops", 1900.0))
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4), "traffic": None,
                    "kernel": "paged_attention_multi_token",
                    "peak_source": "measured bf16 GEMM burst" if "bf16_tflops" in peaks else "fallback",
                    "useful_flops_per_call": round(flops / steps / world), "call_us": round(ms * 1e3, 2)}
    else:
        achieved = alg / (ms / 1e3) / 1e9
        peak = float(peaks.get("hbm_gbs", 6800.0))
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": None,
                    "kernel": "paged_attention_multi_token", "algorithmic_bytes": round(alg),
                    "peak_source": "measured" if "hbm_gbs" in peaks else "fallback", "call_us": round(ms * 1e3, 2)}
    launches = steps * MT_LAUNCHES_PER_CALL
    return {"value": round(kvb / total_s / 1e9, 2), "unit": "GB/s", "ms_per_step": round(1e3 * total_s / steps, 5),
            "sustained": {"value": round(kvb * sus_reps / sus_s / 1e9, 2), "unit": "GB/s",
                          "steps_timed": steps * sus_reps, "timed_ms": round(sus_ms, 2), "ms_per_step": round(ms, 5)},
            "query_tokens_per_s": round(world * S * Q / (ms / 1e3), 1), "roofline": roofline,
            "clocks": clocks.summary(), "gpu_launches": launches,
            "config": (f"{args.workload}: {S} seqs x {Q} query tokens, "
                       f"{'context ' + str(L_fixed) if L_fixed else 'GQA context lengths U[64, 2048]'}, "
                       f"32q/8kv heads, head_dim 128, block 16"),
            "l2": f"inputs larger than L2: {nrot} resident batches rotated"}


# kernels one multi-token call launches (the attention kernel merges split
# contexts itself)
MT_LAUNCHES_PER_CALL = 1


def run_multi_token_bench(args):
    rank, world, local = dist_env()
    import paged_kv_cache_279_gb300 as pkv
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    stream = torch.cuda.Stream(device)
    steps, warmup = args.steps, max(3, args.warmup)
    r = measure_multi_token(pkv, args, device, stream, args.seed + 1000 * rank, world, steps, warmup,
                            SUSTAINED_MS)
    if rank == 0:
        line = {
            "metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": r["config"], "l2": r["l2"]},
            "query_tokens_per_s": r["query_tokens_per_s"], "sustained": r["sustained"],
            "roofline": r["roofline"], "cpu_baseline": None, "e2e": None,
            "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in MULTI_TOKEN:
        return run_multi_token_bench(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
