"""Seeded synthetic workloads for paged relative-bias attention.

This module only draws random inputs -- q, k, v, rel, sequence lengths and
paged block tables -- with the shapes and distributions of the Inkling-family
attention layers.  It holds none of the attention arithmetic; the CUDA path
and the float64 oracle are both fed from here, and nothing else is shared.

Recipe: q, k, v ~ N(0, 1) in bf16, rel ~ N(0, 1) in fp32.  A data generator
(seed 0 by default) draws q, rel and the caches; a layout generator (seed 1)
draws the lengths and the pool permutation that the block tables are cut
from.  Unused block-table entries are -1.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch

BLOCK_SIZE = 128


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    d_qk: int
    d_v: int
    window: int          # <= 0: global layer
    rel_extent: int
    lengths: tuple       # ("uniform", lo, hi) | ("fixed", L) | ("loguniform", lo, hi)
    pool_blocks: int = 0  # 0: exactly the blocks the sequences need
    max_blocks_per_seq: int = 0  # 0: the longest sequence's block count
    query_tokens: int = 0  # > 0: multi-token decode, q [B, k, Hq, d], rel [B, k, Hq, E]
    rel_dtype: str = "f32"  # "bf16": rel drawn in fp32 and rounded to bf16
    # "fp8": caches quantised to e4m3 with one scale each, head-major blocks
    # [pool, Hkv, 128, d] (a token's head row is only 128 bytes)
    kv_dtype: str = "bf16"


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    d_qk: int
    d_v: int
    window: int
    rel_extent: int
    new_tokens: tuple    # per sequence
    ctx_lens: tuple      # cached prefix per sequence
    block_table: tuple = ()  # explicit table rows; () draws a random one
    pool_blocks: int = 0
    rel_dtype: str = "f32"  # "bf16": rel drawn in fp32 and rounded to bf16
    kv_dtype: str = "bf16"  # "fp8": the cache quantised to e4m3 (head-major), one scale each

    @property
    def batch(self) -> int:
        return len(self.new_tokens)


WORKLOADS = {
    # 1 sequence of 256 tokens, 4/1 heads, window = rel_extent = 64, the
    # sequence's two blocks in physical order [1, 0].
    "tiny_prefill": PrefillWorkload(
        "tiny_prefill", 4, 1, 128, 128, 64, 64, (256,), (0,),
        block_table=((1, 0),), pool_blocks=2),
    # Inkling-Small local layer: 32/8 heads, window 512, rel extent 512.
    "local_decode": DecodeWorkload(
        "local_decode", 16, 32, 8, 128, 128, 512, 512,
        ("uniform", 4096, 32768), pool_blocks=4096, max_blocks_per_seq=256),
    # Global layer at long context, rel extent 1024, no window.
    "global_decode_b1": DecodeWorkload(
        "global_decode_b1", 1, 32, 8, 128, 128, 0, 1024, ("fixed", 100_000)),
    "global_decode_b8": DecodeWorkload(
        "global_decode_b8", 8, 32, 8, 128, 128, 0, 1024, ("fixed", 32_768)),
    # Inkling 2 Small style chunked prefill: 48/8 heads, window 1024.
    "chunked_prefill": PrefillWorkload(
        "chunked_prefill", 48, 8, 128, 128, 1024, 1024,
        (8192,) * 4, (24576,) * 4),
    # head_dim 128 / v_head_dim 64 global decode, log-uniform lengths.
    "diffhead_decode": DecodeWorkload(
        "diffhead_decode", 32, 64, 8, 128, 64, 0, 1024,
        ("loguniform", 1024, 131072)),
    # Speculative verification on the local layer: 8 query tokens per
    # sequence (7 drafted tokens and the last accepted one).
    "verify_decode": DecodeWorkload(
        "verify_decode", 16, 32, 8, 128, 128, 512, 512,
        ("uniform", 4096, 32768), pool_blocks=4096, max_blocks_per_seq=256,
        query_tokens=8),
}


_REL_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def variant(wl, **changes):
    """A copy of a workload with some fields changed (smaller test cases)."""
    return dataclasses.replace(wl, **changes)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, gen, device, dtype):
    return torch.randn(shape, generator=gen, device=device, dtype=dtype)


def draw_lengths(spec, batch: int, gen: torch.Generator) -> list:
    kind = spec[0]
    if kind == "fixed":
        return [int(spec[1])] * batch
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        u = torch.randint(lo, hi + 1, (batch,), generator=gen, device="cpu")
        return [int(x) for x in u]
    if kind == "loguniform":
        lo, hi = spec[1], spec[2]
        u = torch.rand((batch,), generator=gen, dtype=torch.float64, device="cpu")
        vals = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        return [int(min(hi, max(lo, round(float(x))))) for x in vals]
    if kind == "list":
        return [int(x) for x in spec[1]]
    raise ValueError(f"unknown length spec {spec!r}")


def cut_block_tables(blocks_per_seq, max_blocks: int, pool: int,
                     gen: torch.Generator, per_seq_stride: int = 0):
    """Block tables cut from one random permutation of the pool.

    Sequence b takes consecutive entries of the permutation, starting at
    b * per_seq_stride if given, else right after sequence b-1.
    """
    perm = torch.randperm(pool, generator=gen, device="cpu").to(torch.int32)
    B = len(blocks_per_seq)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(blocks_per_seq):
        start = b * per_seq_stride if per_seq_stride else off
        if start + n > pool or n > max_blocks:
            raise ValueError("pool too small for the block tables")
        table[b, :n] = perm[start:start + n]
        off = start + n
    return table


def make_decode(wl: DecodeWorkload, device="cpu", seed_data: int = 0,
                seed_layout: int = 1, seq_lens=None) -> dict:
    """Inputs of one decode call; every tensor lives on ``device``."""
    lay = _gen("cpu", seed_layout)
    lens = list(seq_lens) if seq_lens is not None else draw_lengths(
        wl.lengths, wl.batch, lay)
    nblk = [(L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in lens]
    max_blocks = wl.max_blocks_per_seq or max(nblk)
    if wl.pool_blocks:
        pool = wl.pool_blocks
        stride = max_blocks if pool >= max_blocks * wl.batch else 0
    else:
        pool, stride = sum(nblk), 0
    table = cut_block_tables(nblk, max_blocks, pool, lay, stride)
    g = _gen(device, seed_data)
    B, Hq, Hkv = wl.batch, wl.num_q_heads, wl.num_kv_heads
    tok = (wl.query_tokens,) if wl.query_tokens > 0 else ()
    q = _randn((B, *tok, Hq, wl.d_qk), g, device, torch.bfloat16)
    rel = _randn((B, *tok, Hq, wl.rel_extent), g, device, torch.float32)
    rel = rel.to(_REL_DTYPES[wl.rel_dtype])
    k_cache = _randn((pool, BLOCK_SIZE, Hkv, wl.d_qk), g, device, torch.bfloat16)
    v_cache = _randn((pool, BLOCK_SIZE, Hkv, wl.d_v), g, device, torch.bfloat16)
    scales = {}
    if wl.kv_dtype == "fp8":  # head-major blocks: [pool, Hkv, 128, d]
        k_cache, scales["k_scale"] = quantize_e4m3(k_cache.transpose(1, 2).contiguous())
        v_cache, scales["v_scale"] = quantize_e4m3(v_cache.transpose(1, 2).contiguous())
    return dict(
        q=q, rel=rel, k_cache=k_cache, v_cache=v_cache,
        block_table=table.to(device),
        seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
        window=wl.window, rel_extent=wl.rel_extent, workload=wl, **scales)


def quantize_e4m3(x: torch.Tensor):
    """(e4m3 tensor, scale) with one scale for the whole tensor: the largest
    magnitude maps to 448, the largest finite e4m3 value."""
    scale = float(x.float().abs().max()) / 448.0
    return (x.float() / scale).to(torch.float8_e4m3fn), scale


def relayout_decode(case: dict, seed: int) -> dict:
    """Another decode call over the same KV pool: fresh q and rel, and the
    block table renumbered through a random permutation of the pool, so that
    the call reads other blocks.  Entries of -1 stay -1."""
    dev = case["q"].device
    pool = case["k_cache"].shape[0]
    perm = torch.randperm(pool, generator=_gen("cpu", seed), device="cpu").to(torch.int32)
    t = case["block_table"].cpu()
    table = torch.where(t >= 0, perm[t.clamp(min=0).long()], t)
    g = _gen(dev, seed)
    out = dict(case)
    out.update(q=_randn(tuple(case["q"].shape), g, dev, torch.bfloat16),
               rel=_randn(tuple(case["rel"].shape), g, dev, torch.float32),
               block_table=table.to(dev))
    return out


def make_prefill(wl: PrefillWorkload, device="cpu", seed_data: int = 0,
                 seed_layout: int = 1) -> dict:
    """Inputs of one chunked-prefill call; every tensor lives on ``device``."""
    lay = _gen("cpu", seed_layout)
    B = wl.batch
    totals = [c + n for c, n in zip(wl.ctx_lens, wl.new_tokens)]
    nblk = [(L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in totals]
    if wl.block_table:
        rows = [list(r) for r in wl.block_table]
        max_blocks = max(len(r) for r in rows)
        table = torch.full((B, max_blocks), -1, dtype=torch.int32)
        for b, r in enumerate(rows):
            table[b, :len(r)] = torch.tensor(r, dtype=torch.int32)
        pool = wl.pool_blocks or (int(table.max()) + 1)
    else:
        max_blocks = max(nblk)
        pool = wl.pool_blocks or sum(nblk)
        table = cut_block_tables(nblk, max_blocks, pool, lay)
    T = sum(wl.new_tokens)
    cu = [0]
    for n in wl.new_tokens:
        cu.append(cu[-1] + n)
    g = _gen(device, seed_data)
    Hq, Hkv = wl.num_q_heads, wl.num_kv_heads
    q = _randn((T, Hq, wl.d_qk), g, device, torch.bfloat16)
    k = _randn((T, Hkv, wl.d_qk), g, device, torch.bfloat16)
    v = _randn((T, Hkv, wl.d_v), g, device, torch.bfloat16)
    rel = _randn((T, Hq, wl.rel_extent), g, device, torch.float32)
    rel = rel.to(_REL_DTYPES[wl.rel_dtype])
    k_cache = _randn((pool, BLOCK_SIZE, Hkv, wl.d_qk), g, device, torch.bfloat16)
    v_cache = _randn((pool, BLOCK_SIZE, Hkv, wl.d_v), g, device, torch.bfloat16)
    scales = {}
    if wl.kv_dtype == "fp8":  # head-major blocks: [pool, Hkv, 128, d]
        k_cache, scales["k_scale"] = quantize_e4m3(k_cache.transpose(1, 2).contiguous())
        v_cache, scales["v_scale"] = quantize_e4m3(v_cache.transpose(1, 2).contiguous())
    return dict(
        q=q, k=k, v=v, rel=rel, k_cache=k_cache, v_cache=v_cache, **scales,
        block_table=table.to(device),
        cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=device),
        ctx_lens=torch.tensor(list(wl.ctx_lens), dtype=torch.int32, device=device),
        max_q_len=max(wl.new_tokens), num_tokens=T,
        window=wl.window, rel_extent=wl.rel_extent, workload=wl)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy array of a bf16 tensor's bit patterns (for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
