"""Float64 CPU oracle for paged relative-bias (Inkling-family) attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may import this module. It shares no
code with the CUDA path (``paged_relative_bias_gb300``) and imports nothing
from it; the two meet only through the seeded inputs that the tests hand to
both.

What is computed (every function below is the plain definition, written out;
there is no blocking, fusion or reordering):

* The logit of query i (position P_i, head h) for key j is
  ``q_i . k_j / sqrt(d_qk) + rel[i, h, P_i - j]``.  The additive relative term
  replaces RoPE ("Inkling-Small on Gaudi 2", section "Why it needed a port":
  rel[i, h, i - j] is a per-query, per-distance term; "vLLM TML Inkling
  Support", section "TML Inkling Model Architecture": a learned
  relative-position term added to the pre-softmax logits; "Inkling 2 Small on
  vLLM", architecture table row "attention": GQA with relative bias, no RoPE).
* ``rel`` is the per-query, per-head vector ``r @ rel_logits_proj`` over
  distances ``0 .. rel_extent-1`` ("Inkling-Small on Gaudi 2", section
  "Attention with a relative bias").  It is an input here.
* Reading (pages silent): a distance at or beyond ``rel_extent`` adds 0.
* Window: a sliding-window layer with window W lets query P see keys
  ``P-W+1 .. P`` -- W keys counting its own ("Inkling-Small on Gaudi 2",
  section "Decode window": the mask cuts the 512-key window at exactly 512).
  ``W <= 0`` is a global (full causal) layer.
* GQA: query head h reads KV head ``h // (Hq // Hkv)`` (reading: contiguous
  groups; the pages give only the head counts).
* Paged KV cache of 128-token blocks: the key at position ``pos`` of
  sequence b lives in physical block ``block_table[b][pos // 128]`` at slot
  ``pos % 128`` ("Inkling-Small on Gaudi 2", sections "At a glance" and
  "Attention with a relative bias": key positions come from each block's
  ordinal in the sequence's block list).
* Chunked prefill: new token t of sequence b sits at position
  ``ctx_lens[b] + t``; its key and value are written into the paged cache and
  the cached prefix is prepended ("Inkling-Small on Gaudi 2", section
  "Attention with a relative bias", prefill bullet).
* Decode: ``seq_lens[b]`` counts the current token, whose key and value are
  already in the cache, so the query position is ``seq_lens[b] - 1``
  (reading).
* Multi-token decode (verification of speculative drafts): the k newest
  tokens of a sequence, positions ``seq_lens[b] - k .. seq_lens[b] - 1``,
  each attend causally over the cache, which already holds all k keys
  ("vLLM TML Inkling Support", section "TML Inkling Model Architecture": up
  to 9 tokens per step; reading: ``seq_lens`` counts all k tokens).
* Softmax scale ``1/sqrt(d_qk)`` also when ``d_v != d_qk`` ("Inkling on Two
  DGX Sparks", section "Wall 1": head_dim 128, v_head_dim 64).
* Gated output with a sink (optional; "Inkling 2 Small on vLLM",
  architecture table row for the attention output, and the section on the
  backbone's recent additions: a sigmoid gate on each head's output together
  with a per-token attention sink).  Reading (the pages give no formula): the
  sink is one more logit per (query token, head) that joins the softmax's
  normaliser and carries no value; the gate is a logit per (query token,
  head) whose sigmoid multiplies that head's output.  Both are inputs; the
  projections that produce them are outside attention.

* Log-position scale (optional): global layers scale q and the rel logits
  by a factor that grows with the log of the position beyond 128K ("Inkling-
  Small on Gaudi 2", section "What was built").  Reading (no formula is
  given): one positive factor per query token multiplies both terms of its
  logits, ``s_i * (q_i . k_j / sqrt(d_qk) + rel[i, h, P_i - j])``; the factor
  is an input (1 below 128K), computed by the model, and a sink logit is not
  scaled.

* FP8 KV cache (optional, decode): keys and values stored as e4m3 (1 sign,
  4 exponent bits with bias 7, 3 mantissa bits, no infinities) times one
  scale per cache ("vLLM TML Inkling Support": FP8 global attention is on
  the roadmap; reading, as no format is given: the e4m3 format with a
  per-tensor scale, key = k_scale * e4m3 value, value = v_scale * e4m3
  value).

Data conventions: bf16 tensors are passed as ``np.uint16`` arrays of bf16 bit
patterns and e4m3 tensors as ``np.uint8`` arrays of e4m3 bit patterns (both
converted exactly here); float arrays are used as float64.
Layouts: q ``[rows, Hq, d_qk]``, rel ``[rows, Hq, E]``, k cache
``[NB, 128, Hkv, d_qk]``, v cache ``[NB, 128, Hkv, d_v]``, block_table
``[B, max_blocks]`` int.

Every function here is pinned by ``tests/test_oracle.py`` (brute force,
closed forms, library reductions, invariants); none is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

BLOCK_SIZE = 128


# --------------------------------------------------------------------------
# exact conversions
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns: bf16 is the top half of a binary32."""
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as uint16 bit patterns")
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(bits) -> np.ndarray:
    """Exact value of e4m3 bit patterns: (-1)^s * 2^(e-7) * (1 + m/8) for
    e > 0, (-1)^s * 2^-6 * m/8 for e = 0; the pattern e = 15, m = 7 is NaN."""
    b = np.asarray(bits)
    if b.dtype != np.uint8:
        raise TypeError("e4m3 data must be passed as uint8 bit patterns")
    b = b.astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# every finite non-negative e4m3 value, in code order 0x00 .. 0x7E
_E4M3_POS = None


def e4m3_encode(x) -> np.ndarray:
    """The e4m3 code of each value: the nearest finite e4m3 value, ties to
    the even code (even mantissa), the sign kept (also for zero); magnitudes
    above the largest finite value, 448, give 448 (saturation to finite is
    this library's reading: the pages give no quantiser), NaN gives 0x7F."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    lo = np.clip(np.searchsorted(_E4M3_POS, mag, side="right") - 1, 0, 0x7E)  # value <= mag
    hi = np.minimum(lo + 1, 0x7E)
    d_lo = mag - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - mag
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(mag >= 448.0, 0x7E, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def e4m3_quantize(bf16_bits, scale: float) -> np.ndarray:
    """Codes of bf16 values divided by a per-tensor scale: the division in
    float32 (as the cache-writing kernel does it), then e4m3_encode."""
    x = bf16_bits_to_f64(bf16_bits).astype(np.float32)
    return e4m3_encode(x / np.float32(scale))


def as_f64(x) -> np.ndarray:
    """float64 view of an input: uint16 is read as bf16 bits, uint8 as e4m3
    bits, floats widen."""
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    if a.dtype == np.uint8:
        return e4m3_bits_to_f64(a)
    return a.astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even of float64 values to bf16 bit patterns.

    Used only to build inputs for the oracle's own tests; rounds through
    binary32 first (exact for the values the tests use) and then to bf16.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


# --------------------------------------------------------------------------
# window and block selection (integer, bit-exact)
# --------------------------------------------------------------------------

def visible_keys(P: int, window: int) -> tuple[int, int]:
    """Inclusive key range [lo, P] seen by a query at position P.

    Sliding window W: W keys counting the query's own ("Inkling-Small on
    Gaudi 2", section "Decode window").  W <= 0: every earlier key.
    """
    lo = max(0, P - window + 1) if window > 0 else 0
    return lo, P


def logical_block_range(lo: int, hi: int) -> tuple[int, int]:
    """Inclusive logical block range holding key positions lo..hi."""
    return lo // BLOCK_SIZE, hi // BLOCK_SIZE


def decode_blocks(seq_len: int, window: int, table_row) -> list[tuple[int, int]]:
    """Window-aware block walk for one decode query.

    Returns [(logical_block, physical_block)] for every block holding a key
    the query sees.  A local layer touches only its last ceil(W/128)+1 blocks
    ("Inkling-Small on Gaudi 2", sections "Decode window" -- one block more
    than window/block_size -- and "Attention with a relative bias", local
    window prefill: the last 5 blocks for W = 512).
    """
    P = seq_len - 1
    lo, hi = visible_keys(P, window)
    first, last = logical_block_range(lo, hi)
    return [(l, int(table_row[l])) for l in range(first, last + 1)]


def prefill_blocks(ctx_len: int, t_first: int, t_last: int, window: int,
                   table_row) -> list[tuple[int, int]]:
    """Block walk for the new tokens t_first..t_last of one prefill chunk.

    Their positions are ctx_len + t; the union of their visible keys is
    [max(0, ctx_len + t_first - W + 1), ctx_len + t_last]
    ("Inkling-Small on Gaudi 2", section "Attention with a relative bias").
    """
    lo, _ = visible_keys(ctx_len + t_first, window)
    hi = ctx_len + t_last
    first, last = logical_block_range(lo, hi)
    return [(l, int(table_row[l])) for l in range(first, last + 1)]


# --------------------------------------------------------------------------
# paged cache access
# --------------------------------------------------------------------------

def gather_kv(k_cache, v_cache, table_row, positions, kv_head: int, k_scale=1.0,
              v_scale=1.0):
    """Keys and values at the given positions of one sequence, float64.

    Position pos lives at slot pos % 128 of physical block
    table_row[pos // 128] ("Inkling-Small on Gaudi 2", section "Attention
    with a relative bias": positions from each block's ordinal).  An FP8
    cache's entries are multiplied by its scale.
    """
    pos = np.asarray(positions, dtype=np.int64)
    phys = np.asarray(table_row, dtype=np.int64)[pos // BLOCK_SIZE]
    slot = pos % BLOCK_SIZE
    K = as_f64(k_cache[phys, slot, kv_head]) * float(k_scale)
    V = as_f64(v_cache[phys, slot, kv_head]) * float(v_scale)
    return K, V


def kv_cache_write(k_cache, v_cache, k, v, cu_seqlens, ctx_lens, block_table):
    """Copy of the caches with each new token's key and value scattered in.

    New token t of sequence b (packed row cu_seqlens[b] + t) goes to slot
    (ctx_lens[b] + t) % 128 of physical block
    block_table[b][(ctx_lens[b] + t) // 128].  A pure copy: bit-exact.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    B = len(ctx_lens)
    for b in range(B):
        r0, r1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        for t in range(r1 - r0):
            pos = int(ctx_lens[b]) + t
            phys = int(block_table[b][pos // BLOCK_SIZE])
            kc[phys, pos % BLOCK_SIZE] = k[r0 + t]
            vc[phys, pos % BLOCK_SIZE] = v[r0 + t]
    return kc, vc


def kv_cache_write_e4m3(k_cache, v_cache, k, v, cu_seqlens, ctx_lens, block_table,
                        k_scale: float, v_scale: float):
    """kv_cache_write into e4m3 caches (uint8 codes, layout [NB, 128, Hkv, d]):
    the same slots, each bf16 key quantised with k_scale and each value with
    v_scale (e4m3_quantize).  Bit-exact."""
    return kv_cache_write(k_cache, v_cache, e4m3_quantize(k, k_scale),
                          e4m3_quantize(v, v_scale), cu_seqlens, ctx_lens, block_table)


# --------------------------------------------------------------------------
# the attention of one query row
# --------------------------------------------------------------------------

def rel_bias(rel_vec, P: int, keys, rel_extent: int) -> np.ndarray:
    """Relative term rel[P - j] for each key j; 0 at distances >= rel_extent."""
    d = P - np.asarray(keys, dtype=np.int64)
    out = np.zeros(d.shape, dtype=np.float64)
    inside = d < rel_extent
    out[inside] = as_f64(rel_vec)[d[inside]]
    return out


def logits(q_vec, K, bias, d_qk: int) -> np.ndarray:
    """q . k_j / sqrt(d_qk) + bias_j for every key row of K."""
    return (K @ as_f64(q_vec)) / math.sqrt(d_qk) + bias


def softmax_weights(s) -> np.ndarray:
    """exp(s - max s) / sum: the attention weights of one query."""
    s = np.asarray(s, dtype=np.float64)
    w = np.exp(s - s.max())
    return w / w.sum()


def attend(q_vec, K, V, bias, d_qk: int, sink=None, gate=None, scale=None) -> np.ndarray:
    """Output of one query: softmax(logits) @ V.

    With a log-position factor the logits are ``scale * logits``; with a
    sink logit s the weights are exp(l_j) / (sum_j exp(l_j) + exp(s)); with a
    gate logit g the output is multiplied by 1 / (1 + exp(-g)).
    """
    s = logits(q_vec, K, bias, d_qk)
    if scale is not None:
        s = float(scale) * s
    if sink is None:
        w = softmax_weights(s)
    else:
        m = max(s.max(), float(sink))
        e = np.exp(s - m)
        w = e / (e.sum() + math.exp(float(sink) - m))
    out = w @ V
    if gate is not None:
        out = out / (1.0 + math.exp(-float(gate)))
    return out


def attend_partial(q_vec, K, V, bias, d_qk: int):
    """Un-merged softmax state of one key subset: (normalised o, lse).

    This is what one split of split-KV decode produces ("vLLM TML Inkling
    Support", section "Low-Latency Collectives and Kernels": num_splits).
    lse = m + log(sum exp(s - m)) in natural log.
    """
    s = logits(q_vec, K, bias, d_qk)
    m = s.max()
    w = np.exp(s - m)
    return (w @ V) / w.sum(), m + math.log(w.sum())


def merge_partials(outs, lses) -> np.ndarray:
    """Merge split results: weights exp(lse_s - max lse) over the splits."""
    lses = np.asarray(lses, dtype=np.float64)
    m = lses.max()
    w = np.exp(lses - m)
    return (w[:, None] * np.asarray(outs, dtype=np.float64)).sum(0) / w.sum()


# --------------------------------------------------------------------------
# whole calls
# --------------------------------------------------------------------------

def decode(q, rel, k_cache, v_cache, block_table, seq_lens, window: int,
           rel_extent: int, batch=None, heads=None, sink=None, gate=None, k_scale=1.0,
           v_scale=1.0, logit_scale=None) -> np.ndarray:
    """Paged decode: one query per sequence at position seq_lens[b] - 1.

    ``sink`` / ``gate``: optional [B, Hq] logits, ``logit_scale``: optional
    [B] log-position factors (see ``attend``);
    ``k_scale`` / ``v_scale``: the scales of an FP8 cache.  Returns
    float64 [B, Hq, d_v]; rows/heads not selected by ``batch`` / ``heads``
    are left NaN.
    """
    B, Hq, d_qk = q.shape
    Hkv = k_cache.shape[2]
    g = Hq // Hkv
    d_v = v_cache.shape[3]
    out = np.full((B, Hq, d_v), np.nan)
    for b in (range(B) if batch is None else batch):
        L = int(seq_lens[b])
        P = L - 1
        lo, hi = visible_keys(P, window)
        keys = np.arange(lo, hi + 1)
        for kvh in range(Hkv):
            hs = [h for h in range(kvh * g, (kvh + 1) * g)
                  if heads is None or h in heads]
            if not hs:
                continue
            K, V = gather_kv(k_cache, v_cache, block_table[b], keys, kvh, k_scale, v_scale)
            for h in hs:
                bias = rel_bias(rel[b, h], P, keys, rel_extent)
                out[b, h] = attend(q[b, h], K, V, bias, d_qk,
                                   None if sink is None else sink[b, h],
                                   None if gate is None else gate[b, h],
                                   None if logit_scale is None else logit_scale[b])
    return out


def decode_multi(q, rel, k_cache, v_cache, block_table, seq_lens, window: int,
                 rel_extent: int, batch=None, tokens=None, heads=None, sink=None,
                 gate=None, k_scale=1.0, v_scale=1.0, logit_scale=None) -> np.ndarray:
    """Multi-token decode, the verification step of speculative decoding.

    The k newest tokens of sequence b each attend over the paged cache:
    token i sits at position ``seq_lens[b] - k + i`` and sees keys
    ``max(0, P - W + 1) .. P``, causal and windowed.  The keys and values of
    all k tokens are already in the cache ("vLLM TML Inkling Support",
    section "TML Inkling Model Architecture": chained MTP heads propose up to
    9 tokens per forward step; "Inkling 2 Small on vLLM", section "vLLM
    integration and optimisation": one kernel serves decode and
    verification, with the heads of a KV group packed into one tile).
    Reading (pages silent): ``seq_lens`` counts all k tokens, as it counts
    the one token of a decode step.

    q ``[B, k, Hq, d_qk]``, rel ``[B, k, Hq, E]``, optional ``sink`` /
    ``gate`` ``[B, k, Hq]`` and ``logit_scale`` ``[B, k]``.  Returns float64 ``[B, k, Hq, d_v]``; entries not
    selected by ``batch`` / ``tokens`` / ``heads`` are left NaN.
    """
    B, kq, Hq, d_qk = q.shape
    Hkv = k_cache.shape[2]
    g = Hq // Hkv
    d_v = v_cache.shape[3]
    out = np.full((B, kq, Hq, d_v), np.nan)
    for b in (range(B) if batch is None else batch):
        L = int(seq_lens[b])
        for i in (range(kq) if tokens is None else tokens):
            P = L - kq + i
            lo, hi = visible_keys(P, window)
            keys = np.arange(lo, hi + 1)
            for kvh in range(Hkv):
                hs = [h for h in range(kvh * g, (kvh + 1) * g)
                      if heads is None or h in heads]
                if not hs:
                    continue
                K, V = gather_kv(k_cache, v_cache, block_table[b], keys, kvh, k_scale,
                                 v_scale)
                for h in hs:
                    bias = rel_bias(rel[b, i, h], P, keys, rel_extent)
                    out[b, i, h] = attend(q[b, i, h], K, V, bias, d_qk,
                                          None if sink is None else sink[b, i, h],
                                          None if gate is None else gate[b, i, h],
                                          None if logit_scale is None else logit_scale[b, i])
    return out


def prefill(q, k, v, rel, cu_seqlens, k_cache, v_cache, block_table,
            ctx_lens, window: int, rel_extent: int, rows=None, sink=None, gate=None,
            logit_scale=None, k_scale=1.0, v_scale=1.0):
    """Chunked prefill against the paged cache.

    Writes the new keys/values into copies of the caches, then attends each
    new token (position ctx_lens[b] + t) over the cached prefix plus the new
    tokens, causal and windowed.  ``rows`` selects packed token rows to
    compute (default: all); ``sink`` / ``gate``: optional [T, Hq] logits,
    ``logit_scale``: optional [T] log-position factors (see ``attend``).
    e4m3 caches (uint8 codes) take the new tokens quantised with ``k_scale`` /
    ``v_scale`` (``kv_cache_write_e4m3``) and are read back with them.
    Returns (out float64 [T, Hq, d_v] with unselected rows NaN, k_cache',
    v_cache').
    """
    T, Hq, d_qk = q.shape
    Hkv = k_cache.shape[2]
    g = Hq // Hkv
    d_v = v_cache.shape[3]
    if np.asarray(k_cache).dtype == np.uint8:  # e4m3 caches: quantise the new tokens
        kc, vc = kv_cache_write_e4m3(k_cache, v_cache, k, v, cu_seqlens, ctx_lens,
                                     block_table, k_scale, v_scale)
    else:
        kc, vc = kv_cache_write(k_cache, v_cache, k, v, cu_seqlens, ctx_lens,
                                block_table)
    out = np.full((T, Hq, d_v), np.nan)
    B = len(ctx_lens)
    want = None if rows is None else set(int(r) for r in rows)
    for b in range(B):
        r0, r1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        for t in range(r1 - r0):
            row = r0 + t
            if want is not None and row not in want:
                continue
            P = int(ctx_lens[b]) + t
            lo, hi = visible_keys(P, window)
            keys = np.arange(lo, hi + 1)
            for kvh in range(Hkv):
                K, V = gather_kv(kc, vc, block_table[b], keys, kvh, k_scale, v_scale)
                for h in range(kvh * g, (kvh + 1) * g):
                    bias = rel_bias(rel[row, h], P, keys, rel_extent)
                    out[row, h] = attend(q[row, h], K, V, bias, d_qk,
                                         None if sink is None else sink[row, h],
                                         None if gate is None else gate[row, h],
                                         None if logit_scale is None else logit_scale[row])
    return out, kc, vc


def decode_weights(q_vec, rel_vec, k_cache, v_cache, table_row, seq_len: int,
                   kv_head: int, window: int, rel_extent: int):
    """(keys, weights) of one decode query: the attention distribution."""
    P = seq_len - 1
    lo, hi = visible_keys(P, window)
    keys = np.arange(lo, hi + 1)
    K, _ = gather_kv(k_cache, v_cache, table_row, keys, kv_head)
    bias = rel_bias(rel_vec, P, keys, rel_extent)
    return keys, softmax_weights(logits(q_vec, K, bias, K.shape[1]))
