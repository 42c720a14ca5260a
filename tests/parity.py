"""Helpers for GPU-vs-oracle parity tests.

Tolerance: the GPU computes in bf16 with fp32 accumulation and writes bf16;
outputs must match the float64 oracle within max-abs 2e-2 and mean-abs 2e-3.
"""

import numpy as np
import torch

from oracle import relattn_oracle as O
from paged_relative_bias_gb300.inputs import bf16_bits

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def assert_parity(got, want, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - want)
    assert d.max() <= max_abs, f"{what}: max abs diff {d.max():.3e} > {max_abs}"
    assert d.mean() <= mean_abs, f"{what}: mean abs diff {d.mean():.3e} > {mean_abs}"
    return float(d.max()), float(d.mean())


def to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return O.bf16_bits_to_f64(bf16_bits(t))
    return t.detach().cpu().double().numpy()


def host_cache(t: torch.Tensor):
    """A KV cache for the oracle ([NB, 128, Hkv, d]): bf16 bit patterns, or
    the e4m3 bit patterns of a head-major [NB, Hkv, 128, d] e4m3 cache."""
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).transpose(1, 2).contiguous().cpu().numpy()
    return bf16_bits(t)


def host_rel(rel: torch.Tensor):
    """rel for the oracle: float32 values, or bf16 bit patterns."""
    return bf16_bits(rel) if rel.dtype == torch.bfloat16 else rel.cpu().numpy()


def host_decode_inputs(case):
    """numpy copies of a decode case for the oracle (bf16 kept as bits)."""
    return dict(
        q=bf16_bits(case["q"]), rel=host_rel(case["rel"]),
        k_cache=host_cache(case["k_cache"]), v_cache=host_cache(case["v_cache"]),
        block_table=case["block_table"].cpu().numpy(),
        seq_lens=case["seq_lens"].cpu().numpy())


def host_opt(case, name):
    """An optional per-query-row (and head) input of a case, as numpy or None."""
    t = case.get(name)
    return None if t is None else t.cpu().double().numpy()


def oracle_decode(case, batch=None, heads=None):
    h = host_decode_inputs(case)
    return O.decode(h["q"], h["rel"], h["k_cache"], h["v_cache"], h["block_table"],
                    h["seq_lens"], case["window"], case["rel_extent"], batch=batch,
                    heads=heads, sink=host_opt(case, "sink"), gate=host_opt(case, "gate"),
                    k_scale=case.get("k_scale", 1.0), v_scale=case.get("v_scale", 1.0),
                    logit_scale=host_opt(case, "logit_scale"))


class RowRel:
    """rel rows of a few packed tokens, indexable as rel[row, h]."""

    def __init__(self, rel: torch.Tensor, rows):
        self.rows = {int(r): host_rel(rel[int(r)]) for r in rows}

    def __getitem__(self, idx):
        row, h = idx
        return self.rows[int(row)][h]


class RowQ(RowRel):
    def __init__(self, q: torch.Tensor, rows):
        self.rows = {int(r): bf16_bits(q[int(r)]) for r in rows}

    @property
    def shape(self):
        return self._shape


def snapshot_cache(case):
    """Host copy of the paged cache (take it before a prefill writes into it),
    in the oracle's [NB, 128, Hkv, d] layout."""
    return host_cache(case["k_cache"]), host_cache(case["v_cache"])


def oracle_prefill(case, rows=None, cache=None):
    """Oracle prefill over the case's inputs (rows: packed token rows to check).

    ``cache``: (k, v) host bits of the cache before the prefill; defaults to
    the case's current device cache.
    """
    q, rel = case["q"], case["rel"]
    kc, vc = cache if cache is not None else snapshot_cache(case)
    if rows is None:
        qn, reln = bf16_bits(q), host_rel(rel)
    else:
        qn = RowQ(q, rows)
        qn._shape = tuple(q.shape)
        reln = RowRel(rel, rows)
    return O.prefill(qn, bf16_bits(case["k"]), bf16_bits(case["v"]), reln,
                     case["cu_seqlens"].cpu().numpy(), kc, vc,
                     case["block_table"].cpu().numpy(),
                     case["ctx_lens"].cpu().numpy(), case["window"], case["rel_extent"],
                     rows=rows, sink=host_opt(case, "sink"), gate=host_opt(case, "gate"),
                     logit_scale=host_opt(case, "logit_scale"),
                     k_scale=case.get("k_scale", 1.0), v_scale=case.get("v_scale", 1.0))


def oracle_decode_multi(case, batch=None, tokens=None, heads=None):
    h = host_decode_inputs(case)
    return O.decode_multi(h["q"], h["rel"], h["k_cache"], h["v_cache"], h["block_table"],
                          h["seq_lens"], case["window"], case["rel_extent"], batch=batch,
                          tokens=tokens, heads=heads, sink=host_opt(case, "sink"),
                          gate=host_opt(case, "gate"), k_scale=case.get("k_scale", 1.0),
                          v_scale=case.get("v_scale", 1.0),
                          logit_scale=host_opt(case, "logit_scale"))
