"""The device block walk is bit-exact against the oracle's block selection.

Decode walks 64-key tiles per (sequence, KV head); prefill walks the 64-key
tiles of each 128-row query tile.

The decode and prefill kernels' walk (which tiles, which physical blocks,
which CTA) is replayed by the library's debug entry points and compared with
the oracle's independent integer functions.
"""

from collections import defaultdict

import numpy as np
import pytest
import torch

from oracle import relattn_oracle as O
from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def expected_decode_tiles(seq_len, window, table_row):
    """64-key tiles holding a visible key, from the oracle's block walk."""
    P = seq_len - 1
    lo, hi = O.visible_keys(P, window)
    blocks = dict(O.decode_blocks(seq_len, window, table_row))
    return [(t, t // 2, blocks[t // 2]) for t in range(lo // 64, hi // 64 + 1)]


@pytest.mark.parametrize("window", [0, 1, 64, 100, 512, 1024])
@pytest.mark.parametrize("num_ctas", [0, 1, 5, 300])
def test_decode_walk_bit_exact(window, num_ctas):
    lens = [1, 63, 64, 65, 128, 129, 511, 512, 513, 1000, 4097, 20000, 77, 3]
    wl = I.DecodeWorkload("walk", len(lens), 8, 4, 128, 128, window, 64, ("list", lens))
    case = I.make_decode(wl, DEV)
    rec, status = R.debug_walk_decode(case["block_table"], case["seq_lens"], window,
                                      case["k_cache"], case["v_cache"], 8, num_ctas=num_ctas)
    assert status == 0
    rec = rec.numpy()
    table = case["block_table"].cpu().numpy()
    seen = defaultdict(list)
    for cta, b, kvh, tile, lblk, phys in rec:
        seen[(b, kvh)].append((int(cta), int(tile), int(lblk), int(phys)))
    for b, L in enumerate(lens):
        want = expected_decode_tiles(L, window, table[b])
        if window > 0:
            assert len({l for _, l, _ in want}) <= -(-window // 128) + 1
        for kvh in range(4):
            # records arrive in any order (CTAs append concurrently)
            got = sorted(seen.pop((b, kvh)), key=lambda r: r[1])
            # each tile exactly once; along the tiles the owning CTA never decreases
            assert [(t, l, p) for _, t, l, p in got] == want
            ctas = [c for c, _, _, _ in got]
            assert ctas == sorted(ctas)
    assert not seen
    # each CTA owns one contiguous run of the flattened work
    order = sorted(rec.tolist(), key=lambda r: (r[1], r[2], r[3]))
    ctas = [r[0] for r in order]
    assert ctas == sorted(ctas)


def test_decode_walk_windowed_block_count_matches_page_fact():
    """A 512-key local layer reads at most 5 blocks (512/128 + 1)."""
    lens = list(range(500, 1800, 7))
    wl = I.DecodeWorkload("w512", len(lens), 4, 1, 128, 128, 512, 512, ("list", lens))
    case = I.make_decode(wl, DEV)
    rec, _ = R.debug_walk_decode(case["block_table"], case["seq_lens"], 512,
                                 case["k_cache"], case["v_cache"], 4)
    per_seq = defaultdict(set)
    for _, b, _, _, lblk, _ in rec.tolist():
        per_seq[b].add(lblk)
    assert max(len(s) for s in per_seq.values()) == 5
    for b, L in enumerate(lens):
        assert sorted(per_seq[b]) == [l for l, _ in O.decode_blocks(L, 512, np.arange(300))]


@pytest.mark.parametrize("heads", [(4, 1), (6, 2), (3, 1), (2, 2)])
@pytest.mark.parametrize("window", [0, 1, 100, 1024])
def test_prefill_walk_bit_exact(window, heads):
    """Every (query tile, head pair) item visits exactly the oracle's key
    tiles; the items cover each query head once (pairs of a KV group, the
    last one alone when the group size is odd)."""
    hq, hkv = heads
    g = hq // hkv
    wl = I.PrefillWorkload("pw", hq, hkv, 128, 128, window, 64, (1, 64, 65, 300, 200),
                           (0, 63, 128, 1000, 5))
    case = I.make_prefill(wl, DEV)
    rec, status = R.debug_walk_prefill(case["cu_seqlens"], case["ctx_lens"],
                                       case["block_table"], window, case["k_cache"],
                                       case["v_cache"], hq, case["max_q_len"])
    assert status == 0
    table = case["block_table"].cpu().numpy()
    got = defaultdict(list)
    for b, t0, tile, lblk, phys, h0 in rec.tolist():
        got[(b, t0, h0)].append((tile, lblk, phys))
    firsts = [kvh * g + 2 * j for kvh in range(hkv) for j in range((g + 1) // 2)]
    for b, (n, ctx) in enumerate(zip(wl.new_tokens, wl.ctx_lens)):
        for t0 in range(0, n, 128):
            t1 = min(n, t0 + 128) - 1
            blocks = dict(O.prefill_blocks(ctx, t0, t1, window, table[b]))
            lo, _ = O.visible_keys(ctx + t0, window)
            want = [(t, t // 2, blocks[t // 2]) for t in range(lo // 64, (ctx + t1) // 64 + 1)]
            for h0 in firsts:
                assert sorted(got.pop((b, t0, h0))) == want
    assert not got


@pytest.mark.parametrize("heads", [(4, 1), (6, 2), (3, 1), (2, 2)])
@pytest.mark.parametrize("window", [0, 1, 100, 1024])
def test_prefill_walk_wide_bit_exact(window, heads):
    """With a bf16 rel (d_v = 128, bf16 cache) the prefill's work items are one
    128-row query tile and one head over 128-key tiles: every item visits
    exactly the blocks holding a key that one of its rows sees, the oracle's
    block walk, and the items cover every (query tile, head) once."""
    hq, hkv = heads
    wl = I.PrefillWorkload("pww", hq, hkv, 128, 128, window, 64, (1, 64, 65, 300, 200),
                           (0, 63, 128, 1000, 5))
    case = I.make_prefill(wl, DEV)
    rec, status = R.debug_walk_prefill(case["cu_seqlens"], case["ctx_lens"],
                                       case["block_table"], window, case["k_cache"],
                                       case["v_cache"], hq, case["max_q_len"],
                                       rel_dtype=torch.bfloat16)
    assert status == 0
    table = case["block_table"].cpu().numpy()
    got = defaultdict(list)
    for b, t0, tile, lblk, phys, h in rec.tolist():
        got[(b, t0, h)].append((tile, lblk, phys))
    for b, (n, ctx) in enumerate(zip(wl.new_tokens, wl.ctx_lens)):
        for t0 in range(0, n, 128):
            t1 = min(n, t0 + 128) - 1
            blocks = dict(O.prefill_blocks(ctx, t0, t1, window, table[b]))
            want = [(lb, lb, blocks[lb]) for lb in sorted(blocks)]
            for h in range(hq):
                assert sorted(got.pop((b, t0, h))) == want
    assert not got


def chunk_tokens(k, g):
    """Query tokens per chunk: one 16-row tile's worth of (token, head) rows,
    or 32 rows when more tokens than one tile holds share a KV head (g <= 8)
    in the general kernel (several tokens, or g > 8)."""
    multi = k > 1 or g > 8
    rows = 32 if multi and g <= 8 and k * g > 16 else 16
    return min(k, rows // g)


def expected_chunk_tiles(L, k, kpc, window, table_row, halves):
    """{first token of chunk: [(tile, physical block, first key, keys)]} from
    the oracle's key ranges: a chunk reads the tiles of [lo of its first
    token, position of its last token]; with halves, a tile brings the 32-key
    halves that hold a visible key."""
    out = {}
    for i0 in range(0, k, kpc):
        kc = min(kpc, k - i0)
        pf = L - k + i0
        pl = pf + kc - 1
        lo, _ = O.visible_keys(pf, window)
        tiles = []
        for t in range(lo // 64, pl // 64 + 1):
            key0 = 64 * t
            if halves:
                parts = [h for h in (0, 1) if key0 + 32 * h <= pl and key0 + 32 * h + 31 >= lo]
                first, n = key0 + 32 * parts[0], 32 * len(parts)
            else:
                first, n = key0, 64
            tiles.append((t, int(table_row[t // 2]), first, n))
        out[i0] = tiles
    return out


@pytest.mark.parametrize("k,hq,kv", [(1, 32, "bf16"), (1, 32, "fp8"), (2, 32, "bf16"),
                                     (8, 32, "bf16"), (9, 32, "bf16"), (16, 32, "bf16"),
                                     (3, 48, "bf16"), (1, 128, "bf16"), (9, 32, "fp8"),
                                     (5, 8, "bf16")])
@pytest.mark.parametrize("window", [0, 1, 100, 512])
@pytest.mark.parametrize("num_ctas", [0, 7])
def test_decode_walk_chunks_and_half_tiles_bit_exact(k, hq, kv, window, num_ctas):
    """The walk of the multi-token kernel (chunks of query tokens) and the
    half tiles of the one-token kernel at the edges of the key range, against
    the oracle's key ranges; every tile once per (chunk, KV head)."""
    lens = [16, 17, 63, 64, 65, 127, 128, 129, 500, 513, 1000, 2049]
    hkv = 8
    g = hq // hkv
    wl = I.DecodeWorkload("walk", len(lens), hq, hkv, 128, 128, window, 64, ("list", lens),
                          kv_dtype=kv)
    case = I.make_decode(wl, DEV)
    rec, status = R.debug_walk_decode_ex(case["block_table"], case["seq_lens"], k, window,
                                         case["k_cache"], case["v_cache"], hq,
                                         num_ctas=num_ctas)
    assert status == 0
    table = case["block_table"].cpu().numpy()
    kpc = chunk_tokens(k, g)
    halves = k == 1 and g <= 8 and kv == "bf16"
    seen = defaultdict(list)
    for cta, b, i0, kvh, tile, phys, first, n in rec.tolist():
        seen[(b, i0, kvh)].append((cta, tile, phys, first, n))
    for b, L in enumerate(lens):
        want = expected_chunk_tiles(L, k, kpc, window, table[b], halves)
        for i0, tiles in want.items():
            for kvh in range(hkv):
                got = sorted(seen.pop((b, i0, kvh)), key=lambda r: r[1])
                assert [r[1:] for r in got] == tiles, (b, L, i0, kvh)
                ctas = [r[0] for r in got]
                assert ctas == sorted(ctas)
    assert not seen
