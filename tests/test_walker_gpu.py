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


@pytest.mark.parametrize("window", [0, 1, 100, 1024])
def test_prefill_walk_bit_exact(window):
    wl = I.PrefillWorkload("pw", 4, 1, 128, 128, window, 64, (1, 64, 65, 300, 200),
                           (0, 63, 128, 1000, 5))
    case = I.make_prefill(wl, DEV)
    rec, status = R.debug_walk_prefill(case["cu_seqlens"], case["ctx_lens"],
                                       case["block_table"], window, case["k_cache"],
                                       case["v_cache"], 4, case["max_q_len"])
    assert status == 0
    table = case["block_table"].cpu().numpy()
    got = defaultdict(list)
    for b, t0, tile, lblk, phys, _ in rec.tolist():
        got[(b, t0)].append((tile, lblk, phys))
    for b, (n, ctx) in enumerate(zip(wl.new_tokens, wl.ctx_lens)):
        for t0 in range(0, n, 128):
            t1 = min(n, t0 + 128) - 1
            blocks = dict(O.prefill_blocks(ctx, t0, t1, window, table[b]))
            lo, _ = O.visible_keys(ctx + t0, window)
            want = [(t, t // 2, blocks[t // 2]) for t in range(lo // 64, (ctx + t1) // 64 + 1)]
            assert sorted(got.pop((b, t0))) == want
    assert not got
