"""GPU chunked prefill vs the float64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from paged_relative_bias_gb300.inputs import bf16_bits
from tests.parity import assert_parity, oracle_prefill, snapshot_cache, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def run_prefill(case, ws=None, num_ctas=0):
    return R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"],
                             case["cu_seqlens"], case["k_cache"], case["v_cache"],
                             case["block_table"], case["ctx_lens"], case["window"],
                             case["rel_extent"], case["max_q_len"], workspace=ws,
                             num_ctas=num_ctas)


def check_case(case, rows=None, what="", num_ctas=0):
    cache0 = snapshot_cache(case)
    want, kc_want, vc_want = oracle_prefill(case, rows=rows, cache=cache0)
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"],
                          case["max_q_len"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out = run_prefill(case, ws, num_ctas)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    # the cache write is a copy: bit-exact, everywhere
    assert np.array_equal(bf16_bits(case["k_cache"]), kc_want), "k cache"
    assert np.array_equal(bf16_bits(case["v_cache"]), vc_want), "v cache"
    got = to_f64(out)
    sel = slice(None) if rows is None else list(rows)
    return assert_parity(got[sel], want[sel], what=what)


# num_ctas 0: the library's choice (small calls: one head per work item);
# 148: a forced grid, which keeps two heads of a KV group per work item
GRIDS = [0, 148]


@pytest.mark.parametrize("num_ctas", GRIDS)
def test_tiny_prefill_config(num_ctas):
    """1 x 256 tokens, 4/1 heads, window = rel_extent = 64, table [1, 0]."""
    case = I.make_prefill(I.WORKLOADS["tiny_prefill"], DEV)
    check_case(case, what="tiny", num_ctas=num_ctas)


SMALL = {
    "prefix_window": I.PrefillWorkload("pw", 12, 2, 128, 128, 100, 64, (200, 77), (300, 0)),
    "global_dv64": I.PrefillWorkload("g64", 8, 2, 128, 64, 0, 256, (130, 1, 64), (0, 500, 129)),
    "gqa6_w1024": I.PrefillWorkload("g6", 12, 2, 128, 128, 1024, 1024, (300, 190), (1100, 2000)),
    "extent_lt_window": I.PrefillWorkload("el", 4, 1, 128, 128, 700, 128, (400,), (333,)),
    "window1": I.PrefillWorkload("w1", 4, 2, 128, 128, 1, 4, (70,), (10,)),
    "ragged_many": I.PrefillWorkload("rm", 8, 8, 128, 128, 256, 512,
                                     (1, 63, 64, 65, 127, 128, 129, 200),
                                     (0, 1, 127, 128, 129, 0, 64, 1000)),
}


@pytest.mark.parametrize("num_ctas", GRIDS)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_prefill_small_configs(name, num_ctas):
    case = I.make_prefill(SMALL[name], DEV, seed_data=2, seed_layout=3)
    check_case(case, what=name, num_ctas=num_ctas)


# Head-group sizes and grids for the two-heads-per-item kernel: odd groups
# leave one head alone in an item (the second softmax group skips it), and a
# small grid makes each CTA run many items back to back through its ring.
ITEMS = {
    "g3_three_ctas": (I.PrefillWorkload("g3", 6, 2, 128, 128, 300, 256, (260, 129), (70, 0)), 3),
    "g5_one_cta": (I.PrefillWorkload("g5", 5, 1, 128, 128, 0, 128, (300,), (40,)), 1),
    "g1_two_ctas": (I.PrefillWorkload("g1", 2, 2, 128, 64, 200, 128, (257, 3), (0, 90)), 2),
    "g6_seven_ctas": (I.PrefillWorkload("g6s", 12, 2, 128, 128, 1024, 1024, (384, 100),
                                        (700, 0)), 7),
    "g2_bf16_many_items": (I.PrefillWorkload("g2m", 8, 4, 128, 128, 512, 512, (640, 512),
                                             (1000, 64)), 5),
}


@pytest.mark.parametrize("name", sorted(ITEMS))
def test_prefill_items_and_grids(name):
    wl, ctas = ITEMS[name]
    case = I.make_prefill(wl, DEV, seed_data=6, seed_layout=7)
    check_case(case, what=name, num_ctas=ctas)


def test_prefill_then_decode_agree():
    """Decode after a prefill of L tokens equals the prefill's last row."""
    wl = I.PrefillWorkload("pd", 8, 2, 128, 128, 300, 512, (400,), (0,))
    case = I.make_prefill(wl, DEV, seed_data=4)
    out = run_prefill(case)
    L = 400
    dec = R.relattn_decode(case["q"][L - 1:L].contiguous(), case["rel"][L - 1:L].contiguous(),
                           case["k_cache"], case["v_cache"], case["block_table"],
                           torch.tensor([L], dtype=torch.int32, device=DEV), 300, 512)
    torch.cuda.synchronize()
    d = (dec[0].float() - out[L - 1].float()).abs().max().item()
    assert d <= 2e-2


def test_chunked_prefill_full_size_sampled():
    """4 x 8192 new tokens after 24,576 cached, 48/8 heads, W = E = 1024."""
    case = I.make_prefill(I.WORKLOADS["chunked_prefill"], DEV)
    cu = case["cu_seqlens"].cpu().tolist()
    rng = np.random.default_rng(1)
    rows = set()
    for b in range(len(cu) - 1):
        r0, r1 = cu[b], cu[b + 1]
        rows |= {r0, r0 + 1, r0 + 127, r0 + 128, r1 - 1}
        rows |= set(int(x) for x in rng.integers(r0, r1, size=6))
    check_case(case, rows=sorted(rows), what="chunked_prefill")
