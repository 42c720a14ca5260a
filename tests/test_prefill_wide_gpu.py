"""GPU chunked prefill over a bf16 cache with a bf16 rel and d_v = 128: one
query head per work item and 128-key tiles (a whole cache block per tile),
the two softmax groups splitting each tile's columns.

A forced grid (num_ctas > 0) keeps these calls off the one-wave path, and
small grids make every CTA run many items back to back through its rings
(the next query preloaded during an epilogue, S double-buffered across item
boundaries).  Every case is compared with the float64 oracle element by
element; the cache write stays bit-exact.
"""

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


def bf16_rel(wl):
    return I.variant(wl, rel_dtype="bf16")


def run(case, num_ctas, out_dtype=torch.bfloat16, **extra):
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"],
                          num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out = R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                            case["k_cache"], case["v_cache"], case["block_table"],
                            case["ctx_lens"], case["window"], case["rel_extent"],
                            case["max_q_len"], workspace=ws, out_dtype=out_dtype,
                            num_ctas=num_ctas, **extra)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    return out


def check(case, num_ctas, what, out_dtype=torch.bfloat16, **extra):
    cache0 = snapshot_cache(case)
    want, kc_want, vc_want = oracle_prefill(case, cache=cache0)
    out = run(case, num_ctas, out_dtype, **extra)
    assert np.array_equal(bf16_bits(case["k_cache"]), kc_want), "k cache"
    assert np.array_equal(bf16_bits(case["v_cache"]), vc_want), "v cache"
    assert_parity(to_f64(out), want, what=what)
    return out


# (workload, grids): heads Hq / Hkv, d_qk, d_v, window, rel_extent, new tokens
# per sequence, cached tokens per sequence
CASES = {
    # cached prefixes that are not multiples of 128: the diagonal of a query
    # tile crosses a block boundary, so two key tiles are partly masked
    "offsets": (I.PrefillWorkload("wo", 12, 2, 128, 128, 0, 512, (300, 77, 129), (100, 0, 333)),
                [1, 5, 148]),
    # a window that is not a multiple of 128 and shorter than a tile's span
    "window_300": (I.PrefillWorkload("ww", 8, 1, 128, 128, 300, 256, (520, 260), (700, 40)),
                   [2, 148]),
    # W = E = 1024 with g = 6, as the full-size chunked prefill
    "gqa6_w1024": (I.PrefillWorkload("wg", 12, 2, 128, 128, 1024, 1024, (384, 190),
                                     (1100, 2000)), [3, 148]),
    # rel_extent (8) far below the box width (168 distances) and the window
    "extent_8": (I.PrefillWorkload("we", 4, 2, 128, 128, 200, 8, (150, 70), (10, 260)),
                 [1, 148]),
    # window 1: every row sees only its own key
    "window1": (I.PrefillWorkload("w1", 4, 2, 128, 128, 1, 8, (200,), (10,)), [2]),
    # ragged lengths around the tile and block sizes, many sequences
    "ragged_many": (I.PrefillWorkload("wr", 8, 8, 128, 128, 256, 512,
                                      (1, 63, 64, 65, 127, 128, 129, 200),
                                      (0, 1, 127, 128, 129, 0, 64, 1000)), [1, 7, 148]),
    # global attention over a long prefix: many key tiles per item
    "global_long": (I.PrefillWorkload("wl", 8, 2, 128, 128, 0, 2048, (256, 130), (3000, 1500)),
                    [4, 148]),
}

PARAMS = [(name, ctas) for name in sorted(CASES) for ctas in CASES[name][1]]


@pytest.mark.parametrize("name,num_ctas", PARAMS)
def test_wide_prefill(name, num_ctas):
    case = I.make_prefill(bf16_rel(CASES[name][0]), DEV, seed_data=31, seed_layout=32)
    check(case, num_ctas, what=f"{name} ctas={num_ctas}")


@pytest.mark.parametrize("num_ctas", [3, 148])
def test_wide_prefill_fp32_out(num_ctas):
    case = I.make_prefill(bf16_rel(CASES["offsets"][0]), DEV, seed_data=33, seed_layout=34)
    check(case, num_ctas, what=f"fp32 out ctas={num_ctas}", out_dtype=torch.float32)


def test_wide_fp32_out_rounds_to_the_bf16_out():
    case = I.make_prefill(bf16_rel(CASES["gqa6_w1024"][0]), DEV, seed_data=35)
    k0, v0 = case["k_cache"].clone(), case["v_cache"].clone()
    o32 = run(case, 148, torch.float32)
    case["k_cache"].copy_(k0)
    case["v_cache"].copy_(v0)
    o16 = run(case, 148, torch.bfloat16)
    assert torch.equal(o32.to(torch.bfloat16).view(torch.int16), o16.view(torch.int16))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_wide_prefill_sink_gate_and_factor(out_dtype):
    case = I.make_prefill(bf16_rel(CASES["ragged_many"][0]), DEV, seed_data=36, seed_layout=37)
    T, Hq = case["q"].shape[:2]
    g = torch.Generator(device="cpu")
    g.manual_seed(38)
    case["sink"] = (torch.randn((T, Hq), generator=g) * 2).to(DEV)
    case["gate"] = (torch.randn((T, Hq), generator=g) * 2).to(DEV)
    case["logit_scale"] = (0.25 + 3.75 * torch.rand((T,), generator=g)).to(DEV)
    check(case, 5, what=f"sink gate factor out={out_dtype}", out_dtype=out_dtype,
          sink=case["sink"], gate=case["gate"], logit_scale=case["logit_scale"])


def test_wide_matches_two_heads_kernel_on_fp32_rel_values():
    """The same bf16-valued rel given as fp32 runs the two-heads kernel (64-key
    tiles); both outputs must agree with the oracle and closely with each
    other."""
    wl = CASES["gqa6_w1024"][0]
    case = I.make_prefill(bf16_rel(wl), DEV, seed_data=39)
    k0, v0 = case["k_cache"].clone(), case["v_cache"].clone()
    wide = run(case, 148)
    case["k_cache"].copy_(k0)
    case["v_cache"].copy_(v0)
    pair = run(dict(case, rel=case["rel"].float()), 148)
    d = (wide.float() - pair.float()).abs().max().item()
    assert d <= 2e-2


def test_wide_prefill_two_ring_slots_many_sequences():
    """With 60 sequences the per-sequence arrays leave room for two ring slots
    instead of three: 60 sequences of ragged lengths (partial and full query
    tiles) run that instantiation, on a forced grid and on 7 CTAs."""
    rng = np.random.default_rng(77)
    new = tuple(int(x) for x in rng.integers(100, 300, size=60))
    ctx = tuple(int(x) for x in rng.integers(0, 400, size=60))
    wl = I.PrefillWorkload("w60", 4, 2, 128, 128, 256, 256, new, ctx)
    for ctas in (148, 7):
        case = I.make_prefill(bf16_rel(wl), DEV, seed_data=41, seed_layout=42)
        check(case, ctas, what=f"60 sequences ctas={ctas}")
