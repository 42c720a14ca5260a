"""GPU chunked prefill with a bf16 rel input and with an fp32 output.

relattn_prefill_ex reads rel as fp32 or bf16 and writes out as bf16 or fp32.
The oracle reads a bf16 rel as its exact value; an fp32 output rounded to
bf16 equals the bf16 output bit for bit (the same arithmetic); the cache
write is unchanged and stays bit-exact.
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


def run(case, out_dtype, num_ctas=0):
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"],
                          num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out = R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                            case["k_cache"], case["v_cache"], case["block_table"],
                            case["ctx_lens"], case["window"], case["rel_extent"],
                            case["max_q_len"], workspace=ws, out_dtype=out_dtype,
                            num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    assert out.dtype == out_dtype
    return out


def check(case, out_dtype, rows=None, what="", num_ctas=0):
    cache0 = snapshot_cache(case)
    want, kc_want, vc_want = oracle_prefill(case, rows=rows, cache=cache0)
    out = run(case, out_dtype, num_ctas)
    assert np.array_equal(bf16_bits(case["k_cache"]), kc_want), "k cache"
    assert np.array_equal(bf16_bits(case["v_cache"]), vc_want), "v cache"
    sel = slice(None) if rows is None else list(rows)
    assert_parity(to_f64(out)[sel], want[sel], what=what)
    return out


SMALL = {
    "prefix_window": I.PrefillWorkload("pw", 12, 2, 128, 128, 100, 64, (200, 77), (300, 0)),
    "global_dv64": I.PrefillWorkload("g64", 8, 2, 128, 64, 0, 256, (130, 1, 64), (0, 500, 129)),
    "gqa6_w1024": I.PrefillWorkload("g6", 12, 2, 128, 128, 1024, 1024, (300, 190), (1100, 2000)),
    "extent_lt_window": I.PrefillWorkload("el", 4, 1, 128, 128, 700, 128, (400,), (333,)),
    "window1": I.PrefillWorkload("w1", 4, 2, 128, 128, 1, 8, (70,), (10,)),
    "ragged_many": I.PrefillWorkload("rm", 8, 8, 128, 128, 256, 512,
                                     (1, 63, 64, 65, 127, 128, 129, 200),
                                     (0, 1, 127, 128, 129, 0, 64, 1000)),
}


@pytest.mark.parametrize("num_ctas", [0, 148])  # 148: two heads per work item (forced grid)
@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("rel_dtype,out_dtype", [(torch.bfloat16, torch.bfloat16),
                                                 (torch.float32, torch.float32),
                                                 (torch.bfloat16, torch.float32)])
def test_typed_prefill_small(name, rel_dtype, out_dtype, num_ctas):
    case = I.make_prefill(SMALL[name], DEV, seed_data=7, seed_layout=8)
    case["rel"] = case["rel"].to(rel_dtype)
    check(case, out_dtype, what=f"{name} rel={rel_dtype} out={out_dtype}", num_ctas=num_ctas)


@pytest.mark.parametrize("rel_dtype", [torch.float32, torch.bfloat16])
def test_fp32_out_rounds_to_the_bf16_out(rel_dtype):
    wl = SMALL["gqa6_w1024"]
    case = I.make_prefill(wl, DEV, seed_data=9)
    case["rel"] = case["rel"].to(rel_dtype)
    k0, v0 = case["k_cache"].clone(), case["v_cache"].clone()
    o32 = run(case, torch.float32)
    case["k_cache"].copy_(k0)
    case["v_cache"].copy_(v0)
    o16 = run(case, torch.bfloat16)
    assert torch.equal(o32.to(torch.bfloat16).view(torch.int16), o16.view(torch.int16))


def test_bf16_rel_extent_must_be_a_multiple_of_8():
    wl = I.PrefillWorkload("e12", 4, 1, 128, 128, 0, 12, (100,), (0,))
    case = I.make_prefill(wl, DEV, seed_data=10)
    with pytest.raises(R.RelattnError) as e:
        run(dict(case, rel=case["rel"].to(torch.bfloat16)), torch.bfloat16)
    assert e.value.code == R.ERR_UNSUPPORTED


def test_bf16_rel_full_size_sampled():
    """The 4 x 8192-after-24576 chunked prefill (48/8 heads, W = E = 1024)
    with a bf16 rel, in the bench's launch configuration, on sampled rows."""
    case = I.make_prefill(I.WORKLOADS["chunked_prefill"], DEV, seed_data=0)
    case["rel"] = case["rel"].to(torch.bfloat16)
    T = case["num_tokens"]
    rows = sorted({0, 1, 127, 128, 8191, 8192, 16000, 24576 - 1, 24576, T - 129, T - 1})
    check(case, torch.float32, rows=rows, what="chunked prefill bf16 rel")
