"""GPU decode with a bf16 rel input and with an fp32 output, vs the oracle.

relattn_decode_ex takes rel as fp32 or bf16 and writes out as bf16 or fp32.
The oracle reads a bf16 rel as its exact value (uint16 bit patterns), so the
same tolerance applies; an fp32 output rounded to bf16 must equal the bf16
output bit for bit (the same arithmetic, a different store).
"""

import numpy as np
import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from tests.parity import assert_parity, oracle_decode, oracle_decode_multi, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def ws_for(case, num_ctas=0):
    q = case["q"]
    Hq = q.shape[-2]
    dims = R.Dims(q.shape[0], Hq, case["block_table"].shape[1], 0, 0, num_ctas)
    return R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                                case["v_cache"])), DEV)


def run(case, out_dtype, num_ctas=0):
    ws = ws_for(case, num_ctas)
    fn = R.relattn_decode_multi if case["q"].dim() == 4 else R.relattn_decode
    out = fn(case["q"], case["rel"], case["k_cache"], case["v_cache"], case["block_table"],
             case["seq_lens"], case["window"], case["rel_extent"], workspace=ws,
             num_ctas=num_ctas, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    assert out.dtype == out_dtype
    return out


CASES = {
    "local_w512": I.variant(I.WORKLOADS["local_decode"], batch=5, lengths=("uniform", 1, 3000),
                            pool_blocks=0, max_blocks_per_seq=0),
    "global_e1024": I.variant(I.WORKLOADS["global_decode_b8"], batch=3,
                              lengths=("uniform", 1, 6000)),
    "diffhead_dv64": I.variant(I.WORKLOADS["diffhead_decode"], batch=4,
                               lengths=("loguniform", 64, 5000)),
    "gqa6_w100_e64": I.DecodeWorkload("gqa6", 4, 12, 2, 128, 128, 100, 64, ("uniform", 1, 1500)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bf16_rel(name):
    case = I.make_decode(CASES[name], DEV, seed_data=61)
    case["rel"] = case["rel"].to(torch.bfloat16)
    out = run(case, torch.bfloat16)
    assert_parity(to_f64(out), oracle_decode(case), what=f"bf16 rel {name}")


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("rel_dtype", [torch.float32, torch.bfloat16])
def test_fp32_out(name, rel_dtype):
    case = I.make_decode(CASES[name], DEV, seed_data=62)
    case["rel"] = case["rel"].to(rel_dtype)
    o32 = run(case, torch.float32)
    assert_parity(to_f64(o32), oracle_decode(case), what=f"fp32 out {name}")
    o16 = run(case, torch.bfloat16)
    assert torch.equal(o32.to(torch.bfloat16).view(torch.int16), o16.view(torch.int16))


@pytest.mark.parametrize("num_ctas", [1, 7, 152, 1000])
def test_typed_decode_any_split(num_ctas):
    """Split pieces and their combine with both element types changed."""
    wl = I.DecodeWorkload("split", 6, 16, 4, 128, 128, 0, 256, ("uniform", 1, 4000))
    case = I.make_decode(wl, DEV, seed_data=63)
    case["rel"] = case["rel"].to(torch.bfloat16)
    out = run(case, torch.float32, num_ctas=num_ctas)
    assert_parity(to_f64(out), oracle_decode(case), what=f"num_ctas={num_ctas}")


@pytest.mark.parametrize("k,W", [(4, 0), (8, 512), (9, 100)])
def test_typed_multi_token(k, W):
    wl = I.DecodeWorkload("multi", 5, 16, 4, 128, 128, W, 512, ("uniform", k, 3000),
                          query_tokens=k)
    case = I.make_decode(wl, DEV, seed_data=64 + k)
    case["rel"] = case["rel"].to(torch.bfloat16)
    out = run(case, torch.float32)
    assert_parity(to_f64(out), oracle_decode_multi(case), what=f"multi k={k} W={W}")


EDGE_LENS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025]


@pytest.mark.parametrize("window,extent", [(0, 1024), (128, 64), (1, 8), (129, 256)])
def test_bf16_rel_edge_lengths(window, extent):
    wl = I.DecodeWorkload("edge", len(EDGE_LENS), 32, 8, 128, 128, window, extent,
                          ("list", EDGE_LENS))
    case = I.make_decode(wl, DEV, seed_data=65)
    case["rel"] = case["rel"].to(torch.bfloat16)
    out = run(case, torch.bfloat16)
    assert_parity(to_f64(out), oracle_decode(case), what=f"edge W={window} E={extent}")


def test_bf16_rel_extent_must_be_a_multiple_of_8():
    wl = I.DecodeWorkload("e12", 2, 8, 2, 128, 128, 0, 12, ("uniform", 1, 300))
    case = I.make_decode(wl, DEV, seed_data=66)
    with pytest.raises(R.RelattnError) as e:
        run(dict(case, rel=case["rel"].to(torch.bfloat16)), torch.bfloat16)
    assert e.value.code == R.ERR_UNSUPPORTED
    run(case, torch.float32)  # the fp32 rel of the same extent is fine


def test_bf16_rel_full_size_local_sampled():
    case = I.make_decode(I.WORKLOADS["local_decode"], DEV, seed_data=0)
    case["rel"] = case["rel"].to(torch.bfloat16)
    out = run(case, torch.float32)
    bs, hs = [0, 7, 15], [0, 5, 17, 31]
    want = oracle_decode(case, batch=bs, heads=hs)
    got = to_f64(out)
    assert_parity(got[np.ix_(bs, hs)], want[np.ix_(bs, hs)], what="local bf16 rel")
