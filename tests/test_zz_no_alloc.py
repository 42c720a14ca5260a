"""Decode through the library-owned scratch array, compared with the
workspace entry point.

relattn_decode_noalloc is for callers that cannot allocate device memory (a
host that owns every buffer and hands the library only inputs and outputs).
It runs the same kernel as relattn_decode, on the same grid, with the same
fixed merge order, so its output must equal the workspace call's bit for
bit; the workspace call itself is checked against the float64 oracle.

Collected last on purpose, so that a run that stops at the first failure has
run every other test before this one; it must pass both alone in a fresh
process and after the other tests.
"""

import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from tests.parity import assert_parity, oracle_decode, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def with_workspace(case, num_ctas):
    dims = R.decode_dims(case["q"], case["block_table"], num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                           case["block_table"], case["seq_lens"], case["window"],
                           case["rel_extent"], workspace=ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    return out


def without_workspace(case, out, num_ctas):
    return R.relattn_decode_noalloc(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                                    case["block_table"], case["seq_lens"], case["window"],
                                    case["rel_extent"], out, num_ctas=num_ctas)


@pytest.mark.parametrize("num_ctas", [0, 37])
def test_noalloc_decode_matches_workspace_decode_twice(num_ctas):
    wl = I.variant(I.WORKLOADS["global_decode_b8"], batch=4, lengths=("uniform", 1, 6000))
    case = I.make_decode(wl, DEV, seed_data=13)
    want = with_workspace(case, num_ctas)
    assert_parity(to_f64(want), oracle_decode(case), what="workspace decode vs oracle")
    outs = [torch.empty_like(case["q"][..., :case["v_cache"].shape[-1]]) for _ in range(2)]
    for o in outs:                       # two calls in a row, same stream
        without_workspace(case, o, num_ctas)
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, want), f"noalloc call {i} differs from the workspace call"


def test_noalloc_rejects_sizes_beyond_its_array():
    """Split state larger than the array is refused before anything is enqueued."""
    wl = I.DecodeWorkload("big_split", 2, 32, 2, 128, 128, 0, 64, ("list", [300, 500]))
    case = I.make_decode(wl, DEV, seed_data=1)
    out = torch.zeros(2, 32, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(R.RelattnError) as err:
        without_workspace(case, out, num_ctas=5000)
    assert err.value.code == R.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_noalloc_status_reports_a_bad_block_id_then_clears():
    """The call's device status bits stay in the array until the next call:
    a block id outside the pool sets RELATTN_DEV_BAD_BLOCK_ID, and the next
    clean call starts from zero."""
    wl = I.variant(I.WORKLOADS["global_decode_b8"], batch=2, lengths=("uniform", 200, 900))
    case = I.make_decode(wl, DEV, seed_data=17)
    out = torch.empty_like(case["q"][..., :case["v_cache"].shape[-1]])
    bad = dict(case, block_table=case["block_table"].clone())
    bad["block_table"][1, 0] = case["k_cache"].shape[0] + 5  # outside the pool
    without_workspace(bad, out, 0)
    assert R.noalloc_status(DEV) & R.DEV_BAD_BLOCK_ID
    without_workspace(case, out, 0)
    assert R.noalloc_status(DEV) == 0
