"""Boundary behaviour on the GPU: bad inputs give status codes, never faults.

Block ids outside the pool and lengths beyond the block table are caught by
the kernels' own bounds checks: the affected tile or sequence is skipped and
a status bit is set.  Nothing here can fault the GPU: every access the
kernels make with these inputs is checked before it happens.
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


def small_case(seed=0):
    wl = I.DecodeWorkload("b", 4, 8, 2, 128, 128, 0, 64, ("list", [300, 129, 1000, 50]))
    return I.make_decode(wl, DEV, seed_data=seed)


def call(case, ws, **kw):
    return R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                            case["block_table"], case["seq_lens"], case["window"],
                            case["rel_extent"], workspace=ws, **kw)


def workspace(case):
    dims = R.decode_dims(case["q"], case["block_table"])
    return R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                               case["v_cache"])), DEV)


def test_bad_block_id_sets_status_and_spares_other_sequences():
    case = small_case()
    want = oracle_decode(case)
    nb = case["k_cache"].shape[0]
    case["block_table"][2, 3] = nb + 5   # a block sequence 2 needs
    ws = workspace(case)
    out = call(case, ws)
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_BAD_BLOCK_ID
    got = to_f64(out)
    for b in (0, 1, 3):
        assert_parity(got[b], want[b], what=f"seq {b}")
    R.clear_status(ws)
    assert R.read_status(ws) == 0


def test_negative_block_id_sets_status():
    case = small_case(1)
    case["block_table"][0, 0] = -7
    ws = workspace(case)
    call(case, ws)
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_BAD_BLOCK_ID


@pytest.mark.parametrize("bad_len", [0, -3, 10**6])
def test_bad_length_sets_status_and_zero_output(bad_len):
    case = small_case(2)
    want = oracle_decode(case)
    case["seq_lens"][1] = bad_len
    ws = workspace(case)
    out = call(case, ws)
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_BAD_LENGTH
    assert torch.all(out[1] == 0)
    got = to_f64(out)
    for b in (0, 2, 3):
        assert_parity(got[b], want[b], what=f"seq {b}")


def test_host_side_errors_are_return_codes():
    case = small_case(3)
    ws = workspace(case)
    with pytest.raises(R.RelattnError) as e:
        R.relattn_decode(case["q"], case["rel"][:, :, :62].contiguous(), case["k_cache"],
                         case["v_cache"], case["block_table"], case["seq_lens"], 0, 62,
                         workspace=ws)
    assert e.value.code == R.ERR_UNSUPPORTED
    with pytest.raises(R.RelattnError) as e:
        call(case, ws[:256])
    assert e.value.code == R.ERR_WORKSPACE
    # misaligned q (offset by one element)
    buf = torch.empty(case["q"].numel() + 8, dtype=torch.bfloat16, device=DEV)
    q_mis = buf[1:1 + case["q"].numel()].view(case["q"].shape)
    with pytest.raises(R.RelattnError) as e:
        R.relattn_decode(q_mis, case["rel"], case["k_cache"], case["v_cache"],
                         case["block_table"], case["seq_lens"], 0, 64, workspace=ws)
    assert e.value.code == R.ERR_INVALID_ARG
    # nothing was launched by the failed calls; the workspace is still clean
    assert R.read_status(ws) == 0


def test_prefill_bad_block_and_length():
    wl = I.PrefillWorkload("pb", 4, 1, 128, 128, 0, 64, (100, 100), (0, 50))
    case = I.make_prefill(wl, DEV)
    case["block_table"][1, 0] = 10**6
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                      case["k_cache"], case["v_cache"], case["block_table"], case["ctx_lens"],
                      0, 64, case["max_q_len"], workspace=ws)
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_BAD_BLOCK_ID
    R.clear_status(ws)
    case["ctx_lens"][0] = 10**6
    out = R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                            case["k_cache"], case["v_cache"], case["block_table"],
                            case["ctx_lens"], 0, 64, case["max_q_len"], workspace=ws)
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_BAD_LENGTH
    assert torch.all(out[:100] == 0)
