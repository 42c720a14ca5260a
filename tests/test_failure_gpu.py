"""Failure detection on the GPU without a fault: a bounded wait that cannot
complete gives up, records RELATTN_DEV_WAIT_TIMEOUT in the status word, and
the context stays usable for the next call."""

import ctypes

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


def test_a_wait_that_cannot_complete_reports_and_the_context_survives():
    ws = R.new_workspace(256, DEV)
    rc = R.lib().relattn_debug_wait_timeout(ws.data_ptr(), ws.numel(),
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == R.OK
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_WAIT_TIMEOUT
    # the next call on the same context computes as usual
    wl = I.variant(I.WORKLOADS["local_decode"], batch=3, lengths=("uniform", 100, 2000),
                   pool_blocks=0, max_blocks_per_seq=0)
    case = I.make_decode(wl, DEV, seed_data=301)
    out = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                           case["block_table"], case["seq_lens"], case["window"],
                           case["rel_extent"])
    torch.cuda.synchronize()
    assert_parity(to_f64(out), oracle_decode(case), what="decode after a timed-out wait")


def test_wait_timeout_hook_checks_its_workspace():
    ws = R.new_workspace(256, DEV)
    assert R.lib().relattn_debug_wait_timeout(ws.data_ptr(), 128, None) == R.ERR_WORKSPACE


@pytest.mark.parametrize("piece", [0, 1])
def test_a_decode_that_gives_up_leaves_its_workspace_ready(piece):
    """Consumers that give up (the test hook stands in for a wait that ran
    out) still complete every split segment's arrival count: the counters are
    zero afterwards and the next decode on the same workspace is correct."""
    wl = I.variant(I.WORKLOADS["global_decode_b8"], batch=2, lengths=("uniform", 3000, 6000))
    case = I.make_decode(wl, DEV, seed_data=302)
    num_ctas = 9  # 16 (sequence, KV head) segments over 9 CTAs: most are split
    cache = R.cache_desc(case["k_cache"], case["v_cache"])
    dims = R.decode_dims(case["q"], case["block_table"], num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, cache), DEV)
    out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device=DEV)
    rc = R.lib().relattn_debug_decode_give_up(
        case["q"].data_ptr(), case["rel"].data_ptr(), ctypes.byref(cache),
        case["block_table"].data_ptr(), case["seq_lens"].data_ptr(), 0, case["rel_extent"],
        ctypes.byref(dims), out.data_ptr(), ws.data_ptr(), ws.numel(), piece,
        torch.cuda.current_stream().cuda_stream)
    assert rc == R.OK
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_WAIT_TIMEOUT
    counters = ws[256:256 + 2 * 16 * 8 * 4].view(torch.int32)
    assert torch.count_nonzero(counters).item() == 0
    again = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                             case["block_table"], case["seq_lens"], case["window"],
                             case["rel_extent"], workspace=ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert_parity(to_f64(again), oracle_decode(case), what="decode after a give-up")
    assert torch.count_nonzero(counters).item() == 0
