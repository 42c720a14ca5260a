"""Failure detection on the GPU without a fault: a bounded wait that cannot
complete gives up, records RELATTN_DEV_WAIT_TIMEOUT in the status word, and
the context stays usable for the next call."""

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
