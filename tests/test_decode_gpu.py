"""GPU decode vs the float64 oracle, through the C ABI."""

import numpy as np
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


def run_and_check(case, batch=None, heads=None, num_ctas=0, what=""):
    ws = R.new_workspace(R.workspace_size(R.decode_dims(case["q"], case["block_table"],
                                                        num_ctas),
                                          R.cache_desc(case["k_cache"], case["v_cache"])),
                         DEV)
    out = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                           case["block_table"], case["seq_lens"], case["window"],
                           case["rel_extent"], workspace=ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    want = oracle_decode(case, batch=batch, heads=heads)
    got = to_f64(out)
    bs = list(range(got.shape[0])) if batch is None else list(batch)
    hs = list(range(got.shape[1])) if heads is None else list(heads)
    return assert_parity(got[np.ix_(bs, hs)], want[np.ix_(bs, hs)], what=what), ws


SMALL = {
    "local_w512": I.variant(I.WORKLOADS["local_decode"], batch=5,
                            lengths=("uniform", 1, 3000), pool_blocks=0,
                            max_blocks_per_seq=0),
    "global_e1024": I.variant(I.WORKLOADS["global_decode_b8"], batch=3,
                              lengths=("uniform", 1, 6000)),
    "diffhead_dv64": I.variant(I.WORKLOADS["diffhead_decode"], batch=4,
                               lengths=("loguniform", 64, 5000)),
    "mha_g1": I.DecodeWorkload("mha_g1", 3, 4, 4, 128, 128, 0, 64, ("uniform", 1, 900)),
    "gqa6_w100_e64": I.DecodeWorkload("gqa6", 4, 12, 2, 128, 128, 100, 64,
                                      ("uniform", 1, 1500)),
    "gqa16": I.DecodeWorkload("gqa16", 2, 32, 2, 128, 64, 300, 512, ("uniform", 200, 2500)),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_decode_small_configs(name):
    case = I.make_decode(SMALL[name], DEV, seed_data=3, seed_layout=4)
    run_and_check(case, what=name)


EDGE_LENS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025]


@pytest.mark.parametrize("window,extent", [(0, 1024), (512, 512), (128, 64), (1, 4),
                                           (129, 256)])
def test_decode_edge_lengths(window, extent):
    wl = I.DecodeWorkload("edge", len(EDGE_LENS), 32, 8, 128, 128, window, extent,
                          ("list", EDGE_LENS))
    case = I.make_decode(wl, DEV, seed_data=5)
    run_and_check(case, what=f"edge W={window} E={extent}")


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 1000, 5000])
def test_decode_any_split_matches(num_ctas):
    """Every cut of the key work into CTA ranges gives the same answer."""
    wl = I.DecodeWorkload("split", 6, 16, 4, 128, 128, 0, 256, ("uniform", 1, 4000))
    case = I.make_decode(wl, DEV, seed_data=7)
    run_and_check(case, num_ctas=num_ctas, what=f"num_ctas={num_ctas}")


def test_decode_is_deterministic_and_reusable_workspace():
    wl = I.variant(I.WORKLOADS["local_decode"], batch=4, lengths=("uniform", 100, 3000),
                   pool_blocks=0, max_blocks_per_seq=0)
    case = I.make_decode(wl, DEV, seed_data=9)
    dims = R.decode_dims(case["q"], case["block_table"], 37)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    outs = [R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                             case["block_table"], case["seq_lens"], case["window"],
                             case["rel_extent"], workspace=ws, num_ctas=37)
            for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert R.read_status(ws) == 0


def test_decode_graph_capture_replay_is_bit_identical():
    """Capture and replay equal eager exactly ("Inkling on Two DGX Sparks",
    section "Wall 1": capture/replay regression with max difference 0)."""
    wl = I.variant(I.WORKLOADS["global_decode_b8"], batch=4, lengths=("uniform", 10, 5000))
    case = I.make_decode(wl, DEV, seed_data=11)
    dims = R.decode_dims(case["q"], case["block_table"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out_eager = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                                 case["block_table"], case["seq_lens"], case["window"],
                                 case["rel_extent"], workspace=ws)
    out_graph = torch.empty_like(out_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                             case["block_table"], case["seq_lens"], case["window"],
                             case["rel_extent"], out=out_graph, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_graph, out_eager)
    # new inputs through the same graph follow the data
    case["q"].copy_(torch.randn_like(case["q"], dtype=torch.float32).to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    want = oracle_decode(case)
    assert_parity(to_f64(out_graph), want, what="graph replay with new q")


FULL = ["local_decode", "global_decode_b1", "global_decode_b8", "diffhead_decode"]


@pytest.mark.parametrize("name", FULL)
def test_decode_full_size_sampled(name):
    """The bench workloads at full size; the oracle checks sampled rows."""
    wl = I.WORKLOADS[name]
    case = I.make_decode(wl, DEV)
    B, Hq = case["q"].shape[:2]
    rng = np.random.default_rng(0)
    batch = sorted(set([0, B - 1] + list(rng.choice(B, size=min(B, 3), replace=False))))
    heads = sorted(set([0, Hq - 1] + list(rng.choice(Hq, size=4, replace=False))))
    run_and_check(case, batch=batch, heads=heads, what=name)
