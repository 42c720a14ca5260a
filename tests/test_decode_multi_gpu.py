"""GPU multi-token decode (speculative verification) vs the float64 oracle.

k query tokens per sequence, token i at position seq_lens[b] - k + i; the
kernel packs up to 16 / g tokens with the g heads of a KV group into one
tile and cuts larger k into chunks.  Cases cover one chunk, several chunks
with a ragged last chunk, every head ratio's packing, the edge lengths, the
split into CTA ranges, more chunks than one warp plans, invalid lengths and
the full-size verification workload on sampled rows.
"""

import numpy as np
import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from tests.parity import assert_parity, oracle_decode_multi, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def new_ws(case, num_ctas=0):
    dims = R.Dims(case["q"].shape[0], case["q"].shape[2], case["block_table"].shape[1], 0, 0,
                  num_ctas)
    return R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                                case["v_cache"])), DEV)


def run_multi(case, num_ctas=0):
    ws = new_ws(case, num_ctas)
    out = R.relattn_decode_multi(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                                 case["block_table"], case["seq_lens"], case["window"],
                                 case["rel_extent"], workspace=ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    return out, R.read_status(ws)


def check(case, num_ctas=0, batch=None, tokens=None, heads=None, what=""):
    out, st = run_multi(case, num_ctas)
    assert st == 0, f"{what}: device status {st:#x}"
    want = oracle_decode_multi(case, batch=batch, tokens=tokens, heads=heads)
    got = to_f64(out)
    ix = [list(range(n)) if sel is None else list(sel)
          for n, sel in zip(got.shape[:3], (batch, tokens, heads))]
    sub = np.ix_(*ix)
    return assert_parity(got[sub], want[sub], what=what)


def wl(name, B, Hq, Hkv, W, E, k, lengths, dv=128):
    return I.DecodeWorkload(name, B, Hq, Hkv, 128, dv, W, E, lengths, query_tokens=k)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("W,E", [(0, 256), (100, 64)])
def test_multi_gqa4(k, W, E):
    """g = 4: four tokens per tile; k > 4 takes several chunks."""
    case = I.make_decode(wl("gqa4", 5, 16, 4, W, E, k, ("uniform", k, 3000)), DEV,
                         seed_data=20 + k, seed_layout=21 + k)
    check(case, what=f"k={k} W={W} E={E}")


@pytest.mark.parametrize("Hq,Hkv,k,dv", [(4, 4, 16, 128), (4, 4, 7, 64), (12, 2, 5, 128),
                                         (16, 2, 3, 128), (32, 2, 2, 64), (24, 8, 9, 64),
                                         (4, 2, 16, 128), (16, 2, 2, 64)])
def test_multi_head_ratios(Hq, Hkv, k, dv):
    """Every packing: g = 1 (16 tokens a tile), 2, 3, 6, 8, 16 (one token a
    tile); rows split between the consumer groups when more than 16 rows
    share a KV head (g = 2 with 16 tokens, g = 3 with 9, g = 6 with 5, g = 8
    with 3), one 16-row tile otherwise (g = 8 with 2)."""
    case = I.make_decode(wl("ratio", 3, Hq, Hkv, 300, 512, k, ("uniform", k, 2500), dv=dv),
                         DEV, seed_data=30 + Hq + k, seed_layout=31)
    check(case, what=f"Hq={Hq} Hkv={Hkv} k={k} dv={dv}")


EDGE_LENS = [1, 2, 8, 9, 63, 64, 65, 71, 72, 73, 127, 128, 129, 135, 136, 137, 255, 256, 257,
             511, 512, 513, 520, 1023, 1024, 1025, 1032]


@pytest.mark.parametrize("k", [1, 4, 8])
@pytest.mark.parametrize("window,extent", [(0, 1024), (512, 512), (128, 64), (1, 4),
                                           (129, 256)])
def test_multi_edge_lengths(k, window, extent):
    """Lengths around tile and block edges, the shortest legal one (L = k)
    included; windows of 1 (each token sees itself only) and odd sizes."""
    lens = sorted(set([k] + [L for L in EDGE_LENS if L >= k]))
    case = I.make_decode(wl("edge", len(lens), 32, 8, window, extent, k, ("list", lens)), DEV,
                         seed_data=40 + k)
    check(case, what=f"edge k={k} W={window} E={extent}")


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 1000])
def test_multi_any_split_matches(num_ctas):
    case = I.make_decode(wl("split", 6, 16, 4, 0, 256, 6, ("uniform", 6, 4000)), DEV,
                         seed_data=50)
    check(case, num_ctas=num_ctas, what=f"num_ctas={num_ctas}")


def test_multi_many_chunks_block_prologue():
    """More than 32 chunks: the whole block plans the split (not one warp)."""
    case = I.make_decode(wl("many", 40, 32, 8, 512, 512, 8, ("uniform", 8, 5000)), DEV,
                         seed_data=51)
    check(case, what="B=40 k=8")


def test_multi_one_token_equals_decode_bitwise():
    """k = 1 is the one-token decode: the same bits."""
    base = I.DecodeWorkload("k1", 7, 32, 8, 128, 128, 512, 512, ("uniform", 1, 6000))
    case = I.make_decode(base, DEV, seed_data=52)
    ws = R.new_workspace(R.workspace_size(R.decode_dims(case["q"], case["block_table"]),
                                          R.cache_desc(case["k_cache"], case["v_cache"])), DEV)
    one = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                           case["block_table"], case["seq_lens"], case["window"],
                           case["rel_extent"], workspace=ws)
    multi = R.relattn_decode_multi(case["q"][:, None], case["rel"][:, None], case["k_cache"],
                                   case["v_cache"], case["block_table"], case["seq_lens"],
                                   case["window"], case["rel_extent"])
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int16), multi[:, 0].view(torch.int16))


def test_multi_short_sequence_reports_and_zeroes():
    """A sequence shorter than k has no valid query positions: its rows are
    zero and the status says so; the other sequences are unaffected."""
    lens = [700, 3, 1500]
    case = I.make_decode(wl("short", 3, 16, 4, 0, 256, 4, ("list", lens)), DEV, seed_data=53)
    case["seq_lens"][1] = 3
    out, st = run_multi(case)
    assert st & R.DEV_BAD_LENGTH
    assert torch.count_nonzero(out[1]) == 0
    want = oracle_decode_multi(case, batch=[0, 2])
    assert_parity(to_f64(out)[[0, 2]], want[[0, 2]], what="valid rows")


def test_multi_rejects_too_many_tokens():
    case = I.make_decode(wl("k17", 2, 8, 2, 0, 64, 17, ("uniform", 17, 300)), DEV,
                         seed_data=54)
    with pytest.raises(R.RelattnError) as e:
        run_multi(case)
    assert e.value.code == R.ERR_UNSUPPORTED


def test_multi_full_size_verify_sampled():
    """The full verification workload (16 sequences of 4K-32K tokens, 8
    tokens each, 32/8 heads, window 512) in the bench's launch configuration,
    checked on sampled sequences and tokens."""
    case = I.make_decode(I.WORKLOADS["verify_decode"], DEV, seed_data=0)
    check(case, batch=[0, 5, 11, 15], tokens=[0, 3, 4, 7], what="verify_decode")
