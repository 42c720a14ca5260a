"""GPU decode over an FP8 (e4m3) KV cache with per-tensor scales, vs the oracle.

The caches are quantised to e4m3 with one scale each (the input generator);
the oracle reads the e4m3 patterns exactly and applies the scales, so the
same tolerance as the bf16 cache applies.  The kernels widen K and V to f16
in registers and run their MMAs in f16: the one-token kernel and the general
one (several query tokens, or g > 8).
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


def run(case, num_ctas=0, out_dtype=torch.bfloat16):
    q = case["q"]
    dims = R.Dims(q.shape[0], q.shape[-2], case["block_table"].shape[1], 0, 0, num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    fn = R.relattn_decode_multi if q.dim() == 4 else R.relattn_decode
    out = fn(q, case["rel"], case["k_cache"], case["v_cache"], case["block_table"],
             case["seq_lens"], case["window"], case["rel_extent"], workspace=ws,
             num_ctas=num_ctas, out_dtype=out_dtype, sink=case.get("sink"),
             gate=case.get("gate"), k_scale=case.get("k_scale"), v_scale=case.get("v_scale"),
             logit_scale=case.get("logit_scale"))
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    return out


def fp8(wl, **kw):
    return I.variant(wl, kv_dtype="fp8", **kw)


SMALL = {
    "local_w512": fp8(I.WORKLOADS["local_decode"], batch=5, lengths=("uniform", 1, 3000),
                      pool_blocks=0, max_blocks_per_seq=0),
    "global_e1024": fp8(I.WORKLOADS["global_decode_b8"], batch=3, lengths=("uniform", 1, 6000)),
    "mha_g1": fp8(I.DecodeWorkload("mha_g1", 3, 4, 4, 128, 128, 0, 64, ("uniform", 1, 900))),
    "gqa6_w100_e64": fp8(I.DecodeWorkload("gqa6", 4, 12, 2, 128, 128, 100, 64,
                                          ("uniform", 1, 1500))),
    "gqa8": fp8(I.DecodeWorkload("gqa8", 3, 64, 8, 128, 128, 0, 1024,
                                 ("loguniform", 64, 5000))),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_fp8_decode_small_configs(name):
    case = I.make_decode(SMALL[name], DEV, seed_data=111, seed_layout=112)
    assert case["k_cache"].dtype == torch.float8_e4m3fn
    assert_parity(to_f64(run(case)), oracle_decode(case), what=name)


EDGE_LENS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025]


@pytest.mark.parametrize("window,extent", [(0, 1024), (512, 512), (128, 64), (1, 4)])
def test_fp8_decode_edge_lengths(window, extent):
    wl = fp8(I.DecodeWorkload("edge", len(EDGE_LENS), 32, 8, 128, 128, window, extent,
                              ("list", EDGE_LENS)))
    case = I.make_decode(wl, DEV, seed_data=113)
    assert_parity(to_f64(run(case)), oracle_decode(case), what=f"W={window} E={extent}")


@pytest.mark.parametrize("num_ctas", [1, 7, 152, 1000])
def test_fp8_decode_any_split(num_ctas):
    wl = fp8(I.DecodeWorkload("split", 6, 16, 4, 128, 128, 0, 256, ("uniform", 1, 4000)))
    case = I.make_decode(wl, DEV, seed_data=114)
    assert_parity(to_f64(run(case, num_ctas=num_ctas)), oracle_decode(case),
                  what=f"num_ctas={num_ctas}")


def test_fp8_with_bf16_rel_fp32_out_sink_and_gate():
    wl = fp8(SMALL["local_w512"], rel_dtype="bf16")
    case = I.make_decode(wl, DEV, seed_data=115)
    B, Hq = case["q"].shape[:2]
    g = torch.Generator(device="cpu")
    g.manual_seed(116)
    case["sink"] = torch.randn((B, Hq), generator=g).to(DEV)
    case["gate"] = torch.randn((B, Hq), generator=g).to(DEV)
    out = run(case, out_dtype=torch.float32)
    assert_parity(to_f64(out), oracle_decode(case), what="fp8 + bf16 rel + sink/gate")


def test_fp8_decode_full_size_global_b8_sampled():
    case = I.make_decode(fp8(I.WORKLOADS["global_decode_b8"]), DEV, seed_data=0)
    out = run(case)
    bs, hs = [0, 3, 7], [0, 9, 31]
    want = oracle_decode(case, batch=bs, heads=hs)
    assert_parity(to_f64(out)[np.ix_(bs, hs)], want[np.ix_(bs, hs)], what="global b8 fp8")


def test_fp8_decode_dv64_is_refused():
    wl = fp8(I.DecodeWorkload("d", 2, 16, 4, 128, 64, 0, 64, ("uniform", 1, 300)))
    case = I.make_decode(wl, DEV, seed_data=117)
    with pytest.raises(R.RelattnError) as e:
        run(case)
    assert e.value.code == R.ERR_UNSUPPORTED


# ---- the general kernel over an e4m3 cache: several query tokens, or g > 8

@pytest.mark.parametrize("k", [2, 3, 4, 8, 9, 16])
def test_fp8_multi_token_decode(k):
    """Verification over a global layer's e4m3 cache (g = 4: up to 4 tokens
    per chunk, ragged last chunks beyond)."""
    wl = fp8(I.DecodeWorkload("mt", 4, 32, 8, 128, 128, 0, 1024, ("uniform", 16, 5000),
                              query_tokens=k))
    case = I.make_decode(wl, DEV, seed_data=150 + k)
    assert_parity(to_f64(run(case)), oracle_decode_multi(case), what=f"fp8 k={k}")


@pytest.mark.parametrize("g,k", [(1, 5), (3, 4), (6, 2), (8, 2), (16, 1), (16, 3)])
def test_fp8_general_kernel_packings(g, k):
    Hkv = 2
    wl = fp8(I.DecodeWorkload("pk", 3, g * Hkv, Hkv, 128, 128, 300, 256, ("uniform", 16, 2500),
                              query_tokens=k))
    case = I.make_decode(wl, DEV, seed_data=160 + g)
    assert_parity(to_f64(run(case)), oracle_decode_multi(case), what=f"fp8 g={g} k={k}")


@pytest.mark.parametrize("window,extent", [(0, 1024), (512, 512), (129, 64), (1, 4)])
def test_fp8_multi_token_edge_lengths(window, extent):
    lens = [8, 9, 63, 64, 65, 71, 72, 127, 128, 129, 135, 136, 255, 256, 257, 1031]
    wl = fp8(I.DecodeWorkload("edge", len(lens), 32, 8, 128, 128, window, extent,
                              ("list", lens), query_tokens=8))
    case = I.make_decode(wl, DEV, seed_data=170)
    assert_parity(to_f64(run(case)), oracle_decode_multi(case), what=f"W={window} E={extent}")


@pytest.mark.parametrize("num_ctas", [1, 7, 152, 1000])
def test_fp8_multi_token_any_split(num_ctas):
    wl = fp8(I.DecodeWorkload("split", 5, 16, 4, 128, 128, 0, 256, ("uniform", 8, 4000),
                              query_tokens=4))
    case = I.make_decode(wl, DEV, seed_data=171)
    assert_parity(to_f64(run(case, num_ctas=num_ctas)), oracle_decode_multi(case),
                  what=f"num_ctas={num_ctas}")


def test_fp8_multi_token_with_every_option():
    """bf16 rel, fp32 out, sink, gate and log-position factors together."""
    wl = fp8(I.DecodeWorkload("opt", 4, 32, 8, 128, 128, 0, 1024, ("uniform", 16, 3000),
                              query_tokens=4, rel_dtype="bf16"))
    case = I.make_decode(wl, DEV, seed_data=172)
    g = torch.Generator(device="cpu")
    g.manual_seed(173)
    case["sink"] = torch.randn((4, 4, 32), generator=g).to(DEV)
    case["gate"] = torch.randn((4, 4, 32), generator=g).to(DEV)
    case["logit_scale"] = (0.5 + 2 * torch.rand((4, 4), generator=g)).to(DEV)
    out = run(case, out_dtype=torch.float32)
    assert_parity(to_f64(out), oracle_decode_multi(case), what="fp8 multi, every option")


def test_fp8_multi_token_full_size_global_b8_sampled():
    """Four tokens per sequence over the full B=8, 32K global workload."""
    case = I.make_decode(fp8(I.variant(I.WORKLOADS["global_decode_b8"], query_tokens=4)), DEV,
                         seed_data=174)
    out = run(case)
    bs, ts, hs = [0, 5], [0, 3], [1, 30]
    want = oracle_decode_multi(case, batch=bs, tokens=ts, heads=hs)
    got = to_f64(out)
    assert_parity(got[np.ix_(bs, ts, hs)], want[np.ix_(bs, ts, hs)], what="global b8 k=4 fp8")


def test_fp8_one_token_through_the_general_kernel_matches_the_oracle():
    """k = 1 with g = 16 takes the general kernel (16 rows)."""
    wl = fp8(I.DecodeWorkload("g16", 3, 32, 2, 128, 128, 0, 512, ("uniform", 1, 4000)))
    case = I.make_decode(wl, DEV, seed_data=175)
    assert_parity(to_f64(run(case)), oracle_decode(case), what="fp8 g=16 k=1")


def test_prefill_refuses_an_e4m3_cache_with_dv64():
    """e4m3 caches need d_v = 128, in prefill as in decode: relattn_prefill_ex
    returns UNSUPPORTED otherwise (called through the C ABI)."""
    import ctypes
    wl = I.PrefillWorkload("p64", 4, 1, 128, 64, 64, 64, (130,), (0,), kv_dtype="fp8")
    p = I.make_prefill(wl, DEV)
    dims = R.prefill_dims(p["q"], p["block_table"], p["ctx_lens"], p["max_q_len"])
    cache = R.cache_desc(p["k_cache"], p["v_cache"])
    ws = R.new_workspace(R.workspace_size(dims, cache), DEV)
    out = torch.empty((p["num_tokens"], 4, 64), dtype=torch.bfloat16, device=DEV)
    opt = R.Options(R.DTYPE_F32, R.DTYPE_BF16, None, None, R.DTYPE_E4M3, p["k_scale"],
                    p["v_scale"], None)
    rc = R.lib().relattn_prefill_ex(
        p["q"].data_ptr(), p["k"].data_ptr(), p["v"].data_ptr(), p["rel"].data_ptr(),
        ctypes.byref(opt), p["cu_seqlens"].data_ptr(), ctypes.byref(cache),
        p["block_table"].data_ptr(), p["ctx_lens"].data_ptr(), p["window"], p["rel_extent"],
        ctypes.byref(dims), out.data_ptr(), ws.data_ptr(), ws.numel(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == R.ERR_UNSUPPORTED
