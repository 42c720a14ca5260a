"""relattn_cache_write on the GPU vs the oracle: bf16 caches (a bit copy)
and e4m3 caches (quantised with per-tensor scales), bit-exact over the whole
cache, and a decode step that appends its newest token with it first."""

import numpy as np
import pytest
import torch

from oracle import relattn_oracle as O
from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from paged_relative_bias_gb300.inputs import bf16_bits
from tests.parity import assert_parity, host_cache, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


CASES = {
    "prefix_window": I.PrefillWorkload("pw", 12, 2, 128, 128, 100, 64, (200, 77), (300, 0)),
    "ragged_many": I.PrefillWorkload("rm", 8, 8, 128, 128, 256, 512,
                                     (1, 63, 64, 65, 127, 128, 129, 200),
                                     (0, 1, 127, 128, 129, 0, 64, 1000)),
    "dv64": I.PrefillWorkload("g64", 8, 2, 128, 64, 0, 256, (130, 1, 64), (0, 500, 129)),
}


def write(p, k_cache, v_cache, k_scale=None, v_scale=None):
    ws = R.relattn_cache_write(p["k"], p["v"], p["cu_seqlens"], k_cache, v_cache,
                               p["block_table"], p["ctx_lens"], p["max_q_len"],
                               k_scale=k_scale, v_scale=v_scale)
    torch.cuda.synchronize()
    return R.read_status(ws)


def host(p, name):
    return p[name].cpu().numpy()


@pytest.mark.parametrize("name", sorted(CASES))
def test_bf16_cache_write_is_the_oracle_scatter(name):
    p = I.make_prefill(CASES[name], DEV, seed_data=201)
    want_k, want_v = O.kv_cache_write(bf16_bits(p["k_cache"]), bf16_bits(p["v_cache"]),
                                      bf16_bits(p["k"]), bf16_bits(p["v"]), host(p, "cu_seqlens"),
                                      host(p, "ctx_lens"), host(p, "block_table"))
    assert write(p, p["k_cache"], p["v_cache"]) == 0
    assert np.array_equal(bf16_bits(p["k_cache"]), want_k)
    assert np.array_equal(bf16_bits(p["v_cache"]), want_v)


def e4m3_case(name, seed, shrink=1.0):
    """A prefill case whose caches are e4m3 (head-major), with the scales of
    the old cache contents; shrink < 1 makes some new values saturate."""
    p = I.make_prefill(CASES[name], DEV, seed_data=seed)
    k8, ks = I.quantize_e4m3(p["k_cache"].transpose(1, 2).contiguous())
    v8, vs = I.quantize_e4m3(p["v_cache"].transpose(1, 2).contiguous())
    k = p["k"].clone()
    k.view(-1)[:4] = torch.tensor([0.0, -0.0, 1e4, -1e4], dtype=torch.bfloat16)  # zeros, huge
    p["k"] = k
    return p, k8, v8, ks * shrink, vs * shrink


def oracle_e4m3(p, k8, v8, ks, vs):
    nhd = [t.view(torch.uint8).transpose(1, 2).contiguous().cpu().numpy() for t in (k8, v8)]
    return O.kv_cache_write_e4m3(nhd[0], nhd[1], bf16_bits(p["k"]), bf16_bits(p["v"]),
                                 host(p, "cu_seqlens"), host(p, "ctx_lens"),
                                 host(p, "block_table"), ks, vs)


@pytest.mark.parametrize("name,shrink", [("prefix_window", 1.0), ("ragged_many", 1.0),
                                         ("ragged_many", 0.05)])
def test_e4m3_cache_write_is_the_oracle_quantiser(name, shrink):
    p, k8, v8, ks, vs = e4m3_case(name, 202, shrink)
    want_k, want_v = oracle_e4m3(p, k8, v8, ks, vs)
    assert write(p, k8, v8, ks, vs) == 0
    for got, want in ((k8, want_k), (v8, want_v)):
        got = got.view(torch.uint8).transpose(1, 2).contiguous().cpu().numpy()
        assert np.array_equal(got, want)


def test_e4m3_cache_write_needs_dv_128_and_scales():
    p = I.make_prefill(CASES["dv64"], DEV, seed_data=203)
    k8, ks = I.quantize_e4m3(p["k_cache"].transpose(1, 2).contiguous())
    v8, vs = I.quantize_e4m3(p["v_cache"].transpose(1, 2).contiguous())
    with pytest.raises(R.RelattnError) as e:
        write(p, k8, v8, ks, vs)
    assert e.value.code == R.ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        write(p, k8, v8)


def test_bad_block_id_sets_the_status_and_skips_only_that_token():
    p = I.make_prefill(CASES["prefix_window"], DEV, seed_data=204)
    bt = p["block_table"].clone()
    bt[1, 0] = 10_000  # sequence 1's first block is outside the pool
    p["block_table"] = bt
    k0 = bf16_bits(p["k_cache"])
    st = write(p, p["k_cache"], p["v_cache"])
    assert st & R.DEV_BAD_BLOCK_ID
    # sequence 0's tokens are written as the oracle writes them
    ok = dict(p, block_table=bt[:1], cu_seqlens=p["cu_seqlens"][:2], ctx_lens=p["ctx_lens"][:1])
    want_k, _ = O.kv_cache_write(k0, bf16_bits(p["v_cache"]), bf16_bits(p["k"]),
                                 bf16_bits(p["v"]), host(ok, "cu_seqlens"),
                                 host(ok, "ctx_lens"), host(ok, "block_table"))
    got = bf16_bits(p["k_cache"])
    used = sorted({int(x) for x in bt[0].tolist() if x >= 0})
    assert np.array_equal(got[used], want_k[used])


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_decode_step_appends_its_token_then_attends(kv):
    """A decode step's newest key and value are written with
    relattn_cache_write (one token per sequence at position L - 1), then the
    decode reads them: equal to the oracle's write followed by its decode."""
    wl = I.variant(I.WORKLOADS["global_decode_b8"], batch=4, lengths=("uniform", 1, 3000),
                   kv_dtype=kv)
    case = I.make_decode(wl, DEV, seed_data=205)
    B = case["q"].shape[0]
    g = torch.Generator(device="cpu")
    g.manual_seed(206)
    k_new = torch.randn((B, 8, 128), generator=g).to(DEV, torch.bfloat16)
    v_new = torch.randn((B, 8, 128), generator=g).to(DEV, torch.bfloat16)
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    ctx = case["seq_lens"] - 1
    # the oracle: its own write into a copy of the old cache, then its decode
    kc0, vc0 = host_cache(case["k_cache"]), host_cache(case["v_cache"])
    args = (bf16_bits(k_new), bf16_bits(v_new), cu.cpu().numpy(), ctx.cpu().numpy(),
            case["block_table"].cpu().numpy())
    if kv == "fp8":
        kc1, vc1 = O.kv_cache_write_e4m3(kc0, vc0, *args, case["k_scale"], case["v_scale"])
    else:
        kc1, vc1 = O.kv_cache_write(kc0, vc0, *args)
    want = O.decode(bf16_bits(case["q"]), case["rel"].cpu().numpy(), kc1, vc1,
                    case["block_table"].cpu().numpy(), case["seq_lens"].cpu().numpy(),
                    case["window"], case["rel_extent"], k_scale=case.get("k_scale", 1.0),
                    v_scale=case.get("v_scale", 1.0))
    R.relattn_cache_write(k_new, v_new, cu, case["k_cache"], case["v_cache"],
                          case["block_table"], ctx, 1, k_scale=case.get("k_scale"),
                          v_scale=case.get("v_scale"))
    out = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                           case["block_table"], case["seq_lens"], case["window"],
                           case["rel_extent"], k_scale=case.get("k_scale"),
                           v_scale=case.get("v_scale"))
    torch.cuda.synchronize()
    assert np.array_equal(host_cache(case["k_cache"]), kc1)
    assert np.array_equal(host_cache(case["v_cache"]), vc1)
    assert_parity(to_f64(out), want, what=f"append + decode ({kv})")
