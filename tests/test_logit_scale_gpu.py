"""GPU attention with a per-token log-position scale, vs the oracle.

Each query token has a factor that multiplies both terms of its logits, q.k
/ sqrt(d) and rel (the log-position scale of the global layers), through
relattn_decode_ex / relattn_prefill_ex.  A factor of 1 reproduces the plain
output bit for bit; a sink logit is not scaled.
"""

import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from tests.parity import (assert_parity, oracle_decode, oracle_decode_multi, oracle_prefill,
                          snapshot_cache, to_f64)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def factors(shape, seed, lo=0.5, hi=2.5):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (lo + (hi - lo) * torch.rand(shape, generator=g, dtype=torch.float32)).to(DEV)


def run_decode(case, num_ctas=0, out_dtype=torch.bfloat16):
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


def run_prefill(case, out_dtype=torch.bfloat16, num_ctas=0):
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"],
                          num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out = R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                            case["k_cache"], case["v_cache"], case["block_table"],
                            case["ctx_lens"], case["window"], case["rel_extent"],
                            case["max_q_len"], workspace=ws, out_dtype=out_dtype,
                            sink=case.get("sink"), gate=case.get("gate"),
                            logit_scale=case.get("logit_scale"), num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    return out


DECODE = {
    "local_w512": I.variant(I.WORKLOADS["local_decode"], batch=5, lengths=("uniform", 1, 3000),
                            pool_blocks=0, max_blocks_per_seq=0),
    "global_e1024": I.variant(I.WORKLOADS["global_decode_b8"], batch=3,
                              lengths=("uniform", 1, 6000)),
    "gqa16": I.DecodeWorkload("gqa16", 2, 32, 2, 128, 64, 300, 512, ("uniform", 200, 2500)),
    "global_dv64": I.variant(I.WORKLOADS["diffhead_decode"], batch=4,
                             lengths=("loguniform", 64, 5000)),
}


@pytest.mark.parametrize("name", sorted(DECODE))
@pytest.mark.parametrize("num_ctas", [0, 7, 1000])
def test_scaled_decode(name, num_ctas):
    """Whole segments and split ones (the combine sees the scaled logits)."""
    case = I.make_decode(DECODE[name], DEV, seed_data=131)
    case["logit_scale"] = factors(case["q"].shape[:1], 132)
    out = run_decode(case, num_ctas=num_ctas)
    assert_parity(to_f64(out), oracle_decode(case), what=f"{name} num_ctas={num_ctas}")


@pytest.mark.parametrize("k", [2, 5, 8])
def test_scaled_multi_token_decode(k):
    wl = I.DecodeWorkload("multi", 5, 16, 4, 128, 128, 512, 512, ("uniform", 8, 3000),
                          query_tokens=k)
    case = I.make_decode(wl, DEV, seed_data=133)
    case["logit_scale"] = factors((5, k), 134)
    out = run_decode(case)
    assert_parity(to_f64(out), oracle_decode_multi(case), what=f"multi k={k}")


def test_scaled_decode_fp8_cache_with_sink_and_gate():
    wl = I.variant(DECODE["global_e1024"], kv_dtype="fp8")
    case = I.make_decode(wl, DEV, seed_data=135)
    B, Hq = case["q"].shape[:2]
    case["logit_scale"] = factors((B,), 136)
    g = torch.Generator(device="cpu")
    g.manual_seed(137)
    case["sink"] = torch.randn((B, Hq), generator=g).to(DEV)
    case["gate"] = torch.randn((B, Hq), generator=g).to(DEV)
    out = run_decode(case, out_dtype=torch.float32)
    assert_parity(to_f64(out), oracle_decode(case), what="fp8 + sink/gate + factor")


def test_decode_factor_one_is_the_plain_output_bit_for_bit():
    for name in ("local_w512", "gqa16"):
        case = I.make_decode(DECODE[name], DEV, seed_data=138)
        plain = run_decode(case)
        case["logit_scale"] = torch.ones(case["q"].shape[:1], device=DEV)
        scaled = run_decode(case)
        assert torch.equal(plain.view(torch.int16), scaled.view(torch.int16)), name


def test_full_size_global_b1_sampled():
    """The long-context global layer (100,000 tokens, 19 pieces per segment)
    with a factor above 1, as past 128K."""
    case = I.make_decode(I.WORKLOADS["global_decode_b1"], DEV, seed_data=139)
    case["logit_scale"] = torch.full((1,), 1.37, device=DEV)
    out = run_decode(case)
    hs = [0, 13, 31]
    want = oracle_decode(case, heads=hs)
    assert_parity(to_f64(out)[:, hs], want[:, hs], what="global b1 100K")


PREFILL = {
    "prefix_window": I.PrefillWorkload("pw", 12, 2, 128, 128, 100, 64, (200, 77), (300, 0)),
    "global_dv64": I.PrefillWorkload("g64", 8, 2, 128, 64, 0, 256, (130, 1, 64), (0, 500, 129)),
    "ragged_many": I.PrefillWorkload("rm", 8, 8, 128, 128, 256, 512,
                                     (1, 63, 64, 65, 127, 128, 129, 200),
                                     (0, 1, 127, 128, 129, 0, 64, 1000)),
}


@pytest.mark.parametrize("num_ctas", [0, 148])  # 148: two heads per work item (forced grid)
@pytest.mark.parametrize("name", sorted(PREFILL))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_scaled_prefill(name, out_dtype, num_ctas):
    case = I.make_prefill(PREFILL[name], DEV, seed_data=141)
    case["logit_scale"] = factors(case["q"].shape[:1], 142, lo=0.25, hi=4.0)
    cache0 = snapshot_cache(case)
    want, _, _ = oracle_prefill(case, cache=cache0)
    out = run_prefill(case, out_dtype, num_ctas)
    assert_parity(to_f64(out), want, what=f"{name} out={out_dtype}")


def test_scaled_prefill_with_sink_and_bf16_rel():
    wl = I.variant(PREFILL["prefix_window"], rel_dtype="bf16")
    case = I.make_prefill(wl, DEV, seed_data=143)
    T, Hq = case["q"].shape[:2]
    case["logit_scale"] = factors((T,), 144)
    g = torch.Generator(device="cpu")
    g.manual_seed(145)
    case["sink"] = (torch.randn((T, Hq), generator=g) * 2).to(DEV)
    cache0 = snapshot_cache(case)
    want, _, _ = oracle_prefill(case, cache=cache0)
    out = run_prefill(case)
    assert_parity(to_f64(out), want, what="prefill + sink + bf16 rel + factor")


def test_prefill_factor_one_is_the_plain_output_bit_for_bit():
    case = I.make_prefill(PREFILL["ragged_many"], DEV, seed_data=146)
    k0, v0 = case["k_cache"].clone(), case["v_cache"].clone()
    plain = run_prefill(case)
    case["k_cache"].copy_(k0)
    case["v_cache"].copy_(v0)
    case["logit_scale"] = torch.ones(case["q"].shape[:1], device=DEV)
    scaled = run_prefill(case)
    assert torch.equal(plain.view(torch.int16), scaled.view(torch.int16))


def test_logit_scale_shape_is_checked():
    case = I.make_decode(DECODE["local_w512"], DEV, seed_data=147)
    case["logit_scale"] = torch.ones((case["q"].shape[0], 2), device=DEV)
    with pytest.raises(ValueError):
        run_decode(case)
