"""GPU attention with the gated output and a per-token sink, vs the oracle.

Each query row and head has a sink logit (one more term of the softmax's
normaliser, with no value) and a gate logit (its sigmoid scales the head's
output), through relattn_decode_ex / relattn_prefill_ex.  A sink of -inf and
a gate of +inf reproduce the plain output bit for bit.
"""

import numpy as np
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


def logits_like(shape, seed, scale=2.0, shift=0.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale + shift).to(DEV)


def run_decode(case, num_ctas=0, out_dtype=torch.bfloat16):
    q = case["q"]
    dims = R.Dims(q.shape[0], q.shape[-2], case["block_table"].shape[1], 0, 0, num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    fn = R.relattn_decode_multi if q.dim() == 4 else R.relattn_decode
    out = fn(q, case["rel"], case["k_cache"], case["v_cache"], case["block_table"],
             case["seq_lens"], case["window"], case["rel_extent"], workspace=ws,
             num_ctas=num_ctas, out_dtype=out_dtype, sink=case.get("sink"),
             gate=case.get("gate"))
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    return out


DECODE = {
    "local_w512": I.variant(I.WORKLOADS["local_decode"], batch=5, lengths=("uniform", 1, 3000),
                            pool_blocks=0, max_blocks_per_seq=0),
    "gqa16": I.DecodeWorkload("gqa16", 2, 32, 2, 128, 64, 300, 512, ("uniform", 200, 2500)),
    "global_dv64": I.variant(I.WORKLOADS["diffhead_decode"], batch=4,
                             lengths=("loguniform", 64, 5000)),
}


@pytest.mark.parametrize("name", sorted(DECODE))
@pytest.mark.parametrize("num_ctas", [0, 7, 1000])
def test_gated_decode(name, num_ctas):
    """Whole segments (no split) and split ones (the combine adds the sink
    once and applies the gate once)."""
    case = I.make_decode(DECODE[name], DEV, seed_data=91)
    B, Hq = case["q"].shape[:2]
    case["sink"] = logits_like((B, Hq), 92)
    case["gate"] = logits_like((B, Hq), 93)
    out = run_decode(case, num_ctas=num_ctas, out_dtype=torch.float32)
    assert_parity(to_f64(out), oracle_decode(case), what=f"{name} num_ctas={num_ctas}")


def test_gated_multi_token_decode():
    wl = I.DecodeWorkload("multi", 5, 16, 4, 128, 128, 512, 512, ("uniform", 8, 3000),
                          query_tokens=8)
    case = I.make_decode(wl, DEV, seed_data=94)
    case["sink"] = logits_like((5, 8, 16), 95)
    case["gate"] = logits_like((5, 8, 16), 96)
    out = run_decode(case)
    assert_parity(to_f64(out), oracle_decode_multi(case), what="multi k=8")


def test_large_sink_and_negative_gate_drive_the_output_to_zero():
    case = I.make_decode(DECODE["local_w512"], DEV, seed_data=97)
    B, Hq = case["q"].shape[:2]
    case["sink"] = logits_like((B, Hq), 98, scale=10.0, shift=150.0)  # e^150 overflows fp32
    case["gate"] = logits_like((B, Hq), 99, scale=1.0, shift=-5.0)
    out = run_decode(case, out_dtype=torch.float32)
    want = oracle_decode(case)
    assert np.all(np.isfinite(to_f64(out)))
    assert_parity(to_f64(out), want, what="saturated sink")


def test_no_op_sink_and_gate_give_the_plain_output_bit_for_bit():
    case = I.make_decode(DECODE["local_w512"], DEV, seed_data=100)
    plain = run_decode(case)
    B, Hq = case["q"].shape[:2]
    case["sink"] = torch.full((B, Hq), float("-inf"), device=DEV)
    case["gate"] = torch.full((B, Hq), float("inf"), device=DEV)
    gated = run_decode(case)
    assert torch.equal(plain.view(torch.int16), gated.view(torch.int16))


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
def test_gated_prefill(name, out_dtype, num_ctas):
    case = I.make_prefill(PREFILL[name], DEV, seed_data=101)
    T, Hq = case["q"].shape[:2]
    case["sink"] = logits_like((T, Hq), 102)
    case["gate"] = logits_like((T, Hq), 103)
    cache0 = snapshot_cache(case)
    want, _, _ = oracle_prefill(case, cache=cache0)
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"],
                          num_ctas)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    out = R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                            case["k_cache"], case["v_cache"], case["block_table"],
                            case["ctx_lens"], case["window"], case["rel_extent"],
                            case["max_q_len"], workspace=ws, out_dtype=out_dtype,
                            sink=case["sink"], gate=case["gate"], num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    assert_parity(to_f64(out), want, what=f"{name} out={out_dtype}")


def test_sink_needs_only_4_byte_alignment():
    case = I.make_decode(DECODE["local_w512"], DEV, seed_data=104)
    B, Hq = case["q"].shape[:2]
    buf = torch.zeros(B * Hq + 1, dtype=torch.float32, device=DEV)
    sink = buf[1:].view(B, Hq)  # 4-byte aligned: accepted
    run_decode(dict(case, sink=sink))
