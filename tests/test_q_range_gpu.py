"""Over an e4m3 cache the kernels compute in f16, so a bf16 query element
beyond f16's range (|q| > 65504) cannot be represented: the call reports
RELATTN_DEV_Q_RANGE in the status word.  Every other row is still correct;
over a bf16 cache the same query is no error (no narrowing)."""

import numpy as np
import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from tests.parity import assert_parity, oracle_decode, oracle_decode_multi, oracle_prefill, \
    snapshot_cache, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BIG = 1.0e5  # a bf16 value (99840) past f16's largest finite value, 65504


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def decode(case, tokens):
    q = case["q"]
    dims = R.Dims(q.shape[0], q.shape[-2], case["block_table"].shape[1], 0, 0, 0)
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), DEV)
    fn = R.relattn_decode_multi if tokens else R.relattn_decode
    out = fn(q, case["rel"], case["k_cache"], case["v_cache"], case["block_table"],
             case["seq_lens"], case["window"], case["rel_extent"], workspace=ws,
             k_scale=case.get("k_scale"), v_scale=case.get("v_scale"))
    torch.cuda.synchronize()
    return out, R.read_status(ws)


@pytest.mark.parametrize("kv,tokens", [("fp8", 0), ("fp8", 4), ("bf16", 0), ("bf16", 4)])
def test_decode_query_beyond_f16(kv, tokens):
    wl = I.DecodeWorkload("qr", 3, 32, 8, 128, 128, 0, 256, ("uniform", 10, 900),
                          query_tokens=tokens, kv_dtype=kv)
    case = I.make_decode(wl, DEV, seed_data=401)
    bad = (1, 0, 9) if tokens == 0 else (1, 2, 0, 9)  # (sequence, [token,] head, dim)
    case["q"][bad] = BIG
    out, status = decode(case, tokens)
    if kv == "bf16":
        assert status == 0
    else:
        assert status & R.DEV_Q_RANGE
    # every other (sequence, token, head) row matches the oracle
    want = oracle_decode_multi(case) if tokens else oracle_decode(case)
    got = to_f64(out)
    mask = np.ones(got.shape[:-1], dtype=bool)
    mask[bad[:-1]] = False
    assert_parity(got[mask], want[mask], what=f"{kv} k={tokens} other rows")


def test_prefill_query_beyond_f16():
    wl = I.variant(I.PrefillWorkload("qp", 8, 2, 128, 128, 0, 256, (150, 70), (40, 300)),
                   kv_dtype="fp8")
    p = I.make_prefill(wl, DEV, seed_data=402)
    row, head = 160, 5  # sequence 1, token 10
    p["q"][row, head, 3] = BIG
    cache0 = snapshot_cache(p)
    dims = R.prefill_dims(p["q"], p["block_table"], p["ctx_lens"], p["max_q_len"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(p["k_cache"], p["v_cache"])), DEV)
    out = R.relattn_prefill(p["q"], p["k"], p["v"], p["rel"], p["cu_seqlens"], p["k_cache"],
                            p["v_cache"], p["block_table"], p["ctx_lens"], p["window"],
                            p["rel_extent"], p["max_q_len"], workspace=ws, k_scale=p["k_scale"],
                            v_scale=p["v_scale"])
    torch.cuda.synchronize()
    assert R.read_status(ws) & R.DEV_Q_RANGE
    want, _, _ = oracle_prefill(p, cache=cache0)
    got = to_f64(out)
    mask = np.ones(got.shape[:-1], dtype=bool)
    mask[row, head] = False
    assert_parity(got[mask], want[mask], what="prefill other rows")
