"""GPU chunked prefill over an FP8 (e4m3) KV cache, vs the oracle.

The prefill first quantises the new keys and values into the e4m3 cache
(head-major blocks, per-tensor scales), then attends over the cache with f16
MMAs (every e4m3 value, and q and P, in f16).  The oracle writes the same
codes and reads them back exactly, so the cache is compared bit for bit and
the output within the usual tolerance."""

import numpy as np
import pytest
import torch

from paged_relative_bias_gb300 import inputs as I
from paged_relative_bias_gb300 import relattn as R
from tests.parity import (assert_parity, host_cache, oracle_decode, oracle_prefill,
                          snapshot_cache, to_f64)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_relative_bias_gb300 import build
    build.build()
    R.lib()


def fp8(wl, **kw):
    return I.variant(wl, kv_dtype="fp8", **kw)


CASES = {
    "prefix_window": fp8(I.PrefillWorkload("pw", 12, 2, 128, 128, 100, 64, (200, 77),
                                           (300, 0))),
    "ragged_many": fp8(I.PrefillWorkload("rm", 8, 8, 128, 128, 256, 512,
                                         (1, 63, 64, 65, 127, 128, 129, 200),
                                         (0, 1, 127, 128, 129, 0, 64, 1000))),
    "global": fp8(I.PrefillWorkload("gl", 32, 8, 128, 128, 0, 1024, (300, 130),
                                    (1500, 700))),
}


def run(p, out_dtype=torch.bfloat16):
    dims = R.prefill_dims(p["q"], p["block_table"], p["ctx_lens"], p["max_q_len"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(p["k_cache"], p["v_cache"])),
                         DEV)
    out = R.relattn_prefill(p["q"], p["k"], p["v"], p["rel"], p["cu_seqlens"], p["k_cache"],
                            p["v_cache"], p["block_table"], p["ctx_lens"], p["window"],
                            p["rel_extent"], p["max_q_len"], workspace=ws, out_dtype=out_dtype,
                            sink=p.get("sink"), gate=p.get("gate"),
                            logit_scale=p.get("logit_scale"), k_scale=p["k_scale"],
                            v_scale=p["v_scale"])
    torch.cuda.synchronize()
    assert R.read_status(ws) == 0
    return out


@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_prefill_small_configs(name):
    p = I.make_prefill(CASES[name], DEV, seed_data=221)
    assert p["k_cache"].dtype == torch.float8_e4m3fn
    cache0 = snapshot_cache(p)
    want, kc1, vc1 = oracle_prefill(p, cache=cache0)
    out = run(p)
    assert np.array_equal(host_cache(p["k_cache"]), kc1)  # the quantised write, bit for bit
    assert np.array_equal(host_cache(p["v_cache"]), vc1)
    assert_parity(to_f64(out), want, what=name)


def test_fp8_prefill_with_every_option():
    """bf16 rel, fp32 out, sink, gate and log-position factors together."""
    p = I.make_prefill(fp8(CASES["ragged_many"], rel_dtype="bf16"), DEV, seed_data=222)
    T, Hq = p["q"].shape[:2]
    g = torch.Generator(device="cpu")
    g.manual_seed(223)
    p["sink"] = torch.randn((T, Hq), generator=g).to(DEV)
    p["gate"] = torch.randn((T, Hq), generator=g).to(DEV)
    p["logit_scale"] = (0.5 + 2 * torch.rand((T,), generator=g)).to(DEV)
    cache0 = snapshot_cache(p)
    want, _, _ = oracle_prefill(p, cache=cache0)
    out = run(p, out_dtype=torch.float32)
    assert_parity(to_f64(out), want, what="fp8 prefill, every option")


def test_decode_after_fp8_prefill_reads_what_it_wrote():
    """A decode at the prefill's last position, over the cache the prefill
    just wrote, equals the oracle's decode of the same cache and the prefill's
    own last rows."""
    wl = CASES["global"]
    p = I.make_prefill(wl, DEV, seed_data=224)
    out = run(p)
    B = wl.batch
    cu = p["cu_seqlens"].tolist()
    last = torch.tensor([cu[b + 1] - 1 for b in range(B)], device=DEV)
    case = dict(q=p["q"][last].contiguous(), rel=p["rel"][last].contiguous(),
                k_cache=p["k_cache"], v_cache=p["v_cache"], block_table=p["block_table"],
                seq_lens=(p["ctx_lens"] + p["cu_seqlens"][1:] - p["cu_seqlens"][:-1]).int(),
                window=wl.window, rel_extent=wl.rel_extent, k_scale=p["k_scale"],
                v_scale=p["v_scale"])
    dec = R.relattn_decode(case["q"], case["rel"], case["k_cache"], case["v_cache"],
                           case["block_table"], case["seq_lens"], case["window"],
                           case["rel_extent"], k_scale=case["k_scale"],
                           v_scale=case["v_scale"])
    torch.cuda.synchronize()
    assert_parity(to_f64(dec), oracle_decode(case), what="decode after fp8 prefill")
    assert_parity(to_f64(dec), to_f64(out[last]), what="decode vs prefill last rows")


def test_fp8_full_chunked_prefill_sampled_rows():
    """The chunked-prefill workload (4 x 8192 after 24,576, 48/8 heads,
    W = E = 1024) over an e4m3 cache, on sampled rows of every sequence."""
    p = I.make_prefill(fp8(I.WORKLOADS["chunked_prefill"]), DEV, seed_data=225)
    cache0 = snapshot_cache(p)
    out = run(p)
    cu = p["cu_seqlens"].tolist()
    rows = [r for b in range(4) for r in (cu[b], cu[b] + 1000, cu[b + 1] - 1)]
    want, _, _ = oracle_prefill(p, rows=rows, cache=cache0)
    assert_parity(to_f64(out)[rows], want[rows], what="chunked prefill fp8")
