"""Pins of the float64 oracle against things other than itself.

Brute force on tiny inputs, a float64 library routine (torch SDPA with an
explicit additive bias), closed forms, invariants and the facts the pages
print (tests/golden).  Each pin is chosen so that a plausible slip in the
oracle -- a dropped term, a wrong sign of the distance, an off-by-one window,
a swapped block/slot index, the wrong KV head -- fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import relattn_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def paged_from_contiguous(Kc, Vc, table_row, pool):
    """Scatter contiguous [n, Hkv, d] keys/values into a paged pool."""
    n, Hkv, d = Kc.shape
    kc = np.zeros((pool, 128, Hkv, d))
    vc = np.zeros((pool, 128, Hkv, Vc.shape[2]))
    for j in range(n):
        kc[table_row[j // 128], j % 128] = Kc[j]
        vc[table_row[j // 128], j % 128] = Vc[j]
    return kc, vc


def random_decode_case(seed, L, Hq=4, Hkv=2, d=16, dv=8, E=64, pool_extra=2):
    r = rng(seed)
    nblk = (L + 127) // 128
    pool = nblk + pool_extra
    table = r.permutation(pool)[:nblk]
    Kc = r.standard_normal((L, Hkv, d))
    Vc = r.standard_normal((L, Hkv, dv))
    kc, vc = paged_from_contiguous(Kc, Vc, table, pool)
    q = r.standard_normal((1, Hq, d))
    rel = r.standard_normal((1, Hq, E))
    return dict(q=q, rel=rel, kc=kc, vc=vc, table=table[None, :], Kc=Kc, Vc=Vc,
                seq_lens=np.array([L]))


# ---------------------------------------------------------------------------
# page facts
# ---------------------------------------------------------------------------

def test_golden_block_size_and_window_facts():
    g = json.load(open(os.path.join(GOLDEN, "decode_window.json")))["facts"]
    assert g["pool_tokens"] == g["pool_blocks"] * O.BLOCK_SIZE
    W = g["local_window"]
    lo_seen, hi_seen = g["keys_seen_with_window_div_block_size_blocks"]
    seen = []
    for P in range(W - 1, 4000):
        # what a walker with only window/block_size blocks would show
        last = P // 128
        first = last - W // 128 + 1
        seen.append(P - first * 128 + 1)
        # the oracle's window: exactly W keys once the context is long enough
        lo, hi = O.visible_keys(P, W)
        assert hi - lo + 1 == g["keys_seen_after_one_more_block_and_exact_mask"]
        blocks = O.decode_blocks(P + 1, W, np.arange(last + 1))
        assert len(blocks) <= g["local_prefill_context_blocks"]
        assert blocks[0][0] * 128 <= lo and blocks[-1][0] == last
    assert min(seen) == lo_seen and max(seen) == hi_seen
    # the fix: W/128 + 1 blocks always suffice, and are needed sometimes
    assert g["local_prefill_context_blocks"] == W // 128 + 1


# ---------------------------------------------------------------------------
# block walk: brute force over key sets
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("W", [0, 1, 64, 127, 128, 129, 512, 1024])
def test_decode_blocks_brute_force(W):
    table = np.arange(1000, 1040)
    for L in list(range(1, 300)) + [511, 512, 513, 1023, 1024, 1025, 4000]:
        want = sorted({j // 128 for j in range(L) if W <= 0 or L - 1 - j < W})
        got = O.decode_blocks(L, W, table)
        assert [l for l, _ in got] == want
        assert [p for _, p in got] == [int(table[l]) for l in want]
        if W > 0:
            assert len(got) <= math.ceil(W / 128) + 1


@pytest.mark.parametrize("W", [0, 1, 100, 1024])
def test_prefill_blocks_brute_force(W):
    table = np.arange(500, 560)
    r = rng(3)
    for _ in range(200):
        ctx = int(r.integers(0, 3000))
        t0 = int(r.integers(0, 500))
        t1 = t0 + int(r.integers(0, 300))
        keys = set()
        for t in range(t0, t1 + 1):
            P = ctx + t
            keys |= {j for j in range(P + 1) if W <= 0 or P - j < W}
        want = sorted({j // 128 for j in keys})
        got = O.prefill_blocks(ctx, t0, t1, W, table)
        assert [l for l, _ in got] == want


# ---------------------------------------------------------------------------
# paged addressing, written out by hand for the tiny layout [1, 0]
# ---------------------------------------------------------------------------

def test_gather_by_hand_layout():
    r = rng(7)
    kc = r.standard_normal((2, 128, 1, 4))
    vc = r.standard_normal((2, 128, 1, 3))
    table = np.array([1, 0])
    K, V = O.gather_kv(kc, vc, table, [0, 5, 127, 128, 200, 255], 0)
    np.testing.assert_array_equal(K[0], kc[1, 0, 0])
    np.testing.assert_array_equal(K[1], kc[1, 5, 0])
    np.testing.assert_array_equal(K[2], kc[1, 127, 0])
    np.testing.assert_array_equal(K[3], kc[0, 0, 0])
    np.testing.assert_array_equal(K[4], kc[0, 72, 0])
    np.testing.assert_array_equal(V[5], vc[0, 127, 0])


def test_bf16_conversion_exact():
    vals = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3, -65504.0, 2.0 ** -126])
    bits = O.f64_to_bf16_bits(vals)
    back = O.bf16_bits_to_f64(bits)
    # bf16 keeps 8 significant bits: relative rounding error <= 2^-9
    assert np.all(np.abs(back - vals) <= np.abs(vals) * 2.0 ** -9)
    # values already on the bf16 grid come back exactly
    np.testing.assert_array_equal(O.bf16_bits_to_f64(O.f64_to_bf16_bits(back)), back)
    assert O.bf16_bits_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
    assert O.bf16_bits_to_f64(np.array([0xC020], dtype=np.uint16))[0] == -2.5


# ---------------------------------------------------------------------------
# textbook reductions
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L", [1, 2, 77, 128, 129, 300])
def test_brute_force_causal_softmax_when_rel_zero(L):
    """rel = 0, global: plain causal softmax attention, written as loops."""
    c = random_decode_case(L, L, E=8)
    c["rel"][:] = 0.0
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                   c["seq_lens"], 0, 8)
    Hq, Hkv = 4, 2
    for h in range(Hq):
        kvh = h // 2
        s = [sum(c["q"][0, h, x] * c["Kc"][j, kvh, x] for x in range(16)) / 4.0
             for j in range(L)]
        m = max(s)
        e = [math.exp(v - m) for v in s]
        tot = sum(e)
        for x in range(8):
            o = sum(e[j] * c["Vc"][j, kvh, x] for j in range(L)) / tot
            assert abs(out[0, h, x] - o) < 1e-12


def sdpa_reference(q, Kc, Vc, rel, positions, window, E):
    """torch SDPA in float64 over contiguous keys with an explicit bias."""
    T, Hq, d = q.shape
    n, Hkv, _ = Kc.shape
    g = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)                     # [Hq, T, d]
    kt = torch.from_numpy(Kc).permute(1, 0, 2).repeat_interleave(g, 0)
    vt = torch.from_numpy(Vc).permute(1, 0, 2).repeat_interleave(g, 0)
    mask = torch.full((Hq, T, n), float("-inf"), dtype=torch.float64)
    for i, P in enumerate(positions):
        for j in range(n):
            dist = P - j
            if dist < 0 or (window > 0 and dist >= window):
                continue
            for h in range(Hq):
                mask[h, i, j] = rel[i, h, dist] if dist < E else 0.0
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("L,W,E", [(1, 0, 16), (200, 0, 300), (200, 0, 50),
                                   (260, 64, 64), (260, 100, 40), (129, 1, 4)])
def test_decode_equals_float64_sdpa(L, W, E):
    c = random_decode_case(100 + L, L, E=E, dv=6)
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                   c["seq_lens"], W, E)
    ref = sdpa_reference(c["q"], c["Kc"], c["Vc"], c["rel"], [L - 1], W, E)
    np.testing.assert_allclose(out[0], ref[0], atol=1e-12, rtol=0)


def test_prefill_equals_float64_sdpa():
    r = rng(11)
    ctx, n, Hq, Hkv, d, dv, W, E = 150, 90, 6, 2, 16, 8, 100, 64
    total = ctx + n
    nblk = (total + 127) // 128
    table = r.permutation(nblk + 1)[:nblk]
    Kc = r.standard_normal((total, Hkv, d))
    Vc = r.standard_normal((total, Hkv, dv))
    kc, vc = paged_from_contiguous(Kc[:ctx], Vc[:ctx], table, nblk + 1)
    q = r.standard_normal((n, Hq, d))
    rel = r.standard_normal((n, Hq, E))
    out, kc2, vc2 = O.prefill(q, Kc[ctx:], Vc[ctx:], rel, [0, n], kc, vc,
                              table[None, :], [ctx], W, E)
    ref = sdpa_reference(q, Kc, Vc, rel, [ctx + t for t in range(n)], W, E)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    # the cache now holds the new keys at their positions
    K, V = O.gather_kv(kc2, vc2, table, np.arange(total), 1)
    np.testing.assert_array_equal(K, Kc[:, 1])
    np.testing.assert_array_equal(V, Vc[:, 1])


# ---------------------------------------------------------------------------
# closed forms: zero query, geometric relative bias
# ---------------------------------------------------------------------------

def geometric_case(L, W, E, rho):
    """q = 0, rel[d] = d*ln(rho), value = key position: closed-form output."""
    r = rng(5)
    nblk = (L + 127) // 128
    table = r.permutation(nblk + 3)[:nblk]
    Kc = r.standard_normal((L, 1, 8))
    Vc = np.zeros((L, 1, 2))
    Vc[:, 0, 0] = np.arange(L)
    Vc[:, 0, 1] = 1.0
    kc, vc = paged_from_contiguous(Kc, Vc, table, nblk + 3)
    q = np.zeros((1, 1, 8))
    rel = (np.arange(E) * math.log(rho))[None, None, :]
    out = O.decode(q, rel, kc, vc, table[None, :], np.array([L]), W, E)
    return out[0, 0]


def geometric_expected(P, n, E, rho):
    """sum_d w_d (P - d) / sum_d w_d, w_d = rho^d for d < E else 1."""
    m = min(n, E)
    s0 = (1 - rho ** m) / (1 - rho)
    s1 = rho * (1 - m * rho ** (m - 1) + (m - 1) * rho ** m) / (1 - rho) ** 2
    num = P * s0 - s1
    den = s0
    if n > E:
        k = n - E  # distances E .. n-1, weight 1
        num += k * P - (E + n - 1) * k / 2.0
        den += k
    return num / den


@pytest.mark.parametrize("L,W,E", [(300, 0, 400), (300, 0, 37), (300, 64, 64),
                                   (300, 64, 16), (1, 0, 4), (500, 129, 200)])
def test_geometric_closed_form(L, W, E):
    rho = 0.9
    out = geometric_case(L, W, E, rho)
    P = L - 1
    n = min(L, W) if W > 0 else L
    assert abs(out[0] - geometric_expected(P, n, E, rho)) < 1e-9
    assert abs(out[1] - 1.0) < 1e-12


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_shift_invariance_when_all_distances_below_extent():
    for seed, (L, W, E) in enumerate([(300, 64, 64), (300, 40, 64), (50, 0, 64)]):
        c = random_decode_case(seed, L, E=E)
        base = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                        c["seq_lens"], W, E)
        shift = rng(99).standard_normal((1, 4, 1)) * 5
        moved = O.decode(c["q"], c["rel"] + shift, c["kc"], c["vc"], c["table"],
                         c["seq_lens"], W, E)
        np.testing.assert_allclose(moved, base, atol=1e-12)


def test_shift_changes_output_when_distances_reach_extent():
    # keys beyond rel_extent get 0, so a constant shift of rel is visible
    c = random_decode_case(4, 300, E=32)
    base = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                    c["seq_lens"], 0, 32)
    moved = O.decode(c["q"], c["rel"] + 3.0, c["kc"], c["vc"], c["table"],
                     c["seq_lens"], 0, 32)
    assert np.abs(moved - base).max() > 1e-3


def test_weights_are_a_distribution():
    for seed in range(10):
        c = random_decode_case(seed, 200 + seed * 17, E=64)
        for W in (0, 50):
            keys, w = O.decode_weights(c["q"][0, 1], c["rel"][0, 1], c["kc"],
                                       c["vc"], c["table"][0], int(c["seq_lens"][0]),
                                       0, W, 64)
            assert np.all(w >= 0)
            assert abs(w.sum() - 1.0) < 1e-12
            assert len(keys) == (min(W, len(c["Kc"])) if W > 0 else len(c["Kc"]))


def test_window_truncated_context_equals_full_40_cases():
    """Attending over only the last ceil(W/128)+1 blocks changes nothing.

    ("Inkling-Small on Gaudi 2", section "Attention with a relative bias":
    local-window prefill over the last 5 blocks equals the full-context path
    over 40 random cases.)  Positions of the truncated list come from each
    block's ordinal in it.
    """
    r = rng(2024)
    for case in range(40):
        W = int(r.choice([64, 128, 200, 512]))
        E = int(r.choice([W, W // 2, W + 7]))
        L = int(r.integers(1, 1500))
        c = random_decode_case(1000 + case, L, E=E)
        full = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                        c["seq_lens"], W, E)
        blocks = O.decode_blocks(L, W, c["table"][0])
        assert len(blocks) <= math.ceil(W / 128) + 1
        first = blocks[0][0]
        trunc_row = np.array([p for _, p in blocks])
        P = L - 1
        lo, _ = O.visible_keys(P, W)
        keys = np.arange(lo, P + 1)
        for h in range(4):
            K, V = O.gather_kv(c["kc"], c["vc"], trunc_row, keys - first * 128, h // 2)
            bias = O.rel_bias(c["rel"][0, h], P, keys, E)
            o = O.attend(c["q"][0, h], K, V, bias, 16)
            assert np.array_equal(o, full[0, h])


def test_paging_invariance_under_block_permutations():
    c = random_decode_case(8, 700, E=64)
    base = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                    c["seq_lens"], 0, 64)
    r = rng(9)
    for _ in range(5):
        pool = c["kc"].shape[0]
        perm = r.permutation(pool)          # new physical id of old block b
        kc = np.empty_like(c["kc"])
        vc = np.empty_like(c["vc"])
        kc[perm] = c["kc"]
        vc[perm] = c["vc"]
        table = perm[c["table"]]
        out = O.decode(c["q"], c["rel"], kc, vc, table, c["seq_lens"], 0, 64)
        assert np.array_equal(out, base)


def test_decode_equals_last_row_of_prefill():
    r = rng(21)
    L, Hq, Hkv, d, dv, E = 260, 4, 2, 16, 8, 64
    for W in (0, 100):
        nblk = 3
        table = r.permutation(5)[:nblk]
        K = r.standard_normal((L, Hkv, d))
        V = r.standard_normal((L, Hkv, dv))
        q = r.standard_normal((L, Hq, d))
        rel = r.standard_normal((L, Hq, E))
        kc0 = np.zeros((5, 128, Hkv, d))
        vc0 = np.zeros((5, 128, Hkv, dv))
        pre, kc, vc = O.prefill(q, K, V, rel, [0, L], kc0, vc0, table[None, :],
                                [0], W, E)
        dec = O.decode(q[L - 1:L], rel[L - 1:L], kc, vc, table[None, :],
                       np.array([L]), W, E)
        np.testing.assert_allclose(dec[0], pre[L - 1], atol=1e-13)


def test_chunked_prefill_equals_one_shot():
    r = rng(31)
    L, ctx, Hq, Hkv, d, dv, E, W = 300, 170, 4, 1, 16, 8, 128, 150
    table = r.permutation(4)[:3]
    K = r.standard_normal((L, Hkv, d))
    V = r.standard_normal((L, Hkv, dv))
    q = r.standard_normal((L, Hq, d))
    rel = r.standard_normal((L, Hq, E))
    kc0 = np.zeros((4, 128, Hkv, d))
    vc0 = np.zeros((4, 128, Hkv, dv))
    one, _, _ = O.prefill(q, K, V, rel, [0, L], kc0, vc0, table[None, :], [0], W, E)
    _, kc1, vc1 = O.prefill(q[:ctx], K[:ctx], V[:ctx], rel[:ctx], [0, ctx], kc0,
                            vc0, table[None, :], [0], W, E, rows=[])
    two, _, _ = O.prefill(q[ctx:], K[ctx:], V[ctx:], rel[ctx:], [0, L - ctx],
                          kc1, vc1, table[None, :], [ctx], W, E)
    np.testing.assert_allclose(two, one[ctx:], atol=1e-13)


def test_split_merge_equals_no_split():
    r = rng(41)
    n, d, dv = 500, 16, 8
    q = r.standard_normal(d)
    K = r.standard_normal((n, d))
    V = r.standard_normal((n, dv))
    bias = r.standard_normal(n) * 3
    whole = O.attend(q, K, V, bias, d)
    for _ in range(10):
        cuts = sorted(r.choice(np.arange(1, n), size=int(r.integers(1, 8)),
                               replace=False))
        parts = np.split(np.arange(n), cuts)
        outs, lses = zip(*[O.attend_partial(q, K[p], V[p], bias[p], d) for p in parts])
        np.testing.assert_allclose(O.merge_partials(outs, lses), whole, atol=1e-12)


def test_constant_values_give_that_value():
    c = random_decode_case(51, 333, E=64)
    c["vc"][:] = np.arange(8)[None, None, None, :] * 0.5 - 1.0
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                   c["seq_lens"], 100, 64)
    np.testing.assert_allclose(out[0], np.tile(np.arange(8) * 0.5 - 1.0, (4, 1)),
                               atol=1e-12)


def test_window_one_returns_own_value():
    c = random_decode_case(61, 259, E=8)
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                   c["seq_lens"], 1, 8)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], c["Vc"][258, h // 2])


def test_gqa_head_mapping():
    """Query head h reads KV head h // g: zero all but one KV head's values."""
    c = random_decode_case(71, 150, Hq=6, Hkv=3, E=16)
    c["vc"][:, :, [0, 2]] = 0.0
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"],
                   c["seq_lens"], 0, 16)
    assert np.all(out[0, [0, 1, 4, 5]] == 0.0)
    assert np.all(np.abs(out[0, [2, 3]]).sum(axis=1) > 0)


def test_cache_write_scatter_brute_force():
    r = rng(81)
    Hkv, d, dv = 2, 4, 3
    kc = r.standard_normal((6, 128, Hkv, d))
    vc = r.standard_normal((6, 128, Hkv, dv))
    cu, ctx = [0, 100, 103], [200, 0]
    table = np.array([[4, 1, 3], [0, 5, -1]])
    k = r.standard_normal((103, Hkv, d))
    v = r.standard_normal((103, Hkv, dv))
    kc2, vc2 = O.kv_cache_write(kc, vc, k, v, cu, ctx, table)
    touched = set()
    # sequence 0: positions 200..299 -> block 1 (phys 1) slots 72..127, block 2 (phys 3)
    for t in range(100):
        pos = 200 + t
        phys = [4, 1, 3][pos // 128]
        touched.add((phys, pos % 128))
        assert np.array_equal(kc2[phys, pos % 128], k[t])
    for t in range(3):
        touched.add((0, t))
        assert np.array_equal(vc2[0, t], v[100 + t])
    for b in range(6):
        for s in range(128):
            if (b, s) not in touched:
                assert np.array_equal(kc2[b, s], kc[b, s])
                assert np.array_equal(vc2[b, s], vc[b, s])


# ---------------------------------------------------------------------------
# multi-token decode (verification)
# ---------------------------------------------------------------------------

def random_multi_case(seed, L, k, Hq=4, Hkv=2, d=16, dv=8, E=64, pool_extra=2):
    c = random_decode_case(seed, L, Hq=Hq, Hkv=Hkv, d=d, dv=dv, E=E, pool_extra=pool_extra)
    r = rng(seed + 1000)
    c["qm"] = r.standard_normal((1, k, Hq, d))
    c["relm"] = r.standard_normal((1, k, Hq, E))
    return c


def test_decode_multi_one_token_equals_decode():
    c = random_multi_case(51, 300, 1)
    for W, E in ((0, 64), (100, 64), (1, 4)):
        multi = O.decode_multi(c["qm"], c["relm"], c["kc"], c["vc"], c["table"],
                               c["seq_lens"], W, E)
        dec = O.decode(c["qm"][:, 0], c["relm"][:, 0], c["kc"], c["vc"], c["table"],
                       c["seq_lens"], W, E)
        assert np.array_equal(multi[:, 0], dec)


@pytest.mark.parametrize("k,W", [(2, 0), (4, 64), (9, 100), (5, 1)])
def test_decode_multi_token_equals_decode_at_its_own_length(k, W):
    """Token i sees exactly what a one-token decode at length L - k + i + 1
    sees: later tokens' keys in the cache must not leak into earlier rows."""
    L = 260
    c = random_multi_case(52 + k, L, k)
    multi = O.decode_multi(c["qm"], c["relm"], c["kc"], c["vc"], c["table"],
                           c["seq_lens"], W, 64)
    for i in range(k):
        dec = O.decode(c["qm"][:, i], c["relm"][:, i], c["kc"], c["vc"], c["table"],
                       np.array([L - k + i + 1]), W, 64)
        np.testing.assert_allclose(multi[:, i], dec, atol=1e-13, rtol=0)


@pytest.mark.parametrize("L,k,W,E", [(9, 9, 0, 16), (200, 4, 0, 300), (200, 7, 64, 40),
                                     (260, 3, 100, 64)])
def test_decode_multi_equals_float64_sdpa(L, k, W, E):
    c = random_multi_case(60 + L + k, L, k, E=E, dv=6)
    out = O.decode_multi(c["qm"], c["relm"], c["kc"], c["vc"], c["table"],
                         c["seq_lens"], W, E)
    ref = sdpa_reference(c["qm"][0], c["Kc"], c["Vc"], c["relm"][0],
                         list(range(L - k, L)), W, E)
    np.testing.assert_allclose(out[0], ref, atol=1e-12, rtol=0)


def test_decode_multi_equals_prefill_of_the_same_tokens():
    """A verification step over k cached tokens equals a chunked prefill of
    those k tokens after the L - k cached before them."""
    L, k, Hq, Hkv, d, dv, E = 300, 6, 4, 2, 16, 8, 64
    for W in (0, 100):
        c = random_multi_case(72, L, k, Hq=Hq, Hkv=Hkv, d=d, dv=dv, E=E)
        multi = O.decode_multi(c["qm"], c["relm"], c["kc"], c["vc"], c["table"],
                               c["seq_lens"], W, E)
        newk = c["Kc"][L - k:L]
        newv = c["Vc"][L - k:L]
        pre, kc2, _ = O.prefill(c["qm"][0], newk, newv, c["relm"][0], [0, k], c["kc"], c["vc"],
                                c["table"], [L - k], W, E)
        assert np.array_equal(kc2, c["kc"])  # the same keys written back
        np.testing.assert_allclose(multi[0], pre, atol=1e-13, rtol=0)


# ---------------------------------------------------------------------------
# gated output with a sink
# ---------------------------------------------------------------------------

def test_sink_minus_inf_and_gate_plus_inf_are_the_plain_output():
    c = random_decode_case(81, 300)
    plain = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"], c["seq_lens"], 100, 64)
    Hq = c["q"].shape[1]
    sg = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"], c["seq_lens"], 100, 64,
                  sink=np.full((1, Hq), -np.inf), gate=np.full((1, Hq), np.inf))
    assert np.array_equal(sg, plain)


@pytest.mark.parametrize("n,s,gt", [(1, 0.0, 0.0), (7, 1.5, -0.7), (300, -2.0, 3.0)])
def test_sink_and_gate_closed_form(n, s, gt):
    """q = 0 and rel = 0 make all n visible logits 0: each weight is
    1 / (n + e^s), so out = (sum of the values) / (n + e^s) * sigmoid(g)."""
    c = random_decode_case(82 + n, n)
    q0 = np.zeros_like(c["q"])
    rel0 = np.zeros_like(c["rel"])
    Hq = q0.shape[1]
    out = O.decode(q0, rel0, c["kc"], c["vc"], c["table"], c["seq_lens"], 0, 64,
                   sink=np.full((1, Hq), s), gate=np.full((1, Hq), gt))
    g = Hq // c["Kc"].shape[1]
    for h in range(Hq):
        want = c["Vc"][:, h // g].sum(0) / (n + math.exp(s)) / (1 + math.exp(-gt))
        np.testing.assert_allclose(out[0, h], want, rtol=1e-12, atol=1e-14)


def test_sink_is_an_extra_key_with_a_zero_value():
    """The sink joins the normaliser like one more key whose logit is s and
    whose value is 0: float64 SDPA over the keys plus such a key."""
    L, W, E = 260, 100, 64
    c = random_decode_case(85, L, E=E, dv=6)
    Hq = c["q"].shape[1]
    s = np.linspace(-1.0, 2.0, Hq)[None, :]
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"], c["seq_lens"], W, E,
                   sink=s)
    # extended keys: the visible ones plus a zero key (q.k = 0) at the end
    P = L - 1
    lo, _ = O.visible_keys(P, W)
    keys = np.arange(lo, P + 1)
    d = c["Kc"].shape[2]
    g = Hq // c["Kc"].shape[1]
    for h in range(Hq):
        K = np.concatenate([c["Kc"][keys, h // g], np.zeros((1, d))])
        V = np.concatenate([c["Vc"][keys, h // g], np.zeros((1, c["Vc"].shape[2]))])
        bias = np.array([c["rel"][0, h, P - j] if P - j < E else 0.0 for j in keys] +
                        [s[0, h]])
        qt = torch.from_numpy(c["q"][0, h][None, None, :])
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, torch.from_numpy(K)[None], torch.from_numpy(V)[None],
            attn_mask=torch.from_numpy(bias)[None, None, :])
        np.testing.assert_allclose(out[0, h], o[0, 0].numpy(), atol=1e-12, rtol=0)


def test_gates_g_and_minus_g_sum_to_the_ungated_output():
    """sigmoid(g) + sigmoid(-g) = 1, for every row of a prefill."""
    wl_c = random_decode_case(86, 200)
    T, Hq = 40, 4
    r = rng(87)
    q = r.standard_normal((T, Hq, 16))
    k = r.standard_normal((T, 2, 16))
    v = r.standard_normal((T, 2, 8))
    rel = r.standard_normal((T, Hq, 64))
    gate = r.standard_normal((T, Hq)) * 3
    sink = r.standard_normal((T, Hq))
    args = (q, k, v, rel, [0, T], wl_c["kc"], wl_c["vc"], wl_c["table"], [150], 100, 64)
    a, _, _ = O.prefill(*args, sink=sink, gate=gate)
    b, _, _ = O.prefill(*args, sink=sink, gate=-gate)
    c, _, _ = O.prefill(*args, sink=sink)
    np.testing.assert_allclose(a + b, c, atol=1e-12, rtol=0)


def test_decode_multi_sink_gate_rows_equal_decode_at_their_lengths():
    L, k = 260, 3
    c = random_multi_case(88, L, k)
    Hq = c["qm"].shape[2]
    r = rng(89)
    sink = r.standard_normal((1, k, Hq))
    gate = r.standard_normal((1, k, Hq))
    multi = O.decode_multi(c["qm"], c["relm"], c["kc"], c["vc"], c["table"], c["seq_lens"],
                           64, 64, sink=sink, gate=gate)
    for i in range(k):
        dec = O.decode(c["qm"][:, i], c["relm"][:, i], c["kc"], c["vc"], c["table"],
                       np.array([L - k + i + 1]), 64, 64, sink=sink[:, i], gate=gate[:, i])
        np.testing.assert_allclose(multi[:, i], dec, atol=1e-13, rtol=0)


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache
# ---------------------------------------------------------------------------

def test_e4m3_decoder_against_torch_on_every_code():
    """All 256 patterns against torch's float8_e4m3fn (an independent
    implementation of the format); NaN patterns agree as NaN."""
    codes = np.arange(256, dtype=np.uint8)
    mine = O.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # a few values by hand: 1.0, the largest 448, the smallest subnormal 2^-9
    assert O.e4m3_bits_to_f64(np.array([0x38, 0x7E, 0x01, 0x80, 0xB8], dtype=np.uint8)).tolist() \
        == [1.0, 448.0, 2.0 ** -9, -0.0, -1.0]


def test_fp8_decode_equals_decode_of_the_dequantised_cache():
    """Reading the e4m3 cache with scales is the decode of the float cache
    holding scale * value, exactly."""
    c = random_decode_case(110, 300)
    r = rng(111)
    kc8 = r.integers(0, 256, size=c["kc"].shape, dtype=np.uint8)
    vc8 = r.integers(0, 256, size=c["vc"].shape, dtype=np.uint8)
    kc8[(kc8 & 0x7F) == 0x7F] = 0x38  # no NaN patterns in a cache
    vc8[(vc8 & 0x7F) == 0x7F] = 0x38
    ks, vs = 0.013, 0.7
    a = O.decode(c["q"], c["rel"], kc8, vc8, c["table"], c["seq_lens"], 100, 64,
                 k_scale=ks, v_scale=vs)
    b = O.decode(c["q"], c["rel"], O.e4m3_bits_to_f64(kc8) * ks, O.e4m3_bits_to_f64(vc8) * vs,
                 c["table"], c["seq_lens"], 100, 64)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# log-position scale
# ---------------------------------------------------------------------------

def test_logit_scale_of_one_is_the_plain_output():
    c = random_decode_case(120, 300)
    plain = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"], c["seq_lens"], 100, 64)
    one = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"], c["seq_lens"], 100, 64,
                   logit_scale=np.ones(1))
    assert np.array_equal(one, plain)


@pytest.mark.parametrize("W,E", [(0, 300), (100, 40)])
def test_logit_scale_is_q_and_rel_scaled_in_float64_sdpa(W, E):
    """Scaling q and the rel logits of each query token by its factor, then
    plain float64 SDPA, gives the prefill with per-token factors."""
    r = rng(121)
    ctx, n, Hq, Hkv, d, dv = 150, 90, 6, 2, 16, 8
    total = ctx + n
    nblk = (total + 127) // 128
    table = r.permutation(nblk + 1)[:nblk]
    Kc = r.standard_normal((total, Hkv, d))
    Vc = r.standard_normal((total, Hkv, dv))
    kc, vc = paged_from_contiguous(Kc[:ctx], Vc[:ctx], table, nblk + 1)
    q = r.standard_normal((n, Hq, d))
    rel = r.standard_normal((n, Hq, E))
    s = r.uniform(0.3, 3.0, n)
    out, _, _ = O.prefill(q, Kc[ctx:], Vc[ctx:], rel, [0, n], kc, vc, table[None, :], [ctx],
                          W, E, logit_scale=s)
    ref = sdpa_reference(q * s[:, None, None], Kc, Vc, rel * s[:, None, None],
                         [ctx + t for t in range(n)], W, E)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("n,sink", [(1, 0.5), (300, -1.0), (77, 2.0)])
def test_logit_scale_to_zero_gives_the_mean_and_leaves_the_sink_alone(n, sink):
    """A vanishing factor makes every key's logit 0 while the sink logit
    keeps its value: each weight tends to 1 / (n + e^sink)."""
    c = random_decode_case(122 + n, n)
    Hq = c["q"].shape[1]
    out = O.decode(c["q"], c["rel"], c["kc"], c["vc"], c["table"], c["seq_lens"], 0, 64,
                   sink=np.full((1, Hq), sink), logit_scale=np.array([1e-13]))
    g = Hq // c["Kc"].shape[1]
    for h in range(Hq):
        want = c["Vc"][:, h // g].sum(0) / (n + math.exp(sink))
        np.testing.assert_allclose(out[0, h], want, rtol=0, atol=1e-9)


def test_logit_scale_rows_agree_across_decode_multi_and_prefill():
    """Token i of a verification step with factor s_i equals a one-token
    decode at its length with that factor, and the last row of a prefill."""
    L, k = 260, 4
    c = random_multi_case(125, L, k)
    s = np.array([[0.5, 1.0, 1.7, 2.5]])
    multi = O.decode_multi(c["qm"], c["relm"], c["kc"], c["vc"], c["table"], c["seq_lens"],
                           64, 64, logit_scale=s)
    for i in range(k):
        dec = O.decode(c["qm"][:, i], c["relm"][:, i], c["kc"], c["vc"], c["table"],
                       np.array([L - k + i + 1]), 64, 64, logit_scale=s[:, i])
        np.testing.assert_allclose(multi[:, i], dec, atol=1e-13, rtol=0)
    pre, _, _ = O.prefill(c["qm"][0], c["Kc"][L - k:L], c["Vc"][L - k:L], c["relm"][0], [0, k],
                          c["kc"], c["vc"], c["table"], [L - k], 64, 64, logit_scale=s[0])
    np.testing.assert_allclose(multi[0], pre, atol=1e-13, rtol=0)


# ---------------------------------------------------------------------------
# e4m3 quantisation (the cache write into an e4m3 cache)
# ---------------------------------------------------------------------------

def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_bits_to_f64(codes)), codes)


def test_e4m3_encode_matches_torch_in_range():
    """torch's float32 -> float8_e4m3fn conversion (round to nearest even, an
    independent implementation) on random values inside +-448 and on values
    near every code."""
    r = rng(130)
    vals = O.e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))
    near = np.concatenate([vals * f for f in (0.999, 1.0, 1.001)] +
                          [(vals[:-1] + vals[1:]) / 2])
    x = np.concatenate([r.standard_normal(20000) * 30, r.uniform(-448, 448, 20000),
                        r.standard_normal(5000) * 1e-3, near, -near]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x.astype(np.float64)), ref)


def test_e4m3_encode_ties_go_to_the_even_code_and_large_values_saturate():
    vals = O.e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2          # between code i and i + 1
    want = np.arange(0x7E) + (np.arange(0x7E) % 2)  # the even one of the two
    assert np.array_equal(O.e4m3_encode(mids), want.astype(np.uint8))
    big = np.array([448.0, 463.9, 464.0, 500.0, 1e6, np.inf, -1e30, -np.inf])
    assert O.e4m3_encode(big).tolist() == [0x7E] * 6 + [0xFE] * 2


def test_e4m3_cache_write_is_within_half_a_step_of_the_scaled_values():
    """Quantising and reading back stays within half an e4m3 step of x / scale
    (relative 2^-4 for normal values, 2^-10 absolute below 2^-6), for values
    up to 448 scale, and every other slot is untouched."""
    r = rng(131)
    T, Hkv, d = 50, 2, 16
    k = O.f64_to_bf16_bits(r.standard_normal((T, Hkv, d)) * 3)
    v = O.f64_to_bf16_bits(r.standard_normal((T, Hkv, d)))
    ks, vs = float(np.abs(O.bf16_bits_to_f64(k)).max() / 448), 0.01
    kc = np.zeros((3, 128, Hkv, d), dtype=np.uint8)
    vc = np.zeros((3, 128, Hkv, d), dtype=np.uint8)
    table = np.array([[2, 0]])
    kc2, vc2 = O.kv_cache_write_e4m3(kc, vc, k, v, [0, T], [100], table, ks, vs)
    pos = 100 + np.arange(T)
    for cache, src, sc in ((kc2, k, ks), (vc2, v, vs)):
        got = O.e4m3_bits_to_f64(cache[table[0][pos // 128], pos % 128])
        x = np.clip(O.bf16_bits_to_f64(src) / sc, -448, 448)
        bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10)
        assert np.all(np.abs(got - x) <= bound + 1e-12)
    mask = np.ones(kc2.shape[:2], dtype=bool)
    mask[table[0][pos // 128], pos % 128] = False
    assert not kc2[mask].any() and not vc2[mask].any()


def test_e4m3_prefill_is_the_float_prefill_of_the_dequantised_tokens():
    """Prefill over an e4m3 cache = prefill over float caches holding the
    dequantised old entries, with the new tokens replaced by their quantised
    values read back (the write happens first, then the attention)."""
    r = rng(132)
    ctx, n, Hq, Hkv, d, W, E = 150, 90, 6, 2, 16, 100, 64
    nblk = (ctx + n + 127) // 128
    table = r.permutation(nblk + 1)[:nblk][None, :]
    kc8 = r.integers(0, 256, size=(nblk + 1, 128, Hkv, d), dtype=np.uint8)
    vc8 = r.integers(0, 256, size=(nblk + 1, 128, Hkv, d), dtype=np.uint8)
    kc8[(kc8 & 0x7F) == 0x7F] = 0x38
    vc8[(vc8 & 0x7F) == 0x7F] = 0x38
    q = r.standard_normal((n, Hq, d))
    k = O.f64_to_bf16_bits(r.standard_normal((n, Hkv, d)))
    v = O.f64_to_bf16_bits(r.standard_normal((n, Hkv, d)))
    rel = r.standard_normal((n, Hq, E))
    ks, vs = 0.02, 0.005
    out8, kc2, vc2 = O.prefill(q, k, v, rel, [0, n], kc8, vc8, table, [ctx], W, E,
                               k_scale=ks, v_scale=vs)
    kq = O.e4m3_bits_to_f64(O.e4m3_quantize(k, ks)) * ks
    vq = O.e4m3_bits_to_f64(O.e4m3_quantize(v, vs)) * vs
    outf, _, _ = O.prefill(q, kq, vq, rel, [0, n], O.e4m3_bits_to_f64(kc8) * ks,
                           O.e4m3_bits_to_f64(vc8) * vs, table, [ctx], W, E)
    np.testing.assert_allclose(out8, outf, atol=1e-13, rtol=0)
    # and a decode over the written cache is the prefill's last row
    dec = O.decode(q[-1:], rel[-1:], kc2, vc2, table, np.array([ctx + n]), W, E,
                   k_scale=ks, v_scale=vs)
    np.testing.assert_allclose(dec[0], out8[-1], atol=1e-13, rtol=0)
