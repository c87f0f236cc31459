"""Pins for the CPU oracle (no GPU).

Each test fixes an oracle function to something other than itself: numbers
the pages print (fixtures under tests/golden/, each with its citation),
closed forms, special cases with a textbook answer, brute force on tiny
inputs, and independent library routines (torch's scaled-dot-product
attention in fp64, torch's float8_e4m3fn cast).  Several tests plant a
plausible mistake in a copy of the oracle's inputs or outputs and check that
the pin notices it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------- I1: sizes
def test_bytes_per_token_matches_printed_values():
    for case in _golden("kv_cache_sizes.json")["bytes_per_token"]:
        got = oracle.kv_bytes_per_token(case["layers"], case["kv_heads"],
                                        case["head_dim"], case["elem_bytes"])
        assert got == case["bytes"], case["cite"]


def test_cache_table_at_32k_tokens():
    for case in _golden("kv_cache_sizes.json")["gib_at_32000_tokens"]:
        gib = oracle.kv_bytes(32000, case["layers"], case["kv_heads"],
                              case["head_dim"]) / 1024**3
        assert round(gib, 2) == case["expected"], case["cite"]
        if case["printed"] != case["expected"]:
            # the garbled row: the page's figure really is not what its shape gives
            assert round(gib, 2) != case["printed"]


def test_whole_cache_examples():
    g = _golden("kv_cache_sizes.json")
    for case in g["whole_cache"]:
        got = oracle.kv_bytes(case["tokens"], case["layers"], case["kv_heads"],
                              case["head_dim"], case["elem_bytes"])
        assert got == case["bytes"], case["cite"]
    c = g["conversations_in_10GB"]
    per = oracle.kv_bytes(c["tokens"], c["layers"], c["kv_heads"], c["head_dim"],
                          c["elem_bytes"])
    assert c["budget_bytes"] // per == c["fits"], c["cite"]


def test_fp8_and_gqa_reductions():
    g = _golden("kv_cache_sizes.json")
    f = g["fp8_halves"]
    b16 = oracle.kv_bytes(f["tokens"], f["layers"], f["kv_heads"], f["head_dim"], 2)
    b8 = oracle.kv_bytes(f["tokens"], f["layers"], f["kv_heads"], f["head_dim"], 1)
    assert b16 == f["ratio_fp16_over_fp8"] * b8
    assert 9.5 < b16 / 1024**3 < 10.0 and 4.5 < b8 / 1024**3 < 5.0
    q = g["gqa_plus_fp8"]
    mha = oracle.kv_bytes_per_token(32, q["mha_kv_heads"], 128, 2)
    gqa8 = oracle.kv_bytes_per_token(32, q["gqa_kv_heads"], 128, 1)
    assert mha == q["ratio"] * gqa8


def test_bytes_formula_linear_in_every_factor():
    base = oracle.kv_bytes(7, 3, 5, 11, 2, 13)
    assert base == 2 * 7 * 3 * 5 * 11 * 2 * 13
    for i in range(6):
        args = [7, 3, 5, 11, 2, 13]
        args[i] *= 2
        assert oracle.kv_bytes(*args) == 2 * base


# --------------------------------------------------------------- I2: counts
def test_decode_work_counts():
    for case in _golden("decode_work_counts.json")["cases"]:
        rec = oracle.rows_recomputed(case["prompt"], case["n_new"])
        cac = oracle.rows_cached(case["prompt"], case["n_new"])
        assert rec == case["recomputed"], case["cite"]
        assert cac == case["cached"], case["cite"]
        if "printed_recomputed_approx" in case:
            assert abs(rec - case["printed_recomputed_approx"]) / rec < 0.01
        if "printed_lower_bound" in case:
            assert rec > case["printed_lower_bound"]
        if case["prompt"] == 0:
            n = case["n_new"]
            assert rec == n * (n + 1) // 2  # triangular number


# --------------------------------------------------------------- I3: cache
@pytest.mark.parametrize("n_tokens,d", [(6, 16), (100, 16), (37, 8)])
def test_cached_decode_equals_recompute(n_tokens, d):
    rng = np.random.default_rng(0)
    Wq, Wk, Wv = (rng.standard_normal((d, d)) / math.sqrt(d) for _ in range(3))
    X = rng.standard_normal((n_tokens, d))
    scale = 1.0 / math.sqrt(d)
    outs, rows = oracle.cached_decode(X, Wq, Wk, Wv, scale)
    assert rows == n_tokens
    for t in range(1, n_tokens + 1):
        ref = oracle.causal_attention_last_row(X[:t], Wq, Wk, Wv, scale)
        np.testing.assert_allclose(outs[t - 1], ref, rtol=0, atol=1e-12)


def test_cached_decode_detects_off_by_one_context():
    # Planted mistake: attending before appending (context excludes the new
    # token) gives a different answer, so the pin above would catch it.
    rng = np.random.default_rng(1)
    d = 16
    Wq, Wk, Wv = (rng.standard_normal((d, d)) / 4 for _ in range(3))
    X = rng.standard_normal((6, d))
    t = 5
    K = X[: t - 1] @ Wk
    V = X[: t - 1] @ Wv
    wrong = oracle.attend_row(X[t - 1] @ Wq, K, V, 0.25)
    ref = oracle.causal_attention_last_row(X[:t], Wq, Wk, Wv, 0.25)
    assert np.abs(wrong - ref).max() > 1e-3


# --------------------------------------------------------------- attention
def _sdpa_fp64(q, K, V, ctx, scale):
    """torch SDPA (library routine) per sequence, fp64, GQA by expansion."""
    B, Hq, d = q.shape
    Hkv = K.shape[2]
    g = Hq // Hkv
    out = np.zeros_like(q)
    for b in range(B):
        n = int(ctx[b])
        if n == 0:
            continue
        qt = torch.from_numpy(q[b]).unsqueeze(1)  # [Hq,1,d]
        kt = torch.from_numpy(K[b, :n]).permute(1, 0, 2).repeat_interleave(g, 0)
        vt = torch.from_numpy(V[b, :n]).permute(1, 0, 2).repeat_interleave(g, 0)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt,
                                                             scale=scale)
        out[b] = o[:, 0].numpy()
    return out


@pytest.mark.parametrize("B,Hq,Hkv,d,T", [(3, 8, 2, 32, 40), (2, 4, 4, 16, 17),
                                         (2, 6, 1, 8, 9)])
def test_decode_attention_matches_library_sdpa(B, Hq, Hkv, d, T):
    rng = np.random.default_rng(B * 100 + Hq)
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, T, Hkv, d))
    V = rng.standard_normal((B, T, Hkv, d))
    ctx = rng.integers(1, T + 1, size=B).astype(np.int32)
    scale = 1 / math.sqrt(d)
    got = oracle.decode_attention(q, K, V, ctx, scale)
    ref = _sdpa_fp64(q, K, V, ctx, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_sdpa_pin_catches_planted_mistakes():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, d, T = 2, 8, 2, 16, 20
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, T, Hkv, d))
    V = rng.standard_normal((B, T, Hkv, d))
    ctx = np.array([20, 13], dtype=np.int32)
    ref = _sdpa_fp64(q, K, V, ctx, 0.25)
    # wrong head grouping (hq % Hkv instead of hq // g)
    Kw = K[:, :, [0, 1], :]
    bad = np.zeros_like(ref)
    for b in range(B):
        for hq in range(Hq):
            kv = hq % Hkv
            bad[b, hq] = oracle.attend_row(q[b, hq], Kw[b, :ctx[b], kv],
                                           V[b, :ctx[b], kv], 0.25)
    assert np.abs(bad - ref).max() > 1e-3
    # dropped scale
    assert np.abs(oracle.decode_attention(q, K, V, ctx, 1.0) - ref).max() > 1e-3
    # context off by one (the appended token left out)
    assert np.abs(oracle.decode_attention(q, K, V, ctx - 1, 0.25) - ref).max() > 1e-3


def test_context_one_returns_the_value_row_exactly():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 4, 64))
    K = rng.standard_normal((1, 5, 1, 64))
    V = rng.standard_normal((1, 5, 1, 64))
    out = oracle.decode_attention(q, K, V, np.array([1], np.int32), 0.125)
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, 0, 0])


def test_equal_scores_give_mean_of_values():
    rng = np.random.default_rng(3)
    n, d = 37, 16
    q = rng.standard_normal(d)
    K = np.tile(rng.standard_normal(d), (n, 1))  # identical keys
    V = rng.standard_normal((n, d))
    np.testing.assert_allclose(oracle.attend_row(q, K, V, 0.3), V.mean(0),
                               rtol=0, atol=1e-14)
    # scale 0 also makes every score equal
    K2 = rng.standard_normal((n, d))
    np.testing.assert_allclose(oracle.attend_row(q, K2, V, 0.0), V.mean(0),
                               rtol=0, atol=1e-14)


def test_two_token_closed_form():
    # softmax over two scores is the logistic function of their difference
    q = np.array([1.0, 2.0, -1.0])
    K = np.array([[0.5, 0.0, 1.0], [1.0, 1.0, 0.0]])
    V = np.array([[1.0, 0.0, 2.0], [-1.0, 3.0, 0.5]])
    scale = 0.7
    s0, s1 = scale * (q @ K[0]), scale * (q @ K[1])
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * V[0] + (1 - w0) * V[1]
    np.testing.assert_allclose(oracle.attend_row(q, K, V, scale), expect,
                               rtol=0, atol=1e-15)


def test_sign_and_sharpness():
    # a large positive scale selects the value of the best-aligned key,
    # not the worst (a sign error would pick the minimum)
    rng = np.random.default_rng(4)
    n, d = 12, 8
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    out = oracle.attend_row(q, K, V, 200.0)
    best = int(np.argmax(K @ q))
    np.testing.assert_allclose(out, V[best], atol=1e-6)


def test_gqa_head_mapping_is_consecutive():
    B, Hq, Hkv, d, T = 1, 12, 3, 4, 5
    q = np.ones((B, Hq, d))
    K = np.zeros((B, T, Hkv, d))
    V = np.zeros((B, T, Hkv, d))
    for h in range(Hkv):
        V[0, :, h, :] = h + 1.0
    out = oracle.decode_attention(q, K, V, np.array([T], np.int32), 1.0)
    g = Hq // Hkv
    for hq in range(Hq):
        assert np.all(out[0, hq] == hq // g + 1.0)


def test_token_order_invariance_and_empty_context():
    rng = np.random.default_rng(6)
    n, d = 50, 16
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    perm = rng.permutation(n)
    np.testing.assert_allclose(oracle.attend_row(q, K, V, 0.25),
                               oracle.attend_row(q, K[perm], V[perm], 0.25),
                               rtol=0, atol=1e-14)
    out = oracle.decode_attention(np.ones((1, 2, 4)), np.ones((1, 3, 1, 4)),
                                  np.ones((1, 3, 1, 4)), np.array([0], np.int32), 1.0)
    assert np.all(out == 0.0)


def test_no_overflow_for_large_scores():
    q = np.array([100.0])
    K = np.array([[10.0], [9.0]])
    V = np.array([[1.0], [0.0]])
    out = oracle.attend_row(q, K, V, 1.0)  # scores 1000 and 900
    assert np.isfinite(out).all() and abs(out[0] - 1.0) < 1e-40 + 1e-15


# --------------------------------------------------------------- I4: online
def test_online_softmax_worked_example():
    g = _golden("online_softmax_worked_example.json")
    m, l, mt, lt = oracle.online_softmax_stats(g["scores"], g["tile"])
    dec = g["printed_decimals"]
    assert mt[0] == g["after_tile_1"]["m"]
    assert round(lt[0], dec) == g["after_tile_1"]["l_printed"]
    factor = math.exp(mt[0] - mt[1])
    assert round(factor, dec) == g["rescale_factor_printed"]
    assert round(lt[0] * factor, dec) == g["rescaled_l_printed"]
    assert round(lt[1] - lt[0] * factor, dec) == g["tile_2_sum_printed"]
    assert m == g["final"]["m"] and round(l, dec) == g["final"]["l_printed"]
    # and the exact identity the page states: e^-2 + e^-1 + e^0 + e^-3
    assert abs(l - (math.exp(-2) + math.exp(-1) + 1 + math.exp(-3))) < 1e-15


@pytest.mark.parametrize("tile", [1, 2, 3, 16, 1000])
def test_online_softmax_equals_two_pass(tile):
    rng = np.random.default_rng(tile)
    for n in (1, 7, 64, 257):
        x = rng.standard_normal(n) * 5
        m, l, _, _ = oracle.online_softmax_stats(x, tile)
        assert m == x.max()
        l2 = np.exp(x - x.max()).sum()
        assert abs(l - l2) <= 1e-15 * l2 * 4


@pytest.mark.parametrize("tile", [1, 5, 16, 64])
def test_online_attention_equals_definition(tile):
    rng = np.random.default_rng(10 + tile)
    n, d = 123, 32
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    out, m, l, o = oracle.online_attend_row(q, K, V, 0.2, tile)
    np.testing.assert_allclose(out, oracle.attend_row(q, K, V, 0.2), rtol=0,
                               atol=1e-14)
    s = 0.2 * (K @ q)
    assert m == pytest.approx(s.max(), abs=1e-14)
    assert l == pytest.approx(np.exp(s - s.max()).sum(), rel=1e-14)


def test_merge_of_any_partition_equals_unsplit():
    rng = np.random.default_rng(11)
    n, d = 200, 16
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    ref = oracle.attend_row(q, K, V, 0.3)
    for _ in range(5):
        cuts = np.sort(rng.choice(np.arange(1, n), size=rng.integers(1, 9),
                                  replace=False))
        bounds = [0, *cuts.tolist(), n]
        ms, ls, os_ = [], [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            _, m, l, o = oracle.online_attend_row(q, K[a:b], V[a:b], 0.3, 16)
            ms.append(m), ls.append(l), os_.append(o)
        # an empty split (no tokens) must contribute nothing
        ms.append(-math.inf), ls.append(0.0), os_.append(np.zeros(d))
        got = oracle.merge_partials(ms, ls, np.stack(os_))
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)
    assert np.all(oracle.merge_partials([-math.inf], [0.0], np.zeros((1, d))) == 0)


def test_merge_pin_catches_missing_rescale():
    # planted mistake: adding partial outputs without the exp(m_i - M) factor
    rng = np.random.default_rng(12)
    d = 8
    q = rng.standard_normal(d) * 3
    K = rng.standard_normal((40, d))
    V = rng.standard_normal((40, d))
    ref = oracle.attend_row(q, K, V, 1.0)
    _, m1, l1, o1 = oracle.online_attend_row(q, K[:20], V[:20], 1.0, 8)
    _, m2, l2, o2 = oracle.online_attend_row(q, K[20:], V[20:], 1.0, 8)
    naive = (o1 + o2) / (l1 + l2)
    assert m1 != m2 and np.abs(naive - ref).max() > 1e-3


# --------------------------------------------------------------- fp8 codec
def test_e4m3_decode_known_codes():
    assert oracle.e4m3_decode(0x00) == 0.0
    assert math.copysign(1, oracle.e4m3_decode(0x80)) == -1.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9          # smallest subnormal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6          # smallest normal
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x39) == 1.125
    assert oracle.e4m3_decode(0x40) == 2.0
    assert oracle.e4m3_decode(0x7E) == 448.0              # largest finite
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert math.isnan(oracle.e4m3_decode(0x7F))
    assert math.isnan(oracle.e4m3_decode(0xFF))
    assert oracle.e4m3_decode(0x78) == 256.0              # e=15, m=0 is finite


def test_e4m3_decode_table_structure():
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert vals == sorted(vals) and len(set(vals)) == 127  # 0 + 126 positives
    for c in range(0x80):
        v = oracle.e4m3_decode(c)
        n = oracle.e4m3_decode(c | 0x80)
        assert (math.isnan(v) and math.isnan(n)) or n == -v


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


def test_e4m3_encode_round_trip_and_ties():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        back = oracle.e4m3_encode(v)
        assert back == c or (v == 0.0 and back in (0x00, 0x80) and
                             (back >> 7) == (c >> 7))
    # ties go to the even mantissa
    assert oracle.e4m3_encode(1.0625) == 0x38   # between 1.0 and 1.125
    assert oracle.e4m3_encode(1.1875) == 0x3A   # between 1.125 and 1.25
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02
    # saturation (satfinite) and NaN
    assert oracle.e4m3_encode(449.0) == 0x7E
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F


def test_e4m3_encode_matches_torch_cast_in_range():
    # every finite bf16 value with |x| <= 448: torch's RNE cast is the library pin
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float32)
    keep = torch.isfinite(x) & (x.abs() <= 448)
    xs = x[keep]
    ref = xs.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_quantize(xs.numpy(), 1.0)
    zero = xs.numpy() == 0
    assert np.array_equal(got[~zero], ref[~zero])
    assert np.all((got[zero] & 0x7F) == 0)


def test_e4m3_quantize_divides_in_fp32():
    x = np.array([0.3, -1.7, 5.0, 1000.0], dtype=np.float32)
    s = np.float32(0.01171875)
    got = oracle.e4m3_quantize(x, s)
    for xi, gi in zip(x, got):
        assert gi == oracle.e4m3_encode(float(np.float32(xi) / s))


# --------------------------------------------------------------- append
def test_append_bytes_places_rows_by_slot():
    NB, Hkv, P, d = 4, 2, 4, 3
    cache = np.full((NB, Hkv, P, d), 7, dtype=np.uint16)
    src = np.arange(3 * Hkv * d, dtype=np.uint16).reshape(3, Hkv, d)
    slot = np.array([5, -1, 14])  # block 1 offset 1; skipped; block 3 offset 2
    out = oracle.append_bytes(cache, src, slot)
    assert np.array_equal(out[1, :, 1], src[0])
    assert np.array_equal(out[3, :, 2], src[2])
    changed = (out != cache).any(axis=-1)
    assert changed.sum() == 2 * Hkv - (src[0] == 7).all() - (src[2] == 7).all()
    mask = np.ones((NB, P), bool)
    mask[1, 1] = mask[3, 2] = False
    assert np.array_equal(out.transpose(0, 2, 1, 3)[mask],
                          cache.transpose(0, 2, 1, 3)[mask])


def test_append_e4m3_uses_head_scale():
    NB, Hkv, P, d = 2, 2, 2, 4
    cache = np.zeros((NB, Hkv, P, d), np.uint8)
    src = np.array([[[1.0, 2.0, -3.0, 0.5], [1.0, 2.0, -3.0, 0.5]]], np.float32)
    out = oracle.append_e4m3(cache, src, [3], [1.0, 0.5])
    assert list(out[1, 0, 1]) == [oracle.e4m3_encode(v) for v in src[0, 0]]
    assert list(out[1, 1, 1]) == [oracle.e4m3_encode(2 * v) for v in src[0, 1]]
