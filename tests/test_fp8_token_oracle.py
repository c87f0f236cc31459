"""Pins for the oracle's per-token FP8 (E4M3) scaling: one fp32 scale per
(token, KV head) row, the row's largest magnitude over 448.

"KV Cache & Flash Attention." (kvcache-7e2.pages.dev), memory-cost section
(the cache is quantized to fp8) and Flash Attention section (FP8 with
finer-grained scales).  The E4M3 values below are built from the format's
definition (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, S.1111.111 = NaN), not from the oracle's codec."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _e4m3_values() -> np.ndarray:
    """Every finite non-negative E4M3 value, from the format's definition."""
    vals = [m / 8 * 2.0 ** -6 for m in range(8)]                      # subnormals
    vals += [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8)
             if not (e == 15 and m == 7)]                             # normals, NaN excluded
    return np.array(sorted(set(vals)))


def test_value_table_closed_form():
    v = _e4m3_values()
    assert v.max() == 448.0 and len(v) == 127        # 0, 7 subnormals, 119 normals
    assert v[1] == 2.0 ** -9                         # smallest subnormal


def test_rows_of_scaled_e4m3_values_round_trip_exactly():
    """A row c * 2^k, c E4M3 values with max |c| = 448, has scale exactly 2^k
    and its codes reproduce c: dequantised == row, bit for bit."""
    rng = np.random.default_rng(31)
    table = _e4m3_values()
    for k in (-12, -3, 0, 5):
        c = rng.choice(table, size=(6, 64)) * rng.choice([-1.0, 1.0], size=(6, 64))
        c[:, 7] = 448.0 * rng.choice([-1.0, 1.0], size=6)
        rows = (c * 2.0 ** k).astype(np.float32)
        scales = np.array([oracle.e4m3_token_scale(r) for r in rows], dtype=np.float32)
        assert np.all(scales == np.float32(2.0 ** k))
        codes = np.stack([oracle.e4m3_quantize(r, s) for r, s in zip(rows, scales)])
        back = oracle.e4m3_dequantize_rows(codes, scales)
        assert np.array_equal(back, rows.astype(np.float64))


def test_largest_element_lands_on_448_and_zero_rows():
    rng = np.random.default_rng(32)
    rows = (rng.standard_normal((50, 128)) * np.exp(rng.uniform(-8, 8, (50, 1)))).astype(np.float32)
    for r in rows:
        s = oracle.e4m3_token_scale(r)
        codes = oracle.e4m3_quantize(r, s)
        j = int(np.argmax(np.abs(r)))
        assert codes[j] in (0x7E, 0xFE)                # +-448
        assert 0x7F not in codes and 0xFF not in codes  # no NaN code from finite input
    z = np.zeros(128, dtype=np.float32)
    assert oracle.e4m3_token_scale(z) == 1.0
    assert not oracle.e4m3_quantize(z, 1.0).any()


def test_error_within_half_an_e4m3_step():
    """|dequantised - x| <= 2^-4 |x| (3 mantissa bits, round to nearest) for
    normal codes, <= 2^-10 s in the subnormal range (step 2^-9 s)."""
    rng = np.random.default_rng(33)
    rows = (rng.standard_t(3, (200, 128)) * np.exp(rng.uniform(-5, 5, (200, 1)))).astype(np.float32)
    for r in rows:
        s = oracle.e4m3_token_scale(r)
        back = oracle.e4m3_dequantize_rows(oracle.e4m3_quantize(r, s)[None], [s])[0]
        x = r.astype(np.float64)
        bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s) * (1 + 1e-6)
        assert np.all(np.abs(back - x) <= bound)


def test_scale_follows_powers_of_two():
    rng = np.random.default_rng(34)
    r = rng.standard_normal(128).astype(np.float32)
    s = oracle.e4m3_token_scale(r)
    c = oracle.e4m3_quantize(r, s)
    for k in (-7, 3, 11):
        r2 = (r * np.float32(2.0 ** k)).astype(np.float32)
        s2 = oracle.e4m3_token_scale(r2)
        assert s2 == np.float32(s * 2.0 ** k)
        assert np.array_equal(oracle.e4m3_quantize(r2, s2), c)


def test_append_places_codes_and_scales():
    """One token per call: the per-token append of head h equals the per-head
    append with that head's scale set to the row's own scale; the scale goes
    to the same (block, head, offset) of the scale pool; nothing else moves."""
    rng = np.random.default_rng(35)
    NB, Hkv, P, d = 5, 3, 16, 32
    cache = rng.integers(0, 255, (NB, Hkv, P, d)).astype(np.uint8)
    scales = rng.standard_normal((NB, Hkv, P)).astype(np.float32)
    src = (rng.standard_normal((1, Hkv, d)) * [[[0.01]], [[3.0]], [[200.0]]]).astype(np.float32)
    slot = [3 * P + 9]
    got_c, got_s = oracle.append_e4m3_token(cache, scales, src, slot)
    hs = np.array([oracle.e4m3_token_scale(src[0, h]) for h in range(Hkv)], dtype=np.float32)
    want_c = oracle.append_e4m3(cache, src, slot, hs)
    assert np.array_equal(got_c, want_c)
    want_s = scales.copy()
    want_s[3, :, 9] = hs
    assert np.array_equal(got_s, want_s)
    # a negative slot skips the token
    c2, s2 = oracle.append_e4m3_token(cache, scales, src, [-1])
    assert np.array_equal(c2, cache) and np.array_equal(s2, scales)


def test_per_token_scales_beat_one_head_scale_next_to_an_outlier():
    """The point of finer scales: with one huge token in the head, a single
    head scale flushes the ordinary tokens toward zero; per-token scales keep
    them within the E4M3 step."""
    rng = np.random.default_rng(36)
    rows = rng.standard_normal((64, 128)).astype(np.float32)
    rows[10] *= 1.0e6  # ordinary tokens fall below the smallest E4M3 step of one head scale
    head_s = float(np.float32(np.abs(rows).max()) / np.float32(448.0))
    err_head = np.abs(oracle.e4m3_dequantize(oracle.e4m3_quantize(rows, head_s), head_s) - rows)
    tok_s = np.array([oracle.e4m3_token_scale(r) for r in rows], dtype=np.float32)
    codes = np.stack([oracle.e4m3_quantize(r, s) for r, s in zip(rows, tok_s)])
    err_tok = np.abs(oracle.e4m3_dequantize_rows(codes, tok_s) - rows)
    ordinary = np.arange(64) != 10
    assert err_tok[ordinary].max() < 0.2 * err_head[ordinary].max()
    assert err_tok[ordinary].mean() < 0.1 * err_head[ordinary].mean()
