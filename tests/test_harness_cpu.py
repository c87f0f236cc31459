"""The whole-output oracle helpers of the harness (one sequence, every head
at once, through decode_attention) against the oracle's per-row functions
they regroup: attend_row via oracle_rows, multi_query_decode and
window_decode.  Small seeded workloads on the CPU; no GPU."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_250_gb300 import workloads as wl
from harness import logical_kv_fp64, oracle_multi_seq, oracle_rows, oracle_whole, seq_kv_fp64


@pytest.mark.parametrize("cache", ["bf16", "e4m3", "e4m3tok"])
def test_oracle_whole_equals_rows(cache):
    cfg = wl.small_config(f"whole_{cache}", 4, 8, 2, 64, cache, (0, 70), seed=61)
    w = wl.generate(cfg)
    got = oracle_whole(w)
    ref = oracle_rows(w, [(b, hq) for b in range(cfg.batch) for hq in range(cfg.q_heads)])
    for (b, hq), r in ref.items():
        if int(w.ctx[b]) == 0:
            assert not got[b, hq].any()
        else:
            np.testing.assert_allclose(got[b, hq], r, rtol=0, atol=1e-12)


def test_seq_kv_stacks_heads_in_order():
    cfg = wl.small_config("stack", 2, 8, 4, 64, "e4m3", 40, seed=62)
    w = wl.generate(cfg)
    K, V = seq_kv_fp64(w, 1)
    for h in range(cfg.kv_heads):
        k, v = logical_kv_fp64(w, 1, h)
        assert np.array_equal(K[:, h], k) and np.array_equal(V[:, h], v)


@pytest.mark.parametrize("QL,window,sinks", [(1, 0, 0), (4, 0, 0), (5, 0, 0), (3, 7, 2),
                                             (4, 20, 0), (2, 5, 9), (8, 16, 4)])
def test_oracle_multi_seq_equals_per_head(QL, window, sinks):
    rng = np.random.default_rng(QL * 100 + window)
    n, Hkv, g, d = 37, 2, 4, 32
    q = rng.standard_normal((QL, Hkv * g, d))
    K = rng.standard_normal((n, Hkv, d))
    V = rng.standard_normal((n, Hkv, d))
    got = oracle_multi_seq(q, K, V, 0.2, window, sinks)
    for hq in range(Hkv * g):
        Kh, Vh = K[:, hq // g], V[:, hq // g]
        if window == 0:
            ref = oracle.multi_query_decode(q[:, hq], Kh, Vh, 0.2)
        else:
            ref = oracle.window_decode(q[:, hq], Kh, Vh, 0.2, window, sinks)
        np.testing.assert_allclose(got[:, hq], ref, rtol=0, atol=1e-12)
