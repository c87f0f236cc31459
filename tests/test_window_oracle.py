"""Pins for the oracle's sliding-window decode with attention sinks ([AP]
"Sparse attention: stop looking at everything"; [KVFA] eviction paragraph),
against numpy brute force and the special cases that reduce to plainer
results."""
import numpy as np

import oracle


def _brute(Q, K, V, scale, window, sinks):
    n, QL = K.shape[0], Q.shape[0]
    S = (Q @ K.T) * scale
    t = np.arange(n)[None, :]
    p = np.arange(n - QL, n)[:, None]
    vis = (t <= p) & ((window == 0) | (t >= p - window + 1) | (t < sinks))
    S = np.where(vis, S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return (E / E.sum(axis=1, keepdims=True)) @ V


def test_equals_brute_force_masks():
    rng = np.random.default_rng(21)
    for n, QL, w, s in [(50, 1, 16, 0), (50, 3, 16, 4), (100, 2, 33, 7), (40, 4, 64, 2),
                        (70, 1, 5, 5), (33, 8, 10, 0)]:
        Q, K, V = (rng.standard_normal((QL, 16)), rng.standard_normal((n, 16)),
                   rng.standard_normal((n, 16)))
        got = oracle.window_decode(Q, K, V, 0.25, w, s)
        assert np.allclose(got, _brute(Q, K, V, 0.25, w, s), rtol=0, atol=1e-12)


def test_special_cases():
    rng = np.random.default_rng(22)
    n, d = 30, 8
    Q, K, V = rng.standard_normal((3, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    full = oracle.multi_query_decode(Q, K, V, 0.3)
    # no window, a window covering everything, or sinks covering everything: full attention
    assert np.array_equal(oracle.window_decode(Q, K, V, 0.3, 0, 0), full)
    assert np.array_equal(oracle.window_decode(Q, K, V, 0.3, n, 0), full)
    assert np.array_equal(oracle.window_decode(Q, K, V, 0.3, 1, n), full)
    # a window of one and no sinks: each query sees only itself
    one = oracle.window_decode(Q, K, V, 0.3, 1, 0)
    assert np.array_equal(one, V[n - 3:])


def test_matches_library_sdpa_with_the_window_mask():
    """Against PyTorch's scaled_dot_product_attention in fp64 with the
    boolean mask built from positions (no numpy softmax involved)."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(23)
    for n, QL, w, s in [(200, 1, 64, 4), (200, 8, 17, 16), (90, 3, 1, 0), (130, 2, 500, 3)]:
        Q, K, V = (rng.standard_normal((QL, 32)), rng.standard_normal((n, 32)),
                   rng.standard_normal((n, 32)))
        t = torch.arange(n)[None, :]
        p = torch.arange(n - QL, n)[:, None]
        mask = (t <= p) & ((t >= p - w + 1) | (t < s))
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                             torch.from_numpy(V)[None], attn_mask=mask[None],
                                             scale=0.2)[0].numpy()
        got = oracle.window_decode(Q, K, V, 0.2, w, s)
        assert np.allclose(got, ref, rtol=0, atol=1e-12), (n, QL, w, s)
