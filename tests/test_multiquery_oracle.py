"""Pins for the oracle's multi-query decode (several new tokens of a sequence
attending at once, causal among themselves: [KVFA] speculative-decoding
section, where the target model scores the prefix and the drafted tokens in
one forward pass)."""
import numpy as np

import oracle


def _full_causal_rows(Q, K, V, scale):
    """Rows of full causal attention for queries at the last len(Q) positions,
    with numpy products and a written-out softmax (no oracle code)."""
    n, QL = K.shape[0], Q.shape[0]
    S = (Q @ K.T) * scale
    pos = np.arange(n - QL, n)[:, None]
    S = np.where(np.arange(n)[None, :] <= pos, S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return (E / E.sum(axis=1, keepdims=True)) @ V


def test_equals_full_causal_attention_rows():
    rng = np.random.default_rng(11)
    for n, QL, d in [(1, 1, 8), (5, 5, 16), (37, 4, 32), (100, 8, 64)]:
        Q = rng.standard_normal((QL, d))
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        got = oracle.multi_query_decode(Q, K, V, d ** -0.5)
        assert np.allclose(got, _full_causal_rows(Q, K, V, d ** -0.5), rtol=0, atol=1e-12)


def test_one_query_is_plain_decode():
    rng = np.random.default_rng(12)
    q, K, V = rng.standard_normal((1, 16)), rng.standard_normal((9, 16)), rng.standard_normal((9, 16))
    assert np.array_equal(oracle.multi_query_decode(q, K, V, 0.25)[0],
                          oracle.attend_row(q[0], K, V, 0.25))


def test_a_query_never_sees_later_tokens():
    rng = np.random.default_rng(13)
    n, QL, d = 20, 4, 8
    Q, K, V = rng.standard_normal((QL, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    base = oracle.multi_query_decode(Q, K, V, 0.3)
    K2, V2 = K.copy(), V.copy()
    K2[-1] += 5.0  # only the last query can see the last row
    V2[-1] -= 3.0
    moved = oracle.multi_query_decode(Q, K2, V2, 0.3)
    assert np.array_equal(moved[:-1], base[:-1])
    assert not np.allclose(moved[-1], base[-1])


def test_prefill_chunk_rows_match_library_sdpa():
    """The prefill reading of the same function (a long chunk of new rows at
    the end of a longer context, each row seeing positions 0 .. itself)
    against PyTorch's scaled_dot_product_attention with that mask, in fp64;
    both whole prompts (chunk = context) and chunks after a cached prefix."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(14)
    for n, QL, d in [(300, 120, 64), (257, 257, 32), (64, 1, 128), (513, 40, 16)]:
        Q = rng.standard_normal((QL, d))
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        scale = d ** -0.5
        pos = torch.arange(n - QL, n)[:, None]
        mask = torch.arange(n)[None, :] <= pos  # True: attend
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                             torch.from_numpy(V)[None], attn_mask=mask[None],
                                             scale=scale)[0].numpy()
        got = oracle.multi_query_decode(Q, K, V, scale)
        assert np.allclose(got, ref, rtol=0, atol=1e-12), (n, QL, d)


def test_chunk_attention_equals_the_row_definition():
    """chunk_attention (library products over the whole chunk) against
    multi_query_decode (each row the C definition) and against PyTorch's
    scaled_dot_product_attention with the causal-at-the-end mask."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(15)
    for n, QL, d in [(1, 1, 8), (300, 120, 64), (257, 257, 32), (513, 40, 16), (96, 5, 128)]:
        Q = rng.standard_normal((QL, d)) * 2.0
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        scale = d ** -0.5
        got = oracle.chunk_attention(Q, K, V, scale)
        assert np.allclose(got, oracle.multi_query_decode(Q, K, V, scale), rtol=0, atol=1e-12)
        pos = torch.arange(n - QL, n)[:, None]
        mask = torch.arange(n)[None, :] <= pos
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                             torch.from_numpy(V)[None], attn_mask=mask[None],
                                             scale=scale)[0].numpy()
        assert np.allclose(got, ref, rtol=0, atol=1e-12), (n, QL, d)
