"""Pins for the oracle's block copy (copy-on-write for shared prefixes).

[AP] "Paged attention: stop reserving empty tables": sequences point at the
same physical blocks for a shared beginning, copying only if one of them
would change a block.  [KVFA] PagedAttention section: sharing a prefix hands
the second sequence ceil(prefix / P) of the same blocks, so the last one may
be partly filled.  The checks below use numpy indexing only, never the
oracle's own arithmetic.
"""
import numpy as np

import oracle

P = 16


def test_copy_equals_fancy_indexing_and_skips_bad_ids():
    rng = np.random.default_rng(5)
    cache = rng.integers(0, 1 << 16, size=(12, 3, P, 8), dtype=np.uint16)
    src = np.array([2, 9, 11, -1, 4, 3], dtype=np.int32)
    dst = np.array([5, 0, 7, 6, 12, 3], dtype=np.int32)  # -1 and 12 are outside
    got = oracle.copy_blocks(cache, src, dst)
    want = cache.copy()
    for s, d in zip(src, dst):
        if 0 <= s < 12 and 0 <= d < 12:
            want[d] = want[s]
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.copy_blocks(cache, [], []), cache)


def test_copy_on_write_keeps_both_sequences_intact():
    # sequence A: a 40-token prompt in blocks 3, 8, 1 (block 1 holds 8 tokens)
    # sequence B shares that prefix, then both append one token each
    rng = np.random.default_rng(6)
    Hkv, d, NB = 2, 8, 10
    prefix = rng.integers(0, 1 << 16, size=(40, Hkv, d), dtype=np.uint16)
    a_new = rng.integers(0, 1 << 16, size=(1, Hkv, d), dtype=np.uint16)
    b_new = rng.integers(0, 1 << 16, size=(1, Hkv, d), dtype=np.uint16)
    table_a = [3, 8, 1]
    cache = np.zeros((NB, Hkv, P, d), dtype=np.uint16)
    for t in range(40):
        cache[table_a[t // P], :, t % P] = prefix[t]
    table_b = list(table_a)  # shared: the third block is only partly filled
    # B's token would land in the shared third block: copy it to block 6 first
    cache = oracle.copy_blocks(cache, [table_b[2]], [6])
    table_b[2] = 6
    cache = oracle.append_bytes(cache, a_new, [table_a[2] * P + 8])
    cache = oracle.append_bytes(cache, b_new, [table_b[2] * P + 8])

    def gather(table, n):
        return np.stack([cache[table[t // P], :, t % P] for t in range(n)])

    assert np.array_equal(gather(table_a, 41), np.concatenate([prefix, a_new]))
    assert np.array_equal(gather(table_b, 41), np.concatenate([prefix, b_new]))
