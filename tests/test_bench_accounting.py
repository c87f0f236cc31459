"""The bench's accounting, checked on the CPU: the visible-position count of
the windowed line and the causal flops of the prefill line against brute
force, and the algorithmic bytes against the figures recorded beside the
committed ncu captures (which the reported DRAM traffic is compared with).

"KV Cache & Flash Attention." (kvcache-7e2.pages.dev): eviction paragraph
(a window of recent positions plus the first ones) and the prefill phase;
"Sparse attention: stop looking at everything" for the window."""
import json
import os

import numpy as np
import pytest
import torch

import bench
from paged_kv_cache_250_gb300 import workloads as wl


def _seen_brute(n: int, qlen: int, window: int, sinks: int) -> int:
    """Positions t < n that at least one new token sees: token j sits at
    n - qlen + j (tokens before position 0 see nothing) and sees t <= its
    position with t inside its last `window` positions or t < sinks."""
    seen = set()
    for j in range(qlen):
        p = n - qlen + j
        for t in range(0, p + 1):
            if window <= 0 or t >= p - window + 1 or t < sinks:
                seen.add(t)
    return len(seen)


def test_visible_tokens_brute_force():
    rng = np.random.default_rng(11)
    cases = [(0, 1, 4, 2), (1, 1, 1, 0), (5, 8, 3, 1), (100, 2, 1, 0), (100, 1, 100, 4),
             (300, 4, 16, 300), (64, 3, 0, 5)]
    cases += [(int(rng.integers(0, 400)), int(rng.integers(1, 9)), int(rng.integers(0, 120)),
               int(rng.integers(0, 40))) for _ in range(60)]
    for n, qlen, window, sinks in cases:
        got = bench.visible_tokens(torch.tensor([n]), qlen, window, sinks)
        assert got == _seen_brute(n, qlen, window, sinks), (n, qlen, window, sinks)
    ctx = torch.tensor([n for n, *_ in cases[:10]])
    assert bench.visible_tokens(ctx, 2, 16, 3) == sum(_seen_brute(int(n), 2, 16, 3) for n in ctx)


def test_prefill_flops_brute_force():
    """4 d flops (q.k and p.v) per query head for every (row, visible
    position) pair; a chunk longer than the context covers the whole of it."""
    rng = np.random.default_rng(12)
    for _ in range(20):
        ctx = torch.tensor(rng.integers(1, 700, size=int(rng.integers(1, 5))).tolist())
        chunk, Hq, d = int(rng.integers(1, 800)), int(rng.choice([4, 32])), int(rng.choice([64, 128]))
        pairs = 0
        for n in ctx.tolist():
            for p in range(max(0, n - chunk), n):  # the chunk's rows are the last positions
                pairs += p + 1                      # row at position p sees 0 .. p
        assert bench.prefill_flops(ctx, chunk, Hq, d) == 4 * d * Hq * pairs


def test_algorithmic_bytes_match_the_recorded_profiles():
    """The committed traffic records divide ncu's DRAM bytes by these
    figures: the captured kernel is the one-kernel step (attention and the
    append) for 16-bit caches and the attention alone for E4M3 caches."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert rec, "no traffic records"
    for name, r in rec.items():
        cfg = wl.CONFIGS[name]
        ctx = wl.draw_context_lengths(cfg, torch.Generator().manual_seed(cfg.seed))
        attn, append = bench.algorithmic_bytes(cfg, ctx)
        want = attn + (0 if cfg.is_fp8 else append)
        assert r["algorithmic_bytes_per_launch"] == want, name
        ratio = r["dram_bytes_per_launch"] / want
        assert 1.0 <= ratio < 1.05, (name, ratio)  # each page read once, plus partials


@pytest.mark.parametrize("name", ["llama3_8b_b32_ctx1-4096_bf16", "fp8_8b_b64_ctx8192_e4m3",
                                  "fp8tok_8b_b64_ctx8192_e4m3", "mha_7b_b64_ctx8192_bf16"])
def test_algorithmic_bytes_scale_with_the_cache(name):
    """Doubling every context adds exactly one more copy of the cache bytes
    (K and V of every position, plus per-token scales where kept) and one
    table entry per added page."""
    cfg = wl.CONFIGS[name]
    ctx = wl.draw_context_lengths(cfg, torch.Generator().manual_seed(cfg.seed))
    a1, _ = bench.algorithmic_bytes(cfg, ctx)
    a2, _ = bench.algorithmic_bytes(cfg, 2 * ctx)
    per_pos = cfg.kv_heads * cfg.head_dim * 2 * cfg.cache_elem_bytes
    if cfg.cache == "e4m3tok":
        per_pos += cfg.kv_heads * 8
    added_pages = int(((2 * ctx + 15) // 16).sum() - ((ctx + 15) // 16).sum())
    assert a2 - a1 == int(ctx.sum()) * per_pos + 4 * added_pages
