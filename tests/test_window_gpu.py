"""Sliding-window decode with attention sinks through the C ABI against the
oracle's window_decode.

[AP] "Sparse attention: stop looking at everything": a token sees only the
previous w tokens plus a few global tokens at the start of the text; [KVFA]
eviction paragraph: the window drops the oldest tokens, attention sinks keep
the first few."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl
from harness import (DeviceRun, assert_close, assert_same_rounding, logical_kv_fp64,
                     oracle_multi_seq, seq_kv_fp64)

PAGE = wl.PAGE


def _q(cfg, q_len, seed):
    g = torch.Generator().manual_seed(200 + seed)
    return torch.randn(cfg.batch, q_len, cfg.q_heads, cfg.head_dim, generator=g).to(cfg.qdt)


def _window_call(run, cfg, q, window, sinks, tables=None):
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    n = pkv.pkv_decode_workspace_bytes_multi(run.desc, cfg.batch, q.shape[1],
                                             run.w.max_blocks_per_seq)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_decode_attention_window(run.desc, q.cuda(), run.k_cache, run.v_cache,
                                          run.tables if tables is None else tables, run.ctx,
                                          window, sinks, cfg.softmax_scale, out, ws)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    return out


def _oracle(w, cfg, q, window, sinks):
    q_len = q.shape[1]
    ref = np.zeros(tuple(q.shape), dtype=np.float64)
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            K, V = logical_kv_fp64(w, b, h)
            n = K.shape[0]
            if n == 0:
                continue
            first = max(0, q_len - n)  # tokens at negative positions see nothing
            for hh in range(cfg.group):
                hq = h * cfg.group + hh
                qq = q[b, first:, hq].double().numpy()
                ref[b, first:, hq] = oracle.window_decode(qq, K, V, cfg.softmax_scale,
                                                          window, sinks)
    return ref


def _setup(name, B, Hq, Hkv, d, cache, ctx, seed):
    cfg = wl.small_config(name, B, Hq, Hkv, d, cache, 1, seed=seed)
    w = wl.generate(cfg, ctx_override=torch.tensor(ctx))
    run = DeviceRun(w)
    run.append()
    return cfg, w, run


@pytest.mark.gpu
@pytest.mark.parametrize("case", [
    # name, batch, Hq, Hkv, d, cache, q_len, window, sinks
    ("g4_q1_w100_s4", 6, 32, 8, 128, "bf16", 1, 100, 4),     # single query, window + sinks
    ("g4_q1_w16_s0", 5, 8, 2, 128, "bf16", 1, 16, 0),       # page-sized window, no sinks
    ("g1_q1_w7_s20", 5, 4, 4, 128, "bf16", 1, 7, 20),       # sinks across a page boundary
    ("g2_q3_w50_s3", 5, 8, 4, 128, "bf16", 3, 50, 3),       # causal new tokens + window
    ("g4_q2_w33_s16", 5, 8, 2, 128, "bf16", 2, 33, 16),     # 8 columns: barrier-tree flush
    ("g1_q8_w9_s1", 4, 2, 2, 128, "bf16", 8, 9, 1),         # window shorter than a page
    ("g2_q2_w256_s16_e4m3", 5, 8, 4, 128, "e4m3", 2, 256, 16),
    ("g4_q1_w40_s2_f16_d64", 5, 8, 2, 64, "f16", 1, 40, 2),
    ("g1_q4_w1_s0", 4, 4, 4, 128, "bf16", 4, 1, 0),         # each token sees itself only
    # more than 8 (query token, head) columns per KV head
    ("g4_q4_w9_s1", 6, 8, 2, 128, "bf16", 4, 9, 1),         # window shorter than a page
    ("g4_q5_w100_s4", 6, 8, 2, 128, "bf16", 5, 100, 4),     # two slices
    ("g8_q3_w40_s0", 5, 16, 2, 128, "bf16", 3, 40, 0),      # 24 columns
    ("g8_q8_w5_s2", 5, 8, 1, 128, "bf16", 8, 5, 2),         # 64 columns, four slices
    ("g8_q4_w300_s16_e4m3", 5, 16, 2, 128, "e4m3", 4, 300, 16),
    ("g4_q8_w20_s3_f16_d64", 5, 8, 2, 64, "f16", 8, 20, 3),
])
def test_window_matches_the_oracle(case):
    name, B, Hq, Hkv, d, cache, q_len, window, sinks = case
    ctx = [1, 5, 37, 700, 2100, 333][:B]
    cfg, w, run = _setup(name, B, Hq, Hkv, d, cache, ctx, 51)
    q = _q(cfg, q_len, 1)
    got = _window_call(run, cfg, q, window, sinks).cpu().double().numpy()
    assert_close(got, _oracle(w, cfg, q, window, sinks), cfg, "f32", name)


@pytest.mark.gpu
def test_window_skipped_pages_are_never_read():
    """Table entries of pages no token sees may be anything: a -1 there
    would be a bounds error if the kernel looked it up."""
    window, sinks, q_len = 64, 4, 2
    cfg, w, run = _setup("gap", 4, 8, 2, 128, "bf16", [40, 300, 1000, 2049], 52)
    q = _q(cfg, q_len, 2)
    tables = w.block_tables.clone()
    holes = 0
    for b, n in enumerate(w.ctx.tolist()):
        first_window_page = max(0, n - q_len - window + 1) // PAGE
        sink_pages = -(-min(n, sinks) // PAGE)
        for pg in range(sink_pages, first_window_page):
            tables[b, pg] = -1
            holes += 1
    assert holes > 100
    got = _window_call(run, cfg, q, window, sinks, tables.cuda()).cpu().double().numpy()
    assert_close(got, _oracle(w, cfg, q, window, sinks), cfg, "f32", "gap")


@pytest.mark.gpu
@pytest.mark.parametrize("window,sinks", [(0, 7), (5000, 0), (2100, 3)])
def test_window_covering_everything_equals_plain_decode(window, sinks):
    """No window, or one reaching past position 0, masks nothing: the result
    is that of the multi-query call (up to the order of fp32 partial sums)."""
    q_len = 2
    cfg, w, run = _setup("wide", 5, 8, 2, 128, "bf16", [1, 5, 37, 700, 2100], 53)
    q = _q(cfg, q_len, 3)
    got = _window_call(run, cfg, q, window, sinks)
    out = torch.empty_like(got)
    pkv.pkv_paged_decode_attention_multi(run.desc, q.cuda(), run.k_cache, run.v_cache,
                                         run.tables, run.ctx, cfg.softmax_scale, out,
                                         run.workspace)
    torch.cuda.synchronize()
    assert_same_rounding(got, out, "window covering everything vs multi-query")


@pytest.mark.gpu
def test_window_long_contexts_whole():
    """A long-context batch under a 4096-token window, in the launch the
    bench times: every output row against the oracle."""
    window, sinks = 4096, 4
    cfg, w, run = _setup("long", 8, 32, 8, 128, "bf16",
                         [16384, 9000, 4097, 4096, 12345, 70, 8191, 16000], 54)
    q = _q(cfg, 1, 4)
    got = _window_call(run, cfg, q, window, sinks).cpu().double().numpy()
    qd = q.double().numpy()
    for b in range(cfg.batch):
        K, V = seq_kv_fp64(w, b)
        ref = oracle_multi_seq(qd[b], K, V, cfg.softmax_scale, window, sinks)
        assert_close(got[b], ref, cfg, "f32", f"long b{b}")


@pytest.mark.gpu
def test_window_rejects_negative_arguments():
    cfg, w, run = _setup("neg", 2, 8, 2, 128, "bf16", [10, 20], 55)
    q = _q(cfg, 1, 5)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    for window, sinks in [(-1, 0), (8, -1)]:
        with pytest.raises(pkv.PkvError):
            pkv.pkv_paged_decode_attention_window(run.desc, q.cuda(), run.k_cache, run.v_cache,
                                                  run.tables, run.ctx, window, sinks,
                                                  cfg.softmax_scale, out, run.workspace)
