"""The benchmarked forms of the added operations, at their full sizes and in
the launch configuration the bench times: multi-query decode and the sliding
window with sinks (every output element against the oracle, one sequence at
a time) and whole-block copies (every copied byte compared).

"KV Cache & Flash Attention." (kvcache-7e2.pages.dev): speculative-decoding
section (several new tokens scored at once), eviction paragraph (a window of
recent positions plus the first ones), PagedAttention section (blocks shared
and copied on write).  "Paged attention: stop reserving empty tables" and
"Sparse attention: stop looking at everything" for the same two ideas."""
import numpy as np
import pytest
import torch

import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl
from harness import DeviceRun, assert_close, oracle_multi_seq, seq_kv_fp64

pytestmark = pytest.mark.gpu

BENCH_HINT = {"llama3_8b_b32_ctx1-4096_bf16": 4096}


def _launch(name, q_len, window=None, sinks=0, seed=0):
    """One multi-query (window None) or windowed call on a full-size workload
    with the bench's bf16 output, after the append of the newest token."""
    cfg = wl.CONFIGS[name]
    w = wl.generate(cfg, device="cuda")
    run = DeviceRun(w, hint=BENCH_HINT.get(name, 0))
    run.append()
    # the bench's workspace: partials of group x q_len columns
    n = pkv.pkv_decode_workspace_bytes_multi(run.desc, cfg.batch, q_len, w.max_blocks_per_seq,
                                             run.hint)
    run.workspace = torch.zeros(n, dtype=torch.uint8, device="cuda")
    g = torch.Generator().manual_seed(400 + seed)
    q = torch.randn(cfg.batch, q_len, cfg.q_heads, cfg.head_dim, generator=g).to(cfg.qdt)
    out = torch.empty(cfg.batch, q_len, cfg.q_heads, cfg.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    if window is None:
        pkv.pkv_paged_decode_attention_multi(run.desc, q.cuda(), run.k_cache, run.v_cache,
                                             run.tables, run.ctx, cfg.softmax_scale, out,
                                             run.workspace, run.hint)
    else:
        pkv.pkv_paged_decode_attention_window(run.desc, q.cuda(), run.k_cache, run.v_cache,
                                              run.tables, run.ctx, window, sinks,
                                              cfg.softmax_scale, out, run.workspace, run.hint)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    return cfg, w, q, out.double().cpu().numpy()


def _check_whole(cfg, w, q, got, name, window=0, sinks=0):
    """Every (sequence, query token, head) row against the oracle; query
    tokens before position 0 (a context shorter than q_len) get zero rows."""
    q_len = q.shape[1]
    qd = q.double().numpy()
    for b in range(cfg.batch):
        n = int(w.ctx[b])
        first = max(0, q_len - n)
        assert not got[b, :first].any(), f"{name} b{b}: rows before position 0"
        if first == q_len:
            continue
        K, V = seq_kv_fp64(w, b)
        ref = oracle_multi_seq(qd[b, first:], K, V, cfg.softmax_scale, window, sinks)
        assert_close(got[b, first:], ref, cfg, "bf16", f"{name} b{b}")


@pytest.mark.parametrize("name,q_len", [
    ("mha_7b_b64_ctx8192_bf16", 8),        # g 1: eight tokens fill the MMA's columns
    ("llama3_8b_b32_ctx1-4096_bf16", 2),   # g 4 x 2 tokens, ragged lengths, length hint
    ("llama3_70b_b8_ctx32768_bf16", 1),    # g 8, one token: the multi-query call's QC 1 form
    ("llama3_70b_b8_ctx32768_bf16", 4),    # g 8 x 4 tokens: 32 columns over two slices
    ("llama3_8b_b32_ctx1-4096_bf16", 5),   # g 4 x 5 tokens (capacity 8): 32 columns
])
def test_multi_query_full_size_whole(name, q_len):
    cfg, w, q, got = _launch(name, q_len, seed=1)
    assert np.all(np.isfinite(got))
    _check_whole(cfg, w, q, got, name)


@pytest.mark.parametrize("name,q_len,window,sinks", [
    ("mha_7b_b64_ctx8192_bf16", 2, 4096, 4),      # the windowed bench line
    ("llama3_8b_b32_ctx1-4096_bf16", 1, 1000, 16),  # windows shorter than many contexts
    ("llama3_70b_b8_ctx32768_bf16", 4, 4096, 4),    # 32 columns under a window
])
def test_window_full_size_whole(name, q_len, window, sinks):
    cfg, w, q, got = _launch(name, q_len, window, sinks, seed=2)
    assert np.all(np.isfinite(got))
    _check_whole(cfg, w, q, got, name, window, sinks)


def test_copy_blocks_full_size_bit_exact():
    """The benchmarked copy: 8192 of 16384 bf16 blocks (8 KV heads x 16 x 128,
    K and V) onto the other 8192; every destination block equals its source
    bit for bit, every other block keeps its bits."""
    NB, Hkv, d, n = 16384, 8, 128, 8192
    g = torch.Generator().manual_seed(7)
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    src, dst = perm[:n].cuda(), perm[n:2 * n].cuda()
    kc = torch.randn(NB, Hkv, wl.PAGE, d, device="cuda").to(torch.bfloat16)
    vc = torch.randn(NB, Hkv, wl.PAGE, d, device="cuda").to(torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = pkv.make_desc(NB, wl.PAGE, Hkv, Hkv, d, pkv.PKV_BF16, None, None, err)
    pkv.pkv_copy_blocks(desc, kc, vc, src, dst)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    keep = torch.ones(NB, dtype=torch.bool, device="cuda")
    keep[dst.long()] = False
    for got, before in ((kc, k0), (vc, v0)):
        gb, bb = got.view(torch.int16), before.view(torch.int16)
        assert torch.equal(gb[dst.long()], bb[src.long()])
        assert torch.equal(gb[keep], bb[keep])
