"""Paged prefill attention on the tensor cores (tcgen05) through the C ABI,
against the oracle's causal multi-query attention (each new row at position
ctx - n + j sees positions 0 .. itself).

"KV Cache & Flash Attention." (kvcache-7e2.pages.dev): the prefill phase
processes the prompt in one parallel pass; continuous-batching section:
chunked prefill reads each sequence's pages through its table."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl
from harness import DeviceRun, logical_kv_fp64, assert_close, seq_kv_fp64

pytestmark = pytest.mark.gpu

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _setup(name, Hq, Hkv, cache, ctx, seed, d=128):
    cfg = wl.small_config(name, len(ctx), Hq, Hkv, d, cache, 1, seed=seed)
    w = wl.generate(cfg, ctx_override=torch.tensor(ctx))
    run = DeviceRun(w)
    run.append()  # every position of every sequence is now in the cache
    return cfg, w, run


def _prefill(run, cfg, chunks, out_dtype="f32", seed=0, max_q_len=None):
    g = torch.Generator().manual_seed(300 + seed)
    total = int(sum(chunks))
    d = cfg.head_dim
    q = torch.randn(total, cfg.q_heads, d, generator=g).to(cfg.qdt)
    starts = torch.tensor([0] + list(np.cumsum(chunks)), dtype=torch.int32)
    out = torch.full((total, cfg.q_heads, d), float("nan"), dtype=_DT[out_dtype], device="cuda")
    pkv.pkv_paged_prefill_attention(run.desc, q.cuda(), run.k_cache, run.v_cache, run.tables,
                                    run.ctx, starts.cuda(),
                                    max(chunks) if max_q_len is None else max_q_len,
                                    cfg.softmax_scale, out)
    torch.cuda.synchronize()
    return q, starts, out


def _expected(w, cfg, q, starts, chunks, pairs=None):
    """Oracle rows for (sequence, query head) pairs (all when None)."""
    ref = {}
    grp = cfg.group
    for b, n in enumerate(chunks):
        if n == 0:
            continue
        for hq in range(cfg.q_heads):
            if pairs is not None and (b, hq) not in pairs:
                continue
            K, V = logical_kv_fp64(w, b, hq // grp)
            qq = q[int(starts[b]):int(starts[b]) + n, hq].double().numpy()
            ref[(b, hq)] = oracle.multi_query_decode(qq, K, V, cfg.softmax_scale)
    return ref


@pytest.mark.parametrize("case", [
    # name, Hq, Hkv, cache, ctx, chunk rows, out dtype, head dim
    ("g4_bf16", 8, 2, "bf16", [1, 17, 300, 700, 129], [1, 17, 130, 256, 128], "f32", 128),
    ("g1_f16", 4, 4, "f16", [40, 513, 260], [40, 200, 3], "f32", 128),
    ("g8_bf16_out16", 16, 2, "bf16", [1000, 64], [300, 64], "bf16", 128),
    ("g2_f16_out16", 4, 2, "f16", [2050, 16], [129, 5], "f16", 128),
    ("g4_f16_d64", 4, 1, "f16", [256, 700, 33], [256, 300, 20], "f32", 64),
    ("g2_bf16_d64_out16", 8, 4, "bf16", [1, 1500], [1, 390], "bf16", 64),
])
def test_prefill_matches_the_oracle(case):
    name, Hq, Hkv, cache, ctx, chunks, out_dtype, d = case
    cfg, w, run = _setup(name, Hq, Hkv, cache, ctx, 61, d)
    q, starts, out = _prefill(run, cfg, chunks, out_dtype)
    assert run.err_code() == 0
    ref = _expected(w, cfg, q, starts, chunks)
    got = out.double().cpu().numpy()
    for (b, hq), r in ref.items():
        s0 = int(starts[b])
        assert_close(got[s0:s0 + chunks[b], hq], r, cfg, out_dtype, f"{name} b{b} h{hq}")


def test_prefill_long_chunk_sampled_and_deterministic():
    """A 1024-row chunk over a 4096-token context (8 row tiles, 32 token
    blocks for the last tile): sampled heads against the oracle, and a second
    run bit for bit equal to the first."""
    cfg, w, run = _setup("long", 8, 2, "bf16", [4096, 1500], 62)
    chunks = [1024, 700]
    q, starts, out = _prefill(run, cfg, chunks, "f32", seed=1)
    _, _, out2 = _prefill(run, cfg, chunks, "f32", seed=1)
    assert run.err_code() == 0
    assert torch.equal(out, out2)
    pairs = {(0, 0), (0, 5), (1, 3)}
    ref = _expected(w, cfg, q, starts, chunks, pairs)
    got = out.double().cpu().numpy()
    for (b, hq), r in ref.items():
        s0 = int(starts[b])
        assert_close(got[s0:s0 + chunks[b], hq], r, cfg, "f32", f"long b{b} h{hq}")


def test_prefill_one_row_equals_decode():
    """A chunk of one row per sequence is the decode step's attention row."""
    cfg, w, run = _setup("one", 8, 2, "bf16", [1, 33, 900], 63)
    dec = run.decode("f32")
    starts = torch.arange(4, dtype=torch.int32)
    out = torch.empty(3, 8, 128, dtype=torch.float32, device="cuda")
    pkv.pkv_paged_prefill_attention(run.desc, run.q, run.k_cache, run.v_cache, run.tables,
                                    run.ctx, starts.cuda(), 1, cfg.softmax_scale, out)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    assert (out - dec).abs().max().item() < 1e-3


def test_prefill_bad_rows_are_reported_not_computed():
    cfg, w, run = _setup("bad", 8, 2, "bf16", [20, 50], 64)
    # sequence 0 claims 30 rows but holds only 20 positions
    q = torch.zeros(40, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.full((40, 8, 128), 7.0, dtype=torch.float32, device="cuda")
    starts = torch.tensor([0, 30, 40], dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_attention(run.desc, q, run.k_cache, run.v_cache, run.tables,
                                    run.ctx, starts, 30, cfg.softmax_scale, out)
    torch.cuda.synchronize()
    assert run.err_code() == pkv.PKV_ERR_BOUNDS
    assert torch.all(out[:30] == 7.0)          # sequence 0 untouched
    assert torch.all(torch.isfinite(out[30:]))  # sequence 1 computed


def test_prefill_unsupported_shapes():
    cfg = wl.small_config("fp8", 2, 8, 2, 128, "e4m3", 1, seed=65)
    w = wl.generate(cfg, ctx_override=torch.tensor([10, 20]))
    run = DeviceRun(w)
    q = torch.zeros(4, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(4, 8, 128, dtype=torch.float32, device="cuda")
    starts = torch.tensor([0, 2, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.pkv_paged_prefill_attention(run.desc, q, run.k_cache, run.v_cache, run.tables,
                                        run.ctx, starts, 2, cfg.softmax_scale, out)


def test_prefill_full_size_whole():
    """The benchmarked prefill (8 sequences x 8192 tokens, each one's last 2048
    positions the chunk) in the launch the bench times: every output row of
    every head against the oracle's chunk attention (fp64, each row over
    exactly the positions it sees)."""
    cfg = wl.CONFIGS["llama3_8b_b8_ctx8192_bf16"]
    w = wl.generate(cfg, device="cuda")
    run = DeviceRun(w)
    run.append()
    chunk = 2048
    q, starts, out = _prefill(run, cfg, [chunk] * cfg.batch, "bf16", seed=5)
    assert run.err_code() == 0
    got = out.double().cpu().numpy()
    qd = q.double().numpy()
    for b in range(cfg.batch):
        K, V = seq_kv_fp64(w, b)
        r0 = int(starts[b])
        for hq in range(cfg.q_heads):
            h = hq // cfg.group
            ref = oracle.chunk_attention(qd[r0:r0 + chunk, hq], K[:, h], V[:, h],
                                         cfg.softmax_scale)
            assert_close(got[r0:r0 + chunk, hq], ref, cfg, "bf16", f"b{b} h{hq}")


def test_prefill_empty_chunks_skip_their_sequences():
    """Sequences with no new rows in the batch take no work and write nothing;
    the others match the oracle."""
    cfg, w, run = _setup("empty", 8, 2, "bf16", [100, 300, 50, 700], 66)
    chunks = [0, 130, 0, 5]
    q, starts, out = _prefill(run, cfg, chunks, "f32", seed=2)
    assert run.err_code() == 0
    ref = _expected(w, cfg, q, starts, chunks)
    got = out.double().cpu().numpy()
    assert set(b for b, _ in ref) == {1, 3}
    for (b, hq), r in ref.items():
        s0 = int(starts[b])
        assert_close(got[s0:s0 + chunks[b], hq], r, cfg, "f32", f"empty b{b} h{hq}")


@pytest.mark.parametrize("bad", [-1, "pool"])
def test_prefill_bad_table_entry_is_reported_not_read(bad):
    """A table entry outside the pool in a page the chunk sees: the error word
    says so, the copy reads the fill value instead, outputs stay finite."""
    cfg, w, run = _setup("badtab", 8, 2, "bf16", [300, 600], 67)
    tables = run.tables.clone()
    tables[1, 5] = -1 if bad == -1 else w.num_blocks  # page 5 of sequence 1 (positions 80..95)
    chunks = [20, 200]
    g = torch.Generator().manual_seed(303)
    q = torch.randn(sum(chunks), cfg.q_heads, cfg.head_dim, generator=g).to(cfg.qdt).cuda()
    starts = torch.tensor([0, 20, 220], dtype=torch.int32, device="cuda")
    out = torch.full((220, cfg.q_heads, cfg.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    pkv.pkv_paged_prefill_attention(run.desc, q, run.k_cache, run.v_cache, tables, run.ctx,
                                    starts, 200, cfg.softmax_scale, out)
    torch.cuda.synchronize()
    assert run.err_code() == pkv.PKV_ERR_BOUNDS
    assert torch.all(torch.isfinite(out))
    # sequence 0 does not touch the bad entry: its rows still match the oracle
    ref = _expected(w, cfg, q.cpu(), starts.cpu(), [20, 0])
    got = out.double().cpu().numpy()
    for (b, hq), r in ref.items():
        assert_close(got[0:20, hq], r, cfg, "f32", f"badtab h{hq}")
