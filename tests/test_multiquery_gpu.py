"""Multi-query decode (q_len new tokens per sequence, causal among
themselves) through the C ABI against the oracle's multi_query_decode.

[KVFA] speculative-decoding section: the target model scores the prefix and
the drafted tokens in one forward pass."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl
from harness import GpuRun, logical_kv_fp64, assert_close

_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _run(cfg, ctx, q_len, out_dtype="f32", seed=0):
    w = wl.generate(cfg, ctx_override=torch.tensor(ctx))
    run = GpuRun(w)
    run.append()  # the newest token; the other new tokens are already cached
    qdt = cfg.qdt
    g = torch.Generator().manual_seed(100 + seed)
    q = torch.randn(cfg.batch, q_len, cfg.q_heads, cfg.head_dim, generator=g).to(qdt)
    out = torch.empty(cfg.batch, q_len, cfg.q_heads, cfg.head_dim,
                      dtype=torch.float32 if out_dtype == "f32" else _DT[out_dtype], device="cuda")
    pkv.pkv_paged_decode_attention_multi(run.desc, q.cuda(), run.k_cache, run.v_cache, run.tables,
                                         run.ctx, cfg.softmax_scale, out, run.workspace)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    got = out.cpu().double().numpy()
    ref = np.zeros_like(got)
    grp = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            K, V = logical_kv_fp64(w, b, h)
            n = K.shape[0]
            for hh in range(grp):
                hq = h * grp + hh
                qq = q[b, :, hq].double().numpy()
                if n == 0:
                    continue  # zero rows
                # tokens j with position n - q_len + j < 0 see nothing: zero row
                first = max(0, q_len - n)
                if first < q_len:
                    ref[b, first:, hq] = oracle.multi_query_decode(qq[first:], K, V,
                                                                   cfg.softmax_scale)
    return got, ref


@pytest.mark.gpu
@pytest.mark.parametrize("case", [
    # name, batch, Hq, Hkv, d, cache, q_len
    ("g4_q2_bf16", 5, 8, 2, 128, "bf16", 2),    # 8 MMA columns: barrier-tree flush
    ("g2_q3_bf16", 4, 8, 4, 128, "bf16", 3),    # capacity 4, one padding token
    ("g1_q4_bf16", 3, 4, 4, 128, "bf16", 4),    # 4 columns: asynchronous hand-off
    ("g1_q8_bf16", 3, 2, 2, 128, "bf16", 8),
    ("g2_q2_e4m3", 4, 8, 4, 128, "e4m3", 2),
    ("g4_q2_f16_d64", 3, 8, 2, 64, "f16", 2),
])
def test_multi_query_matches_the_oracle(case):
    name, B, Hq, Hkv, d, cache, q_len = case
    cfg = wl.small_config(name, B, Hq, Hkv, d, cache, 1, seed=41)
    ctx = [1, q_len - 1 if q_len > 1 else 2, 37, 700, 2100][:B] + [17] * max(0, B - 5)
    got, ref = _run(cfg, ctx, q_len)
    assert_close(got, ref, cfg, "f32", name)


@pytest.mark.gpu
def test_multi_query_one_token_equals_single_decode():
    cfg = wl.small_config("q1", 4, 8, 2, 128, "bf16", (1, 900), seed=42)
    w = wl.generate(cfg)
    run = GpuRun(w)
    run.append()
    single = run.decode("f32")
    out = torch.empty(cfg.batch, 1, cfg.q_heads, cfg.head_dim, dtype=torch.float32, device="cuda")
    pkv.pkv_paged_decode_attention_multi(run.desc, run.q.view(cfg.batch, 1, cfg.q_heads,
                                                              cfg.head_dim),
                                         run.k_cache, run.v_cache, run.tables, run.ctx,
                                         cfg.softmax_scale, out, run.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], single)


@pytest.mark.gpu
def test_multi_query_rejects_too_many_tokens():
    cfg = wl.small_config("big_q", 2, 8, 2, 128, "bf16", 64, seed=43)
    w = wl.generate(cfg)
    run = GpuRun(w)
    q = torch.zeros(2, 3, 8, 128, dtype=torch.bfloat16, device="cuda")  # 4 heads x 3 > 8
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_paged_decode_attention_multi(run.desc, q, run.k_cache, run.v_cache, run.tables,
                                             run.ctx, cfg.softmax_scale, out, run.workspace)
