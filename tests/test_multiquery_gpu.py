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
from harness import DeviceRun, logical_kv_fp64, assert_close, assert_same_rounding

_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def multi_workspace(run, cfg, q_len):
    """A zeroed workspace sized for q_len query tokens per sequence."""
    n = pkv.pkv_decode_workspace_bytes_multi(run.desc, cfg.batch, q_len,
                                             run.w.max_blocks_per_seq)
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _run(cfg, ctx, q_len, out_dtype="f32", seed=0):
    w = wl.generate(cfg, ctx_override=torch.tensor(ctx))
    run = DeviceRun(w)
    run.append()  # the newest token; the other new tokens are already cached
    run.workspace = multi_workspace(run, cfg, q_len)
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
    # more than 8 (query token, head) columns: two column groups per warp
    # (16), or the columns split over 2 or 4 warps per page (32, 64)
    ("g4_q3_bf16", 5, 8, 2, 128, "bf16", 3),    # 12 of 16 columns
    ("g4_q4_bf16", 5, 16, 4, 128, "bf16", 4),   # 16
    ("g4_q5_bf16", 5, 8, 2, 128, "bf16", 5),    # 20 of 32: two slices
    ("g4_q8_bf16", 5, 8, 2, 128, "bf16", 8),    # 32
    ("g8_q2_bf16", 5, 16, 2, 128, "bf16", 2),   # 16
    ("g8_q3_bf16", 4, 8, 1, 128, "bf16", 3),    # 24 of 32
    ("g8_q4_bf16", 5, 16, 2, 128, "bf16", 4),   # 32
    ("g8_q5_bf16", 4, 8, 1, 128, "bf16", 5),    # 40 of 64: four slices
    ("g8_q8_bf16", 5, 16, 2, 128, "bf16", 8),   # 64
    ("g8_q4_e4m3", 5, 16, 2, 128, "e4m3", 4),
    ("g4_q8_e4m3tok", 5, 8, 2, 128, "e4m3tok", 8),
    ("g8_q8_f16_d64", 4, 16, 2, 64, "f16", 8),
    ("g2_q8_f16_d64", 4, 8, 4, 64, "f16", 8),
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
    run = DeviceRun(w)
    run.append()
    single = run.decode("f32")
    out = torch.empty(cfg.batch, 1, cfg.q_heads, cfg.head_dim, dtype=torch.float32, device="cuda")
    pkv.pkv_paged_decode_attention_multi(run.desc, run.q.view(cfg.batch, 1, cfg.q_heads,
                                                              cfg.head_dim),
                                         run.k_cache, run.v_cache, run.tables, run.ctx,
                                         cfg.softmax_scale, out, run.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], single)  # q_len 1 is the single-token kernel


@pytest.mark.gpu
def test_multi_query_rejects_too_many_tokens():
    cfg = wl.small_config("big_q", 2, 8, 2, 128, "bf16", 64, seed=43)
    w = wl.generate(cfg)
    run = DeviceRun(w)
    q = torch.zeros(2, 9, 8, 128, dtype=torch.bfloat16, device="cuda")  # 9 query tokens
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_decode_attention_multi(run.desc, q, run.k_cache, run.v_cache, run.tables,
                                             run.ctx, cfg.softmax_scale, out, run.workspace)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    # 3 query tokens at group 4 are 12 columns: the single-token workspace is
    # too small for their partials, the multi-query size is not
    q3 = torch.zeros(2, 3, 8, 128, dtype=torch.bfloat16, device="cuda")
    small = pkv.pkv_decode_workspace_bytes(run.desc, 2, w.max_blocks_per_seq)
    big = pkv.pkv_decode_workspace_bytes_multi(run.desc, 2, 3, w.max_blocks_per_seq)
    assert big > small > 0
