"""E4M3 caches with one fp32 scale per (token, KV head) row, through the C
ABI: the append against the oracle's per-token codec (bytes and scales bit
for bit), attention against the oracle on the dequantised cache, the
one-kernel step and block copies.

"KV Cache & Flash Attention." (kvcache-7e2.pages.dev), memory-cost section
(the cache is quantized to fp8) and Flash Attention section (FP8 with
finer-grained scales)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl
from harness import DeviceRun, assert_close, oracle_all, oracle_rows, oracle_whole

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 15, 16, 17, 31, 33, 250, 600, 1000]


def _bytes(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.uint8)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float16])
def test_append_matches_the_oracle_bit_for_bit(in_dtype):
    NB, Hkv, d, T = 9, 4, 128, 7
    g = torch.Generator().manual_seed(91)
    k = torch.randn(T, Hkv, d, generator=g) * torch.exp(torch.randn(T, Hkv, 1, generator=g) * 3)
    v = torch.randn(T, Hkv, d, generator=g) * torch.exp(torch.randn(T, Hkv, 1, generator=g) * 3)
    k[2, 1] = 0.0                      # an all-zero row: scale 1, codes 0
    k[4, 3, 17] = 3.0e4 if in_dtype == torch.float16 else 1.0e6  # an outlier inside a row
    k, v = k.to(in_dtype), v.to(in_dtype)
    slot = torch.tensor([5, 16 * 3 + 15, -1, 16 * 8, 33, 16 * 6 + 1, 140], dtype=torch.int64)
    kc = torch.full((NB, Hkv, 16, d), 0x7F, dtype=torch.uint8)
    vc = kc.clone()
    pool = torch.full((NB, Hkv, 2, 16), float("nan"), dtype=torch.float32)  # K, then V scales
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kcd, vcd, pd = kc.cuda(), vc.cuda(), pool.cuda()
    desc = pkv.make_desc(NB, 16, Hkv, Hkv, d, pkv.PKV_FP8_E4M3_TOKEN, pd, None, err)
    pkv.pkv_kv_append(desc, kcd, vcd, slot.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_kc, want_ks = oracle.append_e4m3_token(kc.numpy(), pool[:, :, 0].numpy(),
                                                k.float().numpy(), slot.numpy())
    want_vc, want_vs = oracle.append_e4m3_token(vc.numpy(), pool[:, :, 1].numpy(),
                                                v.float().numpy(), slot.numpy())
    assert np.array_equal(kcd.cpu().numpy(), want_kc)
    assert np.array_equal(vcd.cpu().numpy(), want_vc)
    # scales compared as bits (NaN-poisoned slots too)
    got = pd.cpu().numpy()
    assert np.array_equal(got[:, :, 0].view(np.uint32), want_ks.view(np.uint32))
    assert np.array_equal(got[:, :, 1].view(np.uint32), want_vs.view(np.uint32))


@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("q_dtype", ["bf16", "f16"])
def test_decode_matches_the_oracle(g, q_dtype):
    cfg = wl.small_config(f"tok_{g}", len(RAGGED), 2 * g, 2, 128, "e4m3tok", 1, seed=92 + g,
                          q_dtype=q_dtype)
    w = wl.generate(cfg, ctx_override=torch.tensor(RAGGED))
    run = DeviceRun(w)
    out = run.step("f32").double().cpu().numpy()
    out_bf = run.decode("bf16").double().cpu().numpy()
    torch.cuda.synchronize()
    assert run.err_code() == 0
    ref = oracle_all(w)
    err = assert_close(out, ref, cfg, "f32", "per-token fp32 out")
    assert err < 2e-3  # the expected error is far inside the 3e-2 gate
    assert_close(out_bf, ref, cfg, "bf16", "per-token bf16 out")


@pytest.mark.parametrize("B", [104, 105, 300])
def test_both_ring_depths_match_the_oracle(B):
    """Batches on both sides of the size where the per-token kernel's deeper
    ring (four page slots per warp, barrier-tree segment ends) stops fitting
    two CTAs per SM and the three-slot form with the asynchronous hand-off
    runs instead: every output row against the oracle, with many short
    sequences (so many segment ends) and some long ones (split segments)."""
    gen = torch.Generator().manual_seed(B)
    ctx = torch.randint(0, 48, (B,), generator=gen, dtype=torch.int32)
    ctx[::37] = 700
    cfg = wl.small_config(f"tok_depth_{B}", B, 32, 8, 128, "e4m3tok", 1, seed=93)
    w = wl.generate(cfg, ctx_override=ctx)
    run = DeviceRun(w)
    out = run.step("f32").double().cpu().numpy()
    torch.cuda.synchronize()
    assert run.err_code() == 0
    assert_close(out, oracle_whole(w), cfg, "f32", f"per-token B {B}")


def test_one_kernel_step_equals_two_kernel_step():
    cfg = wl.small_config("tok_step", len(RAGGED), 8, 2, 128, "e4m3tok", 1, seed=97)
    w = wl.generate(cfg, ctx_override=torch.tensor(RAGGED))
    one, two = DeviceRun(w), DeviceRun(w)
    o1 = one.step_one_kernel("f32")
    o2 = two.step("f32", fused=True)
    torch.cuda.synchronize()
    assert one.err_code() == 0 and two.err_code() == 0
    assert torch.equal(o1, o2)
    for a, b in ((one.k_cache, two.k_cache), (one.v_cache, two.v_cache),
                 (one.k_scale, two.k_scale)):
        assert torch.equal(_bytes(a), _bytes(b))


def test_long_sequence_and_window():
    """A long split sequence, and a sliding window (one query token) over a
    per-token cache, against the oracle."""
    cfg = wl.small_config("tok_long", 3, 8, 2, 128, "e4m3tok", 1, seed=98)
    w = wl.generate(cfg, ctx_override=torch.tensor([20000, 5, 3000]))
    run = DeviceRun(w)
    out = run.step("f32").double().cpu().numpy()
    torch.cuda.synchronize()
    assert run.err_code() == 0
    pairs = [(b, hq) for b in range(3) for hq in (0, 7)]
    ref = oracle_rows(w, pairs)
    assert_close(np.stack([out[b, hq] for b, hq in pairs]), np.stack([ref[p] for p in pairs]),
                 cfg, "f32", "tok_long")
    q = run.q.view(3, 1, 8, 128)
    got = torch.empty(3, 1, 8, 128, dtype=torch.float32, device="cuda")
    pkv.pkv_paged_decode_attention_window(run.desc, q, run.k_cache, run.v_cache, run.tables,
                                          run.ctx, 700, 4, cfg.softmax_scale, got, run.workspace)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    from harness import logical_kv_fp64
    for b in range(3):
        K, V = logical_kv_fp64(w, b, 0)
        for hq in range(4):
            ref = oracle.window_decode(w.q[b, hq].double().numpy()[None], K, V,
                                       cfg.softmax_scale, 700, 4)[0]
            assert_close(got[b, 0, hq].double().cpu().numpy(), ref, cfg, "f32", "tok window")


def test_copy_blocks_moves_the_scales():
    cfg = wl.small_config("tok_cow", 2, 8, 2, 128, "e4m3tok", 1, seed=99)
    w = wl.generate(cfg, ctx_override=torch.tensor([40, 20]))
    run = DeviceRun(w)
    tab = w.block_tables
    src = torch.tensor([int(tab[0, 0]), int(tab[0, 2])], dtype=torch.int32)
    dst = torch.tensor([int(tab[1, 0]), w.num_blocks - 1], dtype=torch.int32)
    pkv.pkv_copy_blocks(run.desc, run.k_cache, run.v_cache, src.cuda(), dst.cuda())
    torch.cuda.synchronize()
    assert run.err_code() == 0
    for s_, d_ in zip(src.tolist(), dst.tolist()):
        for a in (run.k_cache, run.v_cache, run.k_scale):
            assert torch.equal(_bytes(a[d_]), _bytes(a[s_]))


@pytest.mark.parametrize("g,q_len", [(4, 2), (1, 8), (2, 3)])
def test_multi_query_matches_the_oracle(g, q_len):
    """q_len new tokens per sequence, causal among themselves, over a
    per-token cache."""
    cfg = wl.small_config(f"tok_mq_{g}", 4, 2 * g, 2, 128, "e4m3tok", 1, seed=100 + g)
    w = wl.generate(cfg, ctx_override=torch.tensor([1, 9, 300, 1200]))
    run = DeviceRun(w)
    run.append()
    gq = torch.Generator().manual_seed(7 + g)
    q = torch.randn(4, q_len, cfg.q_heads, 128, generator=gq).to(cfg.qdt)
    out = torch.empty(4, q_len, cfg.q_heads, 128, dtype=torch.float32, device="cuda")
    pkv.pkv_paged_decode_attention_multi(run.desc, q.cuda(), run.k_cache, run.v_cache, run.tables,
                                         run.ctx, cfg.softmax_scale, out, run.workspace)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    from harness import logical_kv_fp64
    got = out.double().cpu().numpy()
    for b in range(4):
        for h in range(cfg.kv_heads):
            K, V = logical_kv_fp64(w, b, h)
            n = K.shape[0]
            first = max(0, q_len - n)
            for hh in range(cfg.group):
                hq = h * cfg.group + hh
                ref = oracle.multi_query_decode(q[b, first:, hq].double().numpy(), K, V,
                                                cfg.softmax_scale)
                assert_close(got[b, first:, hq], ref, cfg, "f32", f"tok mq b{b} h{hq}")
