"""The one-kernel decode step (pkv_decode_step_fused): append and attention
in a single launch, against the oracle and, bit for bit, against the
two-kernel step.

[KVFA] KV-cache section: each step appends the new token's K and V, then
attends over all cached tokens; PagedAttention section: position ->
(block, offset)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl
from harness import DeviceRun, assert_close, oracle_all, oracle_rows, oracle_whole

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 15, 16, 17, 31, 33, 250, 600, 1000]


def _bytes(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.uint8)  # NaN-poisoned slots compare as bytes


def _both_ways(w, out_dtype="f32"):
    """Run the one-kernel step and the two-kernel step on separate copies of
    the same inputs; return both outputs and both runs."""
    one, two = DeviceRun(w), DeviceRun(w)
    out1 = one.step_one_kernel(out_dtype)
    out2 = two.step(out_dtype, fused=True)
    torch.cuda.synchronize()
    assert one.err_code() == 0 and two.err_code() == 0
    return out1, out2, one, two


@pytest.mark.parametrize("cache", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_one_kernel_step_16bit(cache, d, g):
    cfg = wl.small_config(f"one_{cache}_{d}_{g}", len(RAGGED), 2 * g, 2, d, cache, 1,
                          seed=61 + g + d)
    w = wl.generate(cfg, ctx_override=torch.tensor(RAGGED))
    out1, out2, one, two = _both_ways(w)
    assert torch.equal(out1, out2)
    assert torch.equal(_bytes(one.k_cache), _bytes(two.k_cache))
    assert torch.equal(_bytes(one.v_cache), _bytes(two.v_cache))
    assert_close(out1.double().cpu().numpy(), oracle_all(w), cfg, "f32", "one-kernel step")


@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("q_dtype", ["bf16", "f16"])
def test_one_kernel_step_fp8(g, q_dtype):
    """E4M3 cache: the staged row and the cache row carry the encoding
    pkv_kv_append writes (divide by the head's scale, RNE, saturate)."""
    cfg = wl.small_config(f"one_fp8_{g}", len(RAGGED), 2 * g, 2, 128, "e4m3", 1,
                          seed=71 + g, q_dtype=q_dtype)
    w = wl.generate(cfg, ctx_override=torch.tensor(RAGGED))
    out1, out2, one, two = _both_ways(w)
    assert torch.equal(out1, out2)
    assert torch.equal(_bytes(one.k_cache), _bytes(two.k_cache))
    assert torch.equal(_bytes(one.v_cache), _bytes(two.v_cache))
    assert_close(out1.double().cpu().numpy(), oracle_all(w), cfg, "f32", "one-kernel fp8")


def test_one_kernel_step_empty_and_single_token_sequences():
    """ctx 0 appends nothing and gives a zero row; ctx 1 attends to the new
    token alone, so the output is its V row exactly."""
    cfg = wl.small_config("one_edge", 4, 8, 2, 128, "bf16", 1, seed=81)
    w = wl.generate(cfg, ctx_override=torch.tensor([0, 1, 17, 0]))
    run = DeviceRun(w)
    before_k, before_v = _bytes(run.k_cache).clone(), _bytes(run.v_cache).clone()
    out = run.step_one_kernel("f32")
    torch.cuda.synchronize()
    assert run.err_code() == 0
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[3]) == 0
    g = cfg.group
    for hq in range(cfg.q_heads):
        assert torch.equal(out[1, hq], run.v_new[1, hq // g].float())
    # exactly the appended rows (sequences 1 and 2, every KV head) changed:
    # they held the pool's NaN poison before
    row = cfg.head_dim * 2
    changed_k = (_bytes(run.k_cache) != before_k).view(-1, row).any(dim=1).sum().item()
    changed_v = (_bytes(run.v_cache) != before_v).view(-1, row).any(dim=1).sum().item()
    assert changed_k == 2 * cfg.kv_heads and changed_v == 2 * cfg.kv_heads
    ref = oracle_all(w)
    assert_close(out.double().cpu().numpy(), ref, cfg, "f32", "edge")


def test_one_kernel_step_many_splits():
    """A long sequence spread over every warp of the grid: the new token's
    page belongs to one warp of one CTA among many."""
    cfg = wl.small_config("one_long", 3, 8, 2, 128, "bf16", 1, seed=82)
    w = wl.generate(cfg, ctx_override=torch.tensor([70000, 3, 4097]))
    out1, out2, one, two = _both_ways(w)
    assert torch.equal(out1, out2)
    assert torch.equal(_bytes(one.k_cache), _bytes(two.k_cache))
    pairs = [(b, hq) for b in range(3) for hq in (0, 5)]
    ref = oracle_rows(w, pairs)
    assert_close(np.stack([out1[b, hq].double().cpu().numpy() for b, hq in pairs]),
                 np.stack([ref[p] for p in pairs]), cfg, "f32", "one_long")


def test_one_kernel_step_full_size_whole():
    """The benchmarked workload in the one-kernel step without overlap, every
    output element against the oracle, bf16 output (the overlapped form is
    checked whole with the other full-size configs)."""
    cfg = wl.CONFIGS["llama3_8b_b32_ctx1-4096_bf16"]
    w = wl.generate(cfg, device="cuda")
    run = DeviceRun(w, hint=4096)
    out = run.step_one_kernel("bf16", overlap=False).double().cpu().numpy()
    torch.cuda.synchronize()
    assert run.err_code() == 0
    assert_close(out, oracle_whole(w), cfg, "bf16", "full size")


@pytest.mark.parametrize("cache", ["bf16", "e4m3"])
def test_overlapped_steps_chain(cache):
    """Two back-to-back steps with PKV_STEP_OVERLAP on one stream: the second
    reads its lengths and tables while the first finishes, and must still see
    the row the first one appended.  The pool starts without each sequence's
    last two tokens; after both steps the caches and the second step's output
    equal those of the same two steps without the flag, and the output
    matches the oracle over all tokens."""
    cfg = wl.small_config(f"chain_{cache}", len(RAGGED), 8, 2, 128, cache, 1, seed=84)
    w = wl.generate(cfg, ctx_override=torch.tensor(RAGGED))
    ctx = w.ctx.to(torch.int64)
    prev = (ctx - 2).clamp(min=0)
    runs = []
    for overlap in (True, False):
        run = DeviceRun(w)
        tab = run.tables.to(torch.int64)
        ar = torch.arange(cfg.batch, device="cuda")
        pos = prev.cuda()
        blk = tab[ar, pos // wl.PAGE]
        has_prev = (ctx >= 2).cuda()
        # poison the second-newest row too: the first step appends it
        poison = run.k_cache[0, 0, 0, 0].clone().fill_(float("nan")) if cache != "e4m3" \
            else torch.tensor(0x7F, dtype=torch.uint8, device="cuda")
        for b in range(cfg.batch):
            if bool(has_prev[b]):
                run.k_cache[blk[b], :, pos[b] % wl.PAGE, :] = poison
                run.v_cache[blk[b], :, pos[b] % wl.PAGE, :] = poison
        ctx1 = (ctx - 1).clamp(min=0).to(torch.int32).cuda()
        k1 = w.K_log[torch.arange(cfg.batch), prev].to("cuda").contiguous()
        v1 = w.V_log[torch.arange(cfg.batch), prev].to("cuda").contiguous()
        out1 = torch.empty(cfg.batch, cfg.q_heads, cfg.head_dim, dtype=torch.float32,
                           device="cuda")
        out2 = torch.empty_like(out1)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            pkv.pkv_decode_step_fused(run.desc, run.q, run.k_cache, run.v_cache, k1, v1,
                                      run.tables, ctx1, cfg.softmax_scale, out1, run.workspace,
                                      stream=s, overlap=overlap)
            pkv.pkv_decode_step_fused(run.desc, run.q, run.k_cache, run.v_cache, run.k_new,
                                      run.v_new, run.tables, run.ctx, cfg.softmax_scale, out2,
                                      run.workspace, stream=s, overlap=overlap)
        s.synchronize()
        assert run.err_code() == 0
        runs.append((run, out2))
    (ra, oa), (rb, ob) = runs
    assert torch.equal(oa, ob)
    assert torch.equal(_bytes(ra.k_cache), _bytes(rb.k_cache))
    assert torch.equal(_bytes(ra.v_cache), _bytes(rb.v_cache))
    assert_close(oa.double().cpu().numpy(), oracle_all(w), cfg, "f32", "chain")


def test_one_kernel_step_argument_errors():
    cfg = wl.small_config("one_args", 2, 8, 2, 128, "bf16", 1, seed=83)
    w = wl.generate(cfg, ctx_override=torch.tensor([5, 9]))
    run = DeviceRun(w)
    out = torch.empty(2, 8, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PkvError):  # 16-bit cache: new rows must match its dtype
        pkv.pkv_decode_step_fused(run.desc, run.q, run.k_cache, run.v_cache,
                                  run.k_new.half(), run.v_new.half(), run.tables, run.ctx,
                                  cfg.softmax_scale, out, run.workspace)
    lib = pkv.load_library()
    import ctypes
    st = lib.pkv_decode_step_fused(  # an unknown flag bit
        ctypes.byref(run.desc), run.q.data_ptr(), run.k_cache.data_ptr(), run.v_cache.data_ptr(),
        run.k_new.data_ptr(), run.v_new.data_ptr(), pkv.PKV_BF16, run.tables.data_ptr(),
        run.ctx.data_ptr(), 2, int(run.tables.shape[1]), 0, cfg.softmax_scale, out.data_ptr(),
        pkv.PKV_BF16, pkv.PKV_F32, run.workspace.data_ptr(), run.workspace.numel(), 2, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
