"""The no-allocation decode entry point, checked against the regular one.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate device
memory when they attend (no allocator handle inside a custom-op hook, an
engine that owns all device memory, a path that must not risk the device
synchronisation cudaMalloc can cause).  It runs the same kernel on a fixed
scratch array inside the library.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl

from harness import DeviceRun, assert_close, oracle_all

pytestmark = pytest.mark.gpu


def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    cfg = wl.small_config("noalloc", 6, 16, 4, 128, "bf16", 1, seed=21)
    w = wl.generate(cfg, ctx_override=torch.tensor([1, 17, 300, 64, 1000, 33]))
    run = DeviceRun(w)
    run.append()
    ref = run.decode("f32")  # regular entry point with a caller workspace
    outs = []
    for _ in range(2):  # the scratch keeps the last call's contents
        out = torch.full_like(ref, float("nan"))
        pkv.pkv_paged_decode_attention_noalloc(run.desc, run.q, run.k_cache, run.v_cache,
                                               run.tables, run.ctx, cfg.softmax_scale, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert run.err_code() == 0
    r = ref.double().cpu().numpy()
    for out in outs:
        o = out.double().cpu().numpy()
        assert np.all(np.isfinite(o))
        assert np.abs(o - r).max() <= 2e-3
    # and both agree with the oracle
    assert_close(outs[1].double().cpu().numpy(), oracle_all(w), cfg, "f32", "noalloc")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 1200 sequences x 8 KV heads x group 8: the split partials alone exceed
    # the fixed scratch, so the call must refuse before launching anything
    B, Hkv, Hq, d = 1200, 8, 64, 128
    dev = "cuda"
    desc = pkv.make_desc(1, 16, Hkv, Hq, d, pkv.PKV_BF16)
    need = pkv.pkv_decode_workspace_bytes(desc, B, 1, 0)
    assert need > pkv.PKV_NOALLOC_SCRATCH_BYTES
    kc = torch.zeros(1, Hkv, 16, d, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device=dev)
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    tables = torch.zeros(B, 1, dtype=torch.int32, device=dev)
    ctx = torch.zeros(B, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_decode_attention_noalloc(desc, q, kc, vc, tables, ctx, 0.1, out)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE


def test_noalloc_on_a_side_stream_and_argument_errors_first():
    # Each call clears its arrival counters on the stream it is given: two
    # calls in a row on a non-default stream must match the regular entry
    # point.  An invalid argument is refused before anything is queued.
    cfg = wl.small_config("noalloc_stream", 5, 8, 2, 128, "bf16", 1, seed=22)
    w = wl.generate(cfg, ctx_override=torch.tensor([3, 700, 40, 1, 2048]))
    run = DeviceRun(w)
    run.append()
    ref = run.decode("f32")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    with torch.cuda.stream(side):
        for out in outs:
            pkv.pkv_paged_decode_attention_noalloc(run.desc, run.q, run.k_cache, run.v_cache,
                                                   run.tables, run.ctx, cfg.softmax_scale, out,
                                                   stream=side)
    side.synchronize()
    assert run.err_code() == 0
    for out in outs:
        assert np.abs(out.double().cpu().numpy() - ref.double().cpu().numpy()).max() <= 2e-3
    bad = torch.empty_like(ref)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_decode_attention_noalloc(run.desc, run.q, run.k_cache, run.v_cache,
                                               run.tables, run.ctx, float("nan"), bad)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
