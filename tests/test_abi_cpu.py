"""C-ABI library checks that need no GPU: it builds for sm_103a, loads,
exports every symbol include/pkv.h declares, and its host-only helpers and
argument validation behave (no compute calls)."""
import ctypes
import json
import os
import re
import subprocess

import pytest

import paged_kv_cache_250_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text))
    return names


def test_library_builds_and_exports_every_declared_symbol():
    lib = pkv.load_library()
    declared = _declared_symbols()
    assert declared, "no declarations found"
    assert declared == set(pkv.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name
    # nothing else is exported with the pkv_ prefix
    with open(pkv.library_path(), "rb"):
        pass


def test_struct_layout_matches_header(tmp_path):
    # compile a tiny C program against include/pkv.h and compare every field
    # offset and the size with the ctypes mirror
    fields = [f[0] for f in pkv.CacheDesc._fields_]
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "pkv.h"\nint main(void){\n'
                   + "".join(f'printf("%zu\\n", offsetof(pkv_cache_desc, {f}));\n' for f in fields)
                   + 'printf("%zu\\n", sizeof(pkv_cache_desc)); return 0; }\n')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [getattr(pkv.CacheDesc, f).offset for f in fields] + [ctypes.sizeof(pkv.CacheDesc)]
    assert got == want


def test_host_helpers():
    with open(os.path.join(ROOT, "tests", "golden", "kv_cache_sizes.json")) as f:
        g = json.load(f)
    for c in g["bytes_per_token"]:
        assert pkv.pkv_kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"],
                                          c["elem_bytes"]) == c["bytes"]
    assert pkv.pkv_version() >= 100
    assert "WORKSPACE" in pkv.pkv_status_string(pkv.PKV_ERR_WORKSPACE)
    assert pkv.pkv_status_string(99) == "unknown pkv_status"


def test_argument_errors_return_before_any_launch():
    lib = pkv.load_library()
    good = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_BF16)
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    # null cache pointer
    st = lib.pkv_kv_append(ctypes.byref(good), None, fake, fake, fake, fake, 1, pkv.PKV_BF16, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # kv dtype must equal a 16-bit cache's dtype
    st = lib.pkv_kv_append(ctypes.byref(good), fake, fake, fake, fake, fake, 1, pkv.PKV_F16, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # wrong struct size
    bad = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_BF16)
    bad.struct_size = 8
    st = lib.pkv_kv_append(ctypes.byref(bad), fake, fake, fake, fake, fake, 1, pkv.PKV_BF16, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # block copy: negative count, missing pointers; an empty copy is a no-op
    assert lib.pkv_copy_blocks(ctypes.byref(good), fake, fake, fake, fake, -1, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(ctypes.byref(good), fake, None, fake, fake, 4, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(ctypes.byref(good), fake, fake, fake, fake, 0, None) == pkv.PKV_OK
    # unsupported page size / head dim / group; fp8 without scales
    for desc in (pkv.make_desc(64, 32, 2, 8, 128, pkv.PKV_BF16),
                 pkv.make_desc(64, 16, 2, 8, 80, pkv.PKV_BF16),
                 pkv.make_desc(64, 16, 1, 16, 128, pkv.PKV_BF16),
                 pkv.make_desc(64, 16, 2, 8, 64, pkv.PKV_FP8_E4M3)):
        st = lib.pkv_kv_append(ctypes.byref(desc), fake, fake, fake, fake, fake, 1,
                               pkv.PKV_BF16, None)
        assert st == pkv.PKV_ERR_UNSUPPORTED
    nos = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_FP8_E4M3)
    st = lib.pkv_kv_append(ctypes.byref(nos), fake, fake, fake, fake, fake, 1, pkv.PKV_BF16, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # zero tokens / zero batch are no-ops
    assert lib.pkv_kv_append(ctypes.byref(good), None, None, None, None, None, 0,
                             pkv.PKV_BF16, None) == pkv.PKV_OK
    assert lib.pkv_paged_decode_attention(ctypes.byref(good), None, None, None, None, None,
                                          0, 4, 0, 1.0, None, pkv.PKV_BF16, pkv.PKV_BF16,
                                          None, 0, None) == pkv.PKV_OK
    # decode: missing pointers, bad dtypes, NaN scale
    st = lib.pkv_paged_decode_attention(ctypes.byref(good), fake, fake, fake, fake, None, 2, 4, 0,
                                        1.0, fake, pkv.PKV_BF16, pkv.PKV_BF16, fake, 1 << 20, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    st = lib.pkv_paged_decode_attention(ctypes.byref(good), fake, fake, fake, fake, fake, 2, 4, 0,
                                        1.0, fake, pkv.PKV_F32, pkv.PKV_BF16, fake, 1 << 20, None)
    assert st == pkv.PKV_ERR_UNSUPPORTED
    st = lib.pkv_paged_decode_attention(ctypes.byref(good), fake, fake, fake, fake, fake, 2, 4, 0,
                                        float("nan"), fake, pkv.PKV_BF16, pkv.PKV_BF16, fake,
                                        1 << 20, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # a batch whose per-sequence arrays do not fit the largest shared-memory plan
    st = lib.pkv_paged_decode_attention(ctypes.byref(good), fake, fake, fake, fake, fake, 7000, 4,
                                        0, 1.0, fake, pkv.PKV_BF16, pkv.PKV_BF16, fake, 1 << 30,
                                        None)
    assert st == pkv.PKV_ERR_UNSUPPORTED


def test_argument_errors_of_the_later_entry_points():
    """Window, multi-query, one-kernel step, prefill and the per-token FP8
    descriptor: argument errors found on the host, before any CUDA call."""
    lib = pkv.load_library()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    good = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_BF16)
    D = ctypes.byref(good)
    # sliding window: negative window or sinks, q_len 0
    for q_len, window, sinks in ((1, -1, 0), (1, 8, -2), (0, 8, 0)):
        st = lib.pkv_paged_decode_attention_window(D, fake, fake, fake, fake, fake, 2, q_len,
                                                   window, sinks, 4, 0, 1.0, fake, pkv.PKV_BF16,
                                                   pkv.PKV_F32, fake, 1 << 20, None)
        assert st == pkv.PKV_ERR_INVALID_ARG
    # multi-query: q_len 0; more query tokens than the 8 built (at any group)
    st = lib.pkv_paged_decode_attention_multi(D, fake, fake, fake, fake, fake, 2, 0, 4, 0, 1.0,
                                              fake, pkv.PKV_BF16, pkv.PKV_F32, fake, 1 << 20, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    st = lib.pkv_paged_decode_attention_multi(D, fake, fake, fake, fake, fake, 2, 9, 4, 0, 1.0,
                                              fake, pkv.PKV_BF16, pkv.PKV_F32, fake, 1 << 20, None)
    assert st == pkv.PKV_ERR_UNSUPPORTED
    st = lib.pkv_paged_decode_attention_window(D, fake, fake, fake, fake, fake, 2, 9, 100, 4, 4,
                                               0, 1.0, fake, pkv.PKV_BF16, pkv.PKV_F32, fake,
                                               1 << 20, None)
    assert st == pkv.PKV_ERR_UNSUPPORTED
    # the multi-query workspace size refuses q_len outside 1 .. 8
    assert lib.pkv_decode_workspace_bytes_multi(D, 2, 0, 4, 0) == 0
    assert lib.pkv_decode_workspace_bytes_multi(D, 2, 9, 4, 0) == 0
    # one-kernel step: a null q; an empty batch is a no-op
    st = lib.pkv_decode_step_fused(D, None, fake, fake, fake, fake, pkv.PKV_BF16, fake, fake, 2,
                                   4, 0, 1.0, fake, pkv.PKV_BF16, pkv.PKV_F32, fake, 1 << 20, 0,
                                   None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_fused(D, None, None, None, None, None, pkv.PKV_BF16, None, None,
                                     0, 4, 0, 1.0, None, pkv.PKV_BF16, pkv.PKV_F32, None, 0, 0,
                                     None) == pkv.PKV_OK
    # prefill: FP8 caches and head_dims other than 64 and 128 are not built; q
    # must match the cache;
    # negative sizes; empty calls are no-ops
    fp8 = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_FP8_E4M3)
    fp8.k_scale = fp8.v_scale = 0x1000
    d80 = pkv.make_desc(64, 16, 2, 8, 80, pkv.PKV_BF16)

    def prefill(desc, q_dtype=pkv.PKV_BF16, batch=2, total=8, maxq=4):
        return lib.pkv_paged_prefill_attention(ctypes.byref(desc), fake, fake, fake, fake, fake,
                                               fake, batch, total, maxq, 4, 1.0, fake, q_dtype,
                                               pkv.PKV_F32, None)
    assert prefill(fp8) == pkv.PKV_ERR_UNSUPPORTED
    assert prefill(d80) == pkv.PKV_ERR_UNSUPPORTED
    assert prefill(good, q_dtype=pkv.PKV_F16) == pkv.PKV_ERR_INVALID_ARG
    assert prefill(good, total=-1) == pkv.PKV_ERR_INVALID_ARG
    assert prefill(good, batch=0) == pkv.PKV_OK
    assert prefill(good, maxq=0) == pkv.PKV_OK
    # per-token FP8: the scale pool must be 128-byte aligned; v_scale is unused
    tok = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_FP8_E4M3_TOKEN)
    tok.k_scale = 0x1040  # 64-byte aligned only
    st = lib.pkv_kv_append(ctypes.byref(tok), fake, fake, fake, fake, fake, 1, pkv.PKV_BF16, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    tok.k_scale = 0x1080
    assert lib.pkv_kv_append(ctypes.byref(tok), None, None, None, None, None, 0, pkv.PKV_BF16,
                             None) == pkv.PKV_OK
    tok64 = pkv.make_desc(64, 16, 2, 8, 64, pkv.PKV_FP8_E4M3_TOKEN)
    tok64.k_scale = 0x1080
    st = lib.pkv_kv_append(ctypes.byref(tok64), fake, fake, fake, fake, fake, 1, pkv.PKV_BF16,
                           None)
    assert st == pkv.PKV_ERR_UNSUPPORTED


def test_prefill_argument_errors():
    """The prefill's host checks, each before any CUDA call: the scale must be
    positive (the kernel takes row maxima of the raw scores), the output a
    16- or 32-bit float, the pointers present and aligned, the table width
    positive."""
    lib = pkv.load_library()
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)  # not 16-byte aligned
    good = pkv.make_desc(64, 16, 2, 8, 128, pkv.PKV_BF16)

    def call(q=fake, q_start=fake, scale=1.0, out_dtype=pkv.PKV_F32, mbs=4, out=fake):
        return lib.pkv_paged_prefill_attention(ctypes.byref(good), q, fake, fake, fake, fake,
                                               q_start, 2, 8, 4, mbs, scale, out, pkv.PKV_BF16,
                                               out_dtype, None)
    for scale in (0.0, -0.5, float("nan")):
        assert call(scale=scale) == pkv.PKV_ERR_INVALID_ARG
    assert call(out_dtype=pkv.PKV_FP8_E4M3) == pkv.PKV_ERR_UNSUPPORTED
    assert call(q=odd) == pkv.PKV_ERR_INVALID_ARG
    assert call(out=odd) == pkv.PKV_ERR_INVALID_ARG
    assert call(q_start=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(mbs=0) == pkv.PKV_ERR_INVALID_ARG
