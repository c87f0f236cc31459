"""CPU oracle for paged single-token decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``paged_kv_cache_250_gb300``) never imports, links or calls it, and the two
share no code: the oracle is plain C in fp64 (``pkv_oracle.c``), the thin
numpy marshalling below, and a few numpy reference functions (library matrix
products and table lookups in fp64) that restate definitions the C code also
gives row by row.

What it computes, and where each definition comes from, is stated beside each
function in ``pkv_oracle.c``.  Every function here is pinned by the
``-m "not gpu"`` tests (``tests/test_oracle_pins.py`` and the ``*_oracle.py``
files beside it) against values the pages print, closed forms, special cases
and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the compiler offers it)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        D, I32, I64, U64 = (ctypes.c_double, ctypes.c_int32, ctypes.c_int64,
                            ctypes.c_uint64)
        P = ctypes.c_void_p
        lib.pkvo_kv_bytes_per_token.restype = U64
        lib.pkvo_kv_bytes_per_token.argtypes = [I32, I32, I32, I32]
        lib.pkvo_kv_bytes.restype = U64
        lib.pkvo_kv_bytes.argtypes = [I64, I32, I32, I32, I32, I32]
        lib.pkvo_rows_recomputed.restype = I64
        lib.pkvo_rows_recomputed.argtypes = [I64, I64]
        lib.pkvo_rows_cached.restype = I64
        lib.pkvo_rows_cached.argtypes = [I64, I64]
        lib.pkvo_e4m3_decode.restype = D
        lib.pkvo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.pkvo_e4m3_encode.restype = ctypes.c_uint8
        lib.pkvo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.pkvo_e4m3_quantize_array.restype = None
        lib.pkvo_e4m3_quantize_array.argtypes = [P, I64, ctypes.c_float, P]
        lib.pkvo_e4m3_dequantize_array.restype = None
        lib.pkvo_e4m3_dequantize_array.argtypes = [P, I64, D, P]
        lib.pkvo_attend_row.restype = None
        lib.pkvo_attend_row.argtypes = [P, P, P, I64, I64, I32, D, P]
        lib.pkvo_decode_attention.restype = None
        lib.pkvo_decode_attention.argtypes = [P, P, P, P, I32, I32, I32, I32,
                                              I64, D, P, I32]
        lib.pkvo_max_threads.restype = I32
        lib.pkvo_max_threads.argtypes = []
        lib.pkvo_online_softmax_stats.restype = None
        lib.pkvo_online_softmax_stats.argtypes = [P, I64, I64, P, P, P, P]
        lib.pkvo_online_attend_row.restype = None
        lib.pkvo_online_attend_row.argtypes = [P, P, P, I64, I64, I32, D, I64,
                                               P, P, P, P]
        lib.pkvo_merge_partials.restype = None
        lib.pkvo_merge_partials.argtypes = [P, P, P, I32, I32, P]
        lib.pkvo_append_bytes.restype = None
        lib.pkvo_append_bytes.argtypes = [P, P, P, I32, I32, I32, I32, I32, I32]
        lib.pkvo_append_e4m3.restype = None
        lib.pkvo_append_e4m3.argtypes = [P, P, P, P, I32, I32, I32, I32, I32]
        lib.pkvo_e4m3_token_scale.restype = ctypes.c_float
        lib.pkvo_e4m3_token_scale.argtypes = [P, I32]
        lib.pkvo_append_e4m3_token.restype = None
        lib.pkvo_append_e4m3_token.argtypes = [P, P, P, P, I32, I32, I32, I32, I32]
        lib.pkvo_e4m3_dequantize_rows.restype = None
        lib.pkvo_e4m3_dequantize_rows.argtypes = [P, P, I64, I32, P]
        lib.pkvo_copy_blocks.restype = None
        lib.pkvo_copy_blocks.argtypes = [P, P, P, I32, I32, I64]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# ----------------------------------------------------------------- sizes
def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                       elem_bytes: int) -> int:
    return int(_load().pkvo_kv_bytes_per_token(layers, kv_heads, head_dim,
                                               elem_bytes))


def kv_bytes(tokens: int, layers: int, kv_heads: int, head_dim: int,
             elem_bytes: int = 2, batch: int = 1) -> int:
    return int(_load().pkvo_kv_bytes(tokens, layers, kv_heads, head_dim,
                                     elem_bytes, batch))


def rows_recomputed(prompt: int, n_new: int) -> int:
    return int(_load().pkvo_rows_recomputed(prompt, n_new))


def rows_cached(prompt: int, n_new: int) -> int:
    return int(_load().pkvo_rows_cached(prompt, n_new))


# ----------------------------------------------------------------- fp8
def e4m3_decode(code: int) -> float:
    return float(_load().pkvo_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(_load().pkvo_e4m3_encode(float(x)))


def e4m3_quantize(x, scale: float) -> np.ndarray:
    """Stored E4M3 bytes for fp32 values ``x`` under one fp32 scale."""
    xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(xf.shape, dtype=np.uint8)
    _load().pkvo_e4m3_quantize_array(_ptr(xf), xf.size, float(np.float32(scale)),
                                     _ptr(out))
    return out


def e4m3_dequantize(codes, scale: float) -> np.ndarray:
    """fp64 values of stored E4M3 bytes times the (fp32) scale."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().pkvo_e4m3_dequantize_array(_ptr(c), c.size,
                                       float(np.float32(scale)), _ptr(out))
    return out


def e4m3_token_scale(row) -> float:
    """Per-token FP8 scale of one (token, KV head) row: its largest magnitude
    over 448 in IEEE fp32 (1 for an all-zero row)."""
    r = np.ascontiguousarray(np.asarray(row, dtype=np.float32).reshape(-1))
    return float(_load().pkvo_e4m3_token_scale(_ptr(r), r.size))


def e4m3_dequantize_rows(codes, row_scale) -> np.ndarray:
    """fp64 rows [n][d] of E4M3 codes, each times its own fp32 scale."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    n, d = c.shape
    rs = np.ascontiguousarray(np.asarray(row_scale, dtype=np.float32).reshape(n))
    out = np.empty((n, d), dtype=np.float64)
    _load().pkvo_e4m3_dequantize_rows(_ptr(c), _ptr(rs), n, d, _ptr(out))
    return out


# ----------------------------------------------------------------- attention
def attend_row(q, K, V, scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for one query row; K, V are [ctx][d]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    d = q.shape[-1]
    ctx = K.shape[0]
    out = np.empty(d, dtype=np.float64)
    _load().pkvo_attend_row(_ptr(q), _ptr(K), _ptr(V), ctx, d, d, float(scale),
                            _ptr(out))
    return out


def decode_attention(q, K, V, ctx, scale: float, nthreads: int = 0) -> np.ndarray:
    """Decode attention over the logical cache.

    q [B][Hq][d]; K, V [B][T][Hkv][d]; ctx [B] -> out [B][Hq][d] (fp64).
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    ctx = np.ascontiguousarray(np.asarray(ctx, dtype=np.int32))
    B, Hq, d = q.shape
    _, T, Hkv, _ = K.shape
    assert K.shape == V.shape == (B, T, Hkv, d) and Hq % Hkv == 0
    assert ctx.shape == (B,) and int(ctx.max(initial=0)) <= T
    out = np.empty((B, Hq, d), dtype=np.float64)
    _load().pkvo_decode_attention(_ptr(q), _ptr(K), _ptr(V), _ptr(ctx), B, Hq,
                                  Hkv, d, T, float(scale), _ptr(out),
                                  int(nthreads))
    return out


def max_threads() -> int:
    return int(_load().pkvo_max_threads())


def online_softmax_stats(x, tile: int):
    """Streaming (m, l) over ``x`` in tiles; returns (m, l, m_trace, l_trace)."""
    x = _f64(x)
    n = x.size
    k = -(-n // tile)
    m, l = ctypes.c_double(), ctypes.c_double()
    mt = np.empty(k, dtype=np.float64)
    lt = np.empty(k, dtype=np.float64)
    _load().pkvo_online_softmax_stats(_ptr(x), n, tile, ctypes.byref(m),
                                      ctypes.byref(l), _ptr(mt), _ptr(lt))
    return m.value, l.value, mt, lt


def online_attend_row(q, K, V, scale: float, tile: int):
    """Tile-streamed attention row; returns (out, m, l, o_unnormalised)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    d = q.shape[-1]
    out = np.empty(d, dtype=np.float64)
    o = np.empty(d, dtype=np.float64)
    m, l = ctypes.c_double(), ctypes.c_double()
    _load().pkvo_online_attend_row(_ptr(q), _ptr(K), _ptr(V), K.shape[0], d, d,
                                   float(scale), int(tile), _ptr(out),
                                   ctypes.byref(m), ctypes.byref(l), _ptr(o))
    return out, m.value, l.value, o


def merge_partials(m, l, o) -> np.ndarray:
    """Combine partial (m, l, unnormalised o) states; o is [n][d]."""
    m, l, o = _f64(m), _f64(l), _f64(o)
    n, d = o.shape
    out = np.empty(d, dtype=np.float64)
    _load().pkvo_merge_partials(_ptr(m), _ptr(l), _ptr(o), n, d, _ptr(out))
    return out


# ----------------------------------------------------------------- append
def append_bytes(cache: np.ndarray, src: np.ndarray, slot) -> np.ndarray:
    """Expected 16-bit cache after an append; returns a new array.

    cache: [NB][Hkv][P][d] of a 2-byte dtype, src: [T][Hkv][d] same dtype.
    """
    out = np.ascontiguousarray(cache).copy()
    src = np.ascontiguousarray(src)
    assert out.dtype.itemsize == src.dtype.itemsize
    NB, Hkv, P, d = out.shape
    slot = np.ascontiguousarray(np.asarray(slot, dtype=np.int64))
    _load().pkvo_append_bytes(_ptr(out), _ptr(src), _ptr(slot), slot.size, NB,
                              P, Hkv, d, out.dtype.itemsize)
    return out


def append_e4m3(cache: np.ndarray, src, slot, head_scale) -> np.ndarray:
    """Expected E4M3 cache after an append of fp32-valued rows ``src``."""
    out = np.ascontiguousarray(cache, dtype=np.uint8).copy()
    srcf = np.ascontiguousarray(np.asarray(src, dtype=np.float32))
    hs = np.ascontiguousarray(np.asarray(head_scale, dtype=np.float32))
    NB, Hkv, P, d = out.shape
    slot = np.ascontiguousarray(np.asarray(slot, dtype=np.int64))
    _load().pkvo_append_e4m3(_ptr(out), _ptr(srcf), _ptr(slot), _ptr(hs),
                             slot.size, NB, P, Hkv, d)
    return out


def append_e4m3_token(cache: np.ndarray, scales: np.ndarray, src, slot):
    """Expected per-token E4M3 cache [NB][Hkv][P][d] and scale pool
    [NB][Hkv][P] after an append of fp32-valued rows ``src`` [T][Hkv][d]."""
    out = np.ascontiguousarray(cache, dtype=np.uint8).copy()
    sc = np.ascontiguousarray(scales, dtype=np.float32).copy()
    srcf = np.ascontiguousarray(np.asarray(src, dtype=np.float32))
    NB, Hkv, P, d = out.shape
    slot = np.ascontiguousarray(np.asarray(slot, dtype=np.int64))
    _load().pkvo_append_e4m3_token(_ptr(out), _ptr(sc), _ptr(srcf), _ptr(slot), slot.size,
                                   NB, P, Hkv, d)
    return out, sc


def copy_blocks(cache: np.ndarray, src, dst) -> np.ndarray:
    """Expected cache after copying block src[i] to block dst[i] (all heads,
    in order); ids outside the pool are skipped.  Returns a new array.

    cache: [NB][Hkv][P][d] of any element type.
    """
    out = np.ascontiguousarray(cache).copy()
    src = np.ascontiguousarray(np.asarray(src, dtype=np.int32))
    dst = np.ascontiguousarray(np.asarray(dst, dtype=np.int32))
    assert src.shape == dst.shape
    NB = out.shape[0]
    block_bytes = out[0].nbytes if NB > 0 else 0
    _load().pkvo_copy_blocks(_ptr(out), _ptr(src), _ptr(dst), src.size, NB, block_bytes)
    return out


# ----------------------------------------------------------------- decode loop
def multi_query_decode(q, K, V, scale: float) -> np.ndarray:
    """Several new tokens of one sequence at once (verifying drafted tokens,
    [KVFA] speculative-decoding section): q is [QL][d] for the last QL
    positions of a sequence whose cached rows K, V are [n][d] (n >= QL, the
    new tokens' rows included); query i sits at position n - QL + i and
    attends to rows 0 .. n - QL + i, causal among the new tokens.  Each row
    is the plain definition (attend_row)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, QL = K.shape[0], q.shape[0]
    assert n >= QL
    return np.stack([attend_row(q[i], K[:n - QL + i + 1], V[:n - QL + i + 1], scale)
                     for i in range(QL)])


def chunk_attention(q, K, V, scale: float) -> np.ndarray:
    """A chunk of QL new tokens of one sequence at once, for one query head
    ([KVFA] opening section: the prefill processes the prompt in one parallel
    pass; continuous-batching section: chunked prefill): q is [QL][d] for the
    last QL positions of a sequence whose cached rows K, V are [n][d]
    (n >= QL); row i sits at position n - QL + i and attends to rows
    0 .. n - QL + i.  The rows of multi_query_decode, for the whole chunk
    with library matrix products in fp64: scores S = scale q K^T, the
    positions past each row's own masked out, then the two-pass softmax (row
    maximum, exponentials, row sum) and the weighted sum of the V rows."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, QL = K.shape[0], q.shape[0]
    assert n >= QL
    S = scale * (q @ K.T)                                   # [QL][n]
    last = n - QL + np.arange(QL)[:, None]                  # each row's position
    S = np.where(np.arange(n)[None, :] <= last, S, -np.inf)
    E = np.exp(S - S.max(axis=1, keepdims=True))
    return (E @ V) / E.sum(axis=1, keepdims=True)


def window_decode(q, K, V, scale: float, window: int, sinks: int) -> np.ndarray:
    """Multi-query decode under a sliding window with attention sinks ([AP]
    "Sparse attention: stop looking at everything": each token sees only the
    previous w tokens, and a few global tokens at the start of the text are
    seen by everything; [KVFA] eviction paragraph: a sliding window drops the
    oldest tokens, attention sinks always keep the first few).  Reading:
    query j at position p = n - QL + j sees rows t <= p with t >= p - window + 1
    (itself included) or t < sinks; window 0 means no window.  Each row is
    attend_row over exactly those rows, in order."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, QL = K.shape[0], q.shape[0]
    assert n >= QL and window >= 0 and sinks >= 0
    out = []
    for j in range(QL):
        p = n - QL + j
        rows = [t for t in range(p + 1) if window == 0 or t >= p - window + 1 or t < sinks]
        out.append(attend_row(q[j], K[rows], V[rows], scale))
    return np.stack(out)


def causal_attention_last_row(X, Wq, Wk, Wv, scale: float) -> np.ndarray:
    """Recompute-everything step ([KVFA] opening section; [AP] "Arjun's first
    attempt"): project every token so far, form the full causal score matrix,
    softmax each row, multiply by V, and keep only the last row.  Plain fp64
    numpy; the matrix products are library steps, the softmax is written out.
    """
    X = _f64(X)
    Q, K, V = X @ _f64(Wq), X @ _f64(Wk), X @ _f64(Wv)
    n = X.shape[0]
    S = (Q @ K.T) * scale
    S = np.where(np.tril(np.ones((n, n), dtype=bool)), S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    A = E / E.sum(axis=1, keepdims=True)
    return (A @ V)[-1]


def cached_decode(X, Wq, Wk, Wv, scale: float):
    """Cached decode ([AP] "Following one new token through the cache"):
    each step projects only the newest token, appends its K and V rows to the
    logical cache, then attends its query over all rows so far.  Returns the
    per-step outputs and the number of K/V rows computed."""
    X = _f64(X)
    d = Wk.shape[1]
    Kc, Vc, outs = [], [], []
    for t in range(X.shape[0]):
        x = X[t]
        Kc.append(x @ _f64(Wk))
        Vc.append(x @ _f64(Wv))
        outs.append(attend_row(x @ _f64(Wq), np.stack(Kc), np.stack(Vc), scale))
    return np.stack(outs), len(Kc)
