"""Test harness: run a workload through the CUDA path and through the oracle.

The oracle side sees only the logical (unpaged) drawn values and decodes FP8
bytes with its own codec; the CUDA side sees only the paged pool, the block
tables and the slot mapping.  Nothing the CUDA path writes is ever fed to the
oracle.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np
import torch

import oracle
import paged_kv_cache_250_gb300 as pkv
from paged_kv_cache_250_gb300 import workloads as wl

TOL_16BIT = 2e-3   # max abs error vs the oracle, bf16/fp16 cache, fp32 accumulation
TOL_FP8 = 3e-2     # max abs error vs the oracle on the dequantised cache

_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
_CODE = {"f16": pkv.PKV_F16, "bf16": pkv.PKV_BF16, "e4m3": pkv.PKV_FP8_E4M3,
         "e4m3tok": pkv.PKV_FP8_E4M3_TOKEN}


def tolerance(cfg) -> float:
    return TOL_FP8 if cfg.is_fp8 else TOL_16BIT


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half a unit in the last place of `dtype` at |x| (the output rounding)."""
    mant = {torch.float16: 10, torch.bfloat16: 7, torch.float32: 23}[dtype]
    emin = {torch.float16: -14, torch.bfloat16: -126, torch.float32: -126}[dtype]
    ax = np.maximum(np.abs(x), 1e-300)
    e = np.maximum(np.floor(np.log2(ax)), emin)
    return 0.5 * np.exp2(e - mant)


# ------------------------------------------------------------------ oracle side
def logical_kv_fp64(w: wl.DecodeWorkload, b: int, h: int) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 K, V rows [ctx][d] of sequence b, KV head h, as the cache holds them
    after the append: drawn values for 16-bit caches; for E4M3 the stored
    codes (prefix) or the oracle's own encoding of the new token, decoded and
    scaled by the oracle's codec."""
    n = int(w.ctx[b])
    if not w.cfg.is_fp8:
        K = w.K_log[b, :n, h].double().cpu().numpy()
        V = w.V_log[b, :n, h].double().cpu().numpy()
        return K, V
    if w.cfg.cache == "e4m3tok":  # one scale per row; the new row's by the oracle
        Kc = w.K_stored[b, :n, h].cpu().numpy().copy()
        Vc = w.V_stored[b, :n, h].cpu().numpy().copy()
        ks = w.extra["k_tok_scale"][b, :n, h].float().cpu().numpy().copy()
        vs = w.extra["v_tok_scale"][b, :n, h].float().cpu().numpy().copy()
        if n > 0:
            kn = w.k_new[b, h].float().cpu().numpy()
            vn = w.v_new[b, h].float().cpu().numpy()
            ks[n - 1] = oracle.e4m3_token_scale(kn)
            vs[n - 1] = oracle.e4m3_token_scale(vn)
            Kc[n - 1] = oracle.e4m3_quantize(kn, ks[n - 1])
            Vc[n - 1] = oracle.e4m3_quantize(vn, vs[n - 1])
        return oracle.e4m3_dequantize_rows(Kc, ks), oracle.e4m3_dequantize_rows(Vc, vs)
    ks = float(w.k_scale[h])
    vs = float(w.v_scale[h])
    Kc = w.K_stored[b, :n, h].cpu().numpy().copy()
    Vc = w.V_stored[b, :n, h].cpu().numpy().copy()
    if n > 0:
        Kc[n - 1] = oracle.e4m3_quantize(w.k_new[b, h].float().cpu().numpy(), ks)
        Vc[n - 1] = oracle.e4m3_quantize(w.v_new[b, h].float().cpu().numpy(), vs)
    return oracle.e4m3_dequantize(Kc, ks), oracle.e4m3_dequantize(Vc, vs)


def oracle_rows(w: wl.DecodeWorkload, pairs: Iterable[Tuple[int, int]]) -> dict:
    """Expected output rows for the given (b, hq) pairs."""
    g = w.cfg.group
    res = {}
    cache = {}
    for b, hq in pairs:
        h = hq // g
        if (b, h) not in cache:
            cache[(b, h)] = logical_kv_fp64(w, b, h)
        K, V = cache[(b, h)]
        q = w.q[b, hq].double().cpu().numpy()
        res[(b, hq)] = oracle.attend_row(q, K, V, w.cfg.softmax_scale)
    return res


def seq_kv_fp64(w: wl.DecodeWorkload, b: int) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 K, V [ctx][Hkv][d] of sequence b (logical_kv_fp64 for every KV
    head).  16-bit caches widen on the device and copy once."""
    n = int(w.ctx[b])
    if not w.cfg.is_fp8:
        return (w.K_log[b, :n].double().cpu().numpy(), w.V_log[b, :n].double().cpu().numpy())
    kv = [logical_kv_fp64(w, b, h) for h in range(w.cfg.kv_heads)]
    return np.stack([k for k, _ in kv], axis=1), np.stack([v for _, v in kv], axis=1)


def oracle_whole(w: wl.DecodeWorkload) -> np.ndarray:
    """Every output row [B][Hq][d]: the oracle's decode_attention (fp64,
    all host cores) one sequence at a time, so host memory holds one
    sequence's fp64 cache at most."""
    cfg = w.cfg
    q = w.q.double().cpu().numpy()
    out = np.zeros((cfg.batch, cfg.q_heads, cfg.head_dim))
    for b in range(cfg.batch):
        n = int(w.ctx[b])
        if n == 0:
            continue  # no rows: the zero output row
        K, V = seq_kv_fp64(w, b)
        out[b] = oracle.decode_attention(q[b:b + 1], K[None], V[None], [n],
                                         cfg.softmax_scale)[0]
    return out


def oracle_multi_seq(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                     window: int = 0, sinks: int = 0) -> np.ndarray:
    """oracle.multi_query_decode (window 0) or oracle.window_decode for every
    head of one sequence at once: q [QL][Hq][d], K, V [n][Hkv][d] (n >= QL)
    -> [QL][Hq][d].  Query j sits at position p = n - QL + j and sees the rows
    t <= p with t > p - window or t < sinks (all t <= p when window is 0);
    those rows, gathered in order, go through decode_attention."""
    QL = q.shape[0]
    n = K.shape[0]
    assert n >= QL
    out = np.empty(q.shape)
    for j in range(QL):
        p = n - QL + j
        if window > 0:
            lo = max(0, p - window + 1)
            rows = np.concatenate([np.arange(min(sinks, lo)), np.arange(lo, p + 1)])
            Kj, Vj = K[rows], V[rows]
        else:
            Kj, Vj = K[:p + 1], V[:p + 1]
        out[j] = oracle.decode_attention(q[j][None], Kj[None], Vj[None], [Kj.shape[0]],
                                         scale)[0]
    return out


def oracle_all(w: wl.DecodeWorkload) -> np.ndarray:
    B, Hq, d = w.cfg.batch, w.cfg.q_heads, w.cfg.head_dim
    out = np.zeros((B, Hq, d))
    rows = oracle_rows(w, [(b, hq) for b in range(B) for hq in range(Hq)])
    for (b, hq), r in rows.items():
        out[b, hq] = r
    return out


# ------------------------------------------------------------------ CUDA side
class DeviceRun:
    """Device copies of a workload and one append + decode through the C ABI."""

    def __init__(self, w: wl.DecodeWorkload, device="cuda", hint: int = 0,
                 with_err_word: bool = True):
        self.w = w
        cfg = w.cfg
        self.dev = torch.device(device)
        self.k_cache = w.k_cache.to(self.dev).contiguous()
        self.v_cache = w.v_cache.to(self.dev).contiguous()
        self.q = w.q.to(self.dev).contiguous()
        self.k_new = w.k_new.to(self.dev).contiguous()
        self.v_new = w.v_new.to(self.dev).contiguous()
        self.slot = w.slot_mapping.to(self.dev).contiguous()
        self.tables = w.block_tables.to(self.dev).contiguous()
        self.ctx = w.ctx.to(self.dev).contiguous()
        self.k_scale = None if w.k_scale is None else w.k_scale.to(self.dev).float().contiguous()
        self.v_scale = None if w.v_scale is None else w.v_scale.to(self.dev).float().contiguous()
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev) if with_err_word else None
        self.desc = pkv.make_desc(w.num_blocks, wl.PAGE, cfg.kv_heads, cfg.q_heads,
                                  cfg.head_dim, _CODE[cfg.cache], self.k_scale, self.v_scale,
                                  self.err)
        self.hint = hint
        nbytes = pkv.pkv_decode_workspace_bytes(self.desc, cfg.batch, w.max_blocks_per_seq, hint)
        assert nbytes > 0
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=self.dev)

    def append(self):
        pkv.pkv_kv_append(self.desc, self.k_cache, self.v_cache, self.slot, self.k_new,
                          self.v_new)

    def decode(self, out_dtype: str = "f32") -> torch.Tensor:
        cfg = self.w.cfg
        out = torch.empty(cfg.batch, cfg.q_heads, cfg.head_dim, dtype=_DT[out_dtype],
                          device=self.dev)
        pkv.pkv_paged_decode_attention(self.desc, self.q, self.k_cache, self.v_cache,
                                       self.tables, self.ctx, cfg.softmax_scale, out,
                                       self.workspace, self.hint)
        return out

    def step(self, out_dtype: str = "f32", fused: bool = True) -> torch.Tensor:
        """One decode step; fused uses pkv_decode_step, else the two calls."""
        if not fused:
            self.append()
            return self.decode(out_dtype)
        cfg = self.w.cfg
        out = torch.empty(cfg.batch, cfg.q_heads, cfg.head_dim, dtype=_DT[out_dtype],
                          device=self.dev)
        pkv.pkv_decode_step(self.desc, self.q, self.k_cache, self.v_cache, self.slot,
                            self.k_new, self.v_new, self.tables, self.ctx, cfg.softmax_scale,
                            out, self.workspace, self.hint)
        return out

    def step_one_kernel(self, out_dtype: str = "f32", overlap: bool = False) -> torch.Tensor:
        """One decode step as a single kernel (pkv_decode_step_fused): each new
        row lands at its sequence's newest position."""
        cfg = self.w.cfg
        out = torch.empty(cfg.batch, cfg.q_heads, cfg.head_dim, dtype=_DT[out_dtype],
                          device=self.dev)
        pkv.pkv_decode_step_fused(self.desc, self.q, self.k_cache, self.v_cache, self.k_new,
                                  self.v_new, self.tables, self.ctx, cfg.softmax_scale, out,
                                  self.workspace, self.hint, overlap=overlap)
        return out

    def err_code(self) -> int:
        return 0 if self.err is None else int(self.err.item())


def assert_close(got: np.ndarray, ref: np.ndarray, cfg, out_dtype: str, what: str = ""):
    """The parity bar: fp32 outputs within the tolerance; 16-bit outputs within
    the tolerance plus half an output ulp (the output rounding itself)."""
    tol = tolerance(cfg)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if out_dtype == "f32":
        bound = np.full_like(ref, tol)
    else:
        bound = tol + half_ulp(ref, _DT[out_dtype])
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of bound; max abs err "
                           f"{err.max():.3e} (tol {tol})")
    return float(err.max())


def assert_same_rounding(a, b, what: str = ""):
    """Two runs of the same decode: equal up to the order in which fp32
    partial sums were added (each page goes to whichever warp is free, so
    runs differ in the last bits).  fp32 outputs within 1e-5 + 1e-5 |a|
    (reordering a few thousand fp32 terms moves a sum by ~1e-6); 16-bit
    outputs within one unit in the last place of their type."""
    if isinstance(a, torch.Tensor):
        dt = a.dtype
        a = a.double().cpu().numpy()
        b = b.double().cpu().numpy()
    else:
        dt = torch.float32
    assert a.shape == b.shape
    assert np.array_equal(np.isfinite(a), np.isfinite(b)), f"{what}: finiteness differs"
    d = np.abs(a - b)
    if dt == torch.float32:
        bound = 1e-5 + 1e-5 * np.abs(a)
    else:
        bound = 2 * half_ulp(np.maximum(np.abs(a), np.abs(b)), dt)
    bad = d > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements differ beyond rounding; max {d.max():.3e}"
