"""Python binding of libpkv.so: paged-KV single-token decode attention for GB300.

Argument marshalling only.  Every step of the decode path runs in the CUDA
kernels behind the C ABI declared in ``include/pkv.h``; torch supplies device
memory and streams.  The functions carry the C names:

    pkv_kv_append                 write new K/V rows into their cache slots
    pkv_decode_workspace_bytes    workspace size for a decode call
    pkv_decode_workspace_bytes_multi  the same for q_len query tokens per
                                  sequence (multi-query and windowed calls)
    pkv_paged_decode_attention    one (1,N) attention row per query head
    pkv_paged_decode_attention_multi  q_len new tokens per sequence, causal
    pkv_paged_decode_attention_window  the same under a sliding window with
                                  attention sinks
    pkv_paged_prefill_attention   a chunk of new tokens per sequence, causal,
                                  on the tensor cores (tcgen05)
    pkv_decode_step               both, validated together, the attention
                                  kernel overlapping the append's tail
    pkv_decode_step_fused         both in one kernel (new token at its
                                  sequence's newest position)
    pkv_copy_blocks               copy whole blocks (copy-on-write of a
                                  shared prefix's last block)
    pkv_paged_decode_attention_noalloc  decode without a caller workspace
    pkv_kv_bytes_per_token        cache bytes per token (host helper)
    pkv_status_string, pkv_version

If the library is missing it is built on first use with nvcc; if that is not
possible every call raises.  There is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "PkvError", "CacheDesc", "make_desc", "load_library", "library_path",
    "pkv_kv_append", "pkv_decode_workspace_bytes", "pkv_paged_decode_attention",
    "pkv_decode_step", "pkv_kv_bytes_per_token", "pkv_status_string", "pkv_version",
    "pkv_paged_decode_attention_noalloc", "PKV_NOALLOC_SCRATCH_BYTES", "pkv_copy_blocks",
    "pkv_decode_workspace_bytes_multi",
    "pkv_paged_decode_attention_multi", "pkv_paged_decode_attention_window",
    "pkv_decode_step_fused", "pkv_paged_prefill_attention",
    "PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED", "PKV_ERR_WORKSPACE",
    "PKV_ERR_CUDA", "PKV_ERR_BOUNDS", "PKV_ERR_TIMEOUT",
    "PKV_F16", "PKV_BF16", "PKV_FP8_E4M3", "PKV_F32", "PKV_FP8_E4M3_TOKEN", "PKV_STEP_OVERLAP",
    "EXPORTED_SYMBOLS",
]

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE = 0, 1, 2, 3
PKV_ERR_CUDA, PKV_ERR_BOUNDS, PKV_ERR_TIMEOUT = 4, 5, 6
PKV_F16, PKV_BF16, PKV_FP8_E4M3, PKV_F32, PKV_FP8_E4M3_TOKEN = 0, 1, 2, 3, 4
PKV_STEP_OVERLAP = 1

EXPORTED_SYMBOLS = (
    "pkv_kv_append", "pkv_decode_workspace_bytes", "pkv_paged_decode_attention",
    "pkv_decode_step", "pkv_kv_bytes_per_token", "pkv_status_string", "pkv_version",
    "pkv_paged_decode_attention_noalloc", "pkv_copy_blocks", "pkv_paged_decode_attention_multi",
    "pkv_paged_decode_attention_window", "pkv_decode_step_fused", "pkv_paged_prefill_attention",
    "pkv_decode_workspace_bytes_multi",
)
PKV_NOALLOC_SCRATCH_BYTES = 32 << 20

_DTYPE_CODE = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16,
               torch.uint8: PKV_FP8_E4M3, torch.float32: PKV_F32}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPE_CODE[torch.float8_e4m3fn] = PKV_FP8_E4M3


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pkv_status_string(status)}")


class CacheDesc(ctypes.Structure):
    """Mirror of ``pkv_cache_desc`` (include/pkv.h)."""
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("num_blocks", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("cache_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("err_word", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libpkv.so (building it with nvcc if absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        lib = ctypes.CDLL(path)
        P, I32, U64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
        D = ctypes.POINTER(CacheDesc)
        lib.pkv_kv_append.restype = I32
        lib.pkv_kv_append.argtypes = [D, P, P, P, P, P, I32, I32, P]
        lib.pkv_decode_workspace_bytes.restype = SZ
        lib.pkv_decode_workspace_bytes.argtypes = [D, I32, I32, I32]
        lib.pkv_decode_workspace_bytes_multi.restype = SZ
        lib.pkv_decode_workspace_bytes_multi.argtypes = [D, I32, I32, I32, I32]
        lib.pkv_paged_decode_attention.restype = I32
        lib.pkv_paged_decode_attention.argtypes = [D, P, P, P, P, P, I32, I32, I32,
                                                   ctypes.c_float, P, I32, I32, P, SZ, P]
        lib.pkv_decode_step.restype = I32
        lib.pkv_decode_step.argtypes = [D, P, P, P, P, P, P, I32, P, P, I32, I32, I32,
                                        ctypes.c_float, P, I32, I32, P, SZ, P]
        lib.pkv_paged_decode_attention_noalloc.restype = I32
        lib.pkv_paged_decode_attention_noalloc.argtypes = [D, P, P, P, P, P, I32, I32, I32,
                                                           ctypes.c_float, P, I32, I32, P]
        lib.pkv_paged_decode_attention_multi.restype = I32
        lib.pkv_paged_decode_attention_multi.argtypes = [D, P, P, P, P, P, I32, I32, I32, I32,
                                                         ctypes.c_float, P, I32, I32, P, SZ, P]
        lib.pkv_paged_prefill_attention.restype = I32
        lib.pkv_paged_prefill_attention.argtypes = [D, P, P, P, P, P, P, I32, I32, I32, I32,
                                                    ctypes.c_float, P, I32, I32, P]
        lib.pkv_decode_step_fused.restype = I32
        lib.pkv_decode_step_fused.argtypes = [D, P, P, P, P, P, I32, P, P, I32, I32, I32,
                                              ctypes.c_float, P, I32, I32, P, SZ, I32, P]
        lib.pkv_paged_decode_attention_window.restype = I32
        lib.pkv_paged_decode_attention_window.argtypes = [D, P, P, P, P, P, I32, I32, I32, I32,
                                                          I32, I32, ctypes.c_float, P, I32, I32,
                                                          P, SZ, P]
        lib.pkv_copy_blocks.restype = I32
        lib.pkv_copy_blocks.argtypes = [D, P, P, P, P, I32, P]
        lib.pkv_kv_bytes_per_token.restype = U64
        lib.pkv_kv_bytes_per_token.argtypes = [I32, I32, I32, I32]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_status_string.argtypes = [I32]
        lib.pkv_version.restype = I32
        lib.pkv_version.argtypes = []
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _dev_ptr(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(num_blocks: int, page_size: int, num_kv_heads: int, num_q_heads: int,
              head_dim: int, cache_dtype: int, k_scale: Optional[torch.Tensor] = None,
              v_scale: Optional[torch.Tensor] = None,
              err_word: Optional[torch.Tensor] = None) -> CacheDesc:
    """Build a ``pkv_cache_desc``.  Tensors passed here must outlive its use."""
    d = CacheDesc()
    d.struct_size = ctypes.sizeof(CacheDesc)
    d.num_blocks = num_blocks
    d.page_size = page_size
    d.num_kv_heads = num_kv_heads
    d.num_q_heads = num_q_heads
    d.head_dim = head_dim
    d.cache_dtype = cache_dtype
    d.k_scale = k_scale.data_ptr() if k_scale is not None else None
    d.v_scale = v_scale.data_ptr() if v_scale is not None else None
    d.err_word = err_word.data_ptr() if err_word is not None else None
    return d


def _check(status: int, where: str):
    if status != PKV_OK:
        raise PkvError(status, where)


def pkv_kv_append(desc: CacheDesc, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  slot_mapping: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  stream=None) -> None:
    """k, v: [T][Hkv][d] (fp16/bf16); slot_mapping: int64 [T]."""
    lib = load_library()
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if k.dtype != v.dtype or k.shape != v.shape:
        raise ValueError("k and v must match")
    st = lib.pkv_kv_append(ctypes.byref(desc), _dev_ptr(k_cache, "k_cache"),
                           _dev_ptr(v_cache, "v_cache"), _dev_ptr(slot_mapping, "slot_mapping"),
                           _dev_ptr(k, "k"), _dev_ptr(v, "v"), int(k.shape[0]),
                           _DTYPE_CODE.get(k.dtype, -1), _stream_handle(stream, k.device))
    _check(st, "pkv_kv_append")


def pkv_copy_blocks(desc: CacheDesc, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    src_blocks: torch.Tensor, dst_blocks: torch.Tensor, stream=None) -> None:
    """Block dst_blocks[i] of both caches receives block src_blocks[i] (int32)."""
    lib = load_library()
    if src_blocks.dtype != torch.int32 or dst_blocks.dtype != torch.int32:
        raise ValueError("block ids must be int32")
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks must have the same length")
    st = lib.pkv_copy_blocks(ctypes.byref(desc), _dev_ptr(k_cache, "k_cache"),
                             _dev_ptr(v_cache, "v_cache"), _dev_ptr(src_blocks, "src_blocks"),
                             _dev_ptr(dst_blocks, "dst_blocks"), int(src_blocks.numel()),
                             _stream_handle(stream, k_cache.device))
    _check(st, "pkv_copy_blocks")


def pkv_decode_workspace_bytes(desc: CacheDesc, batch: int, max_blocks_per_seq: int,
                               max_context_len_hint: int = 0) -> int:
    lib = load_library()
    return int(lib.pkv_decode_workspace_bytes(ctypes.byref(desc), int(batch),
                                              int(max_blocks_per_seq),
                                              int(max_context_len_hint)))


def pkv_decode_workspace_bytes_multi(desc: CacheDesc, batch: int, q_len: int,
                                     max_blocks_per_seq: int,
                                     max_context_len_hint: int = 0) -> int:
    lib = load_library()
    return int(lib.pkv_decode_workspace_bytes_multi(ctypes.byref(desc), int(batch), int(q_len),
                                                    int(max_blocks_per_seq),
                                                    int(max_context_len_hint)))


def pkv_paged_decode_attention(desc: CacheDesc, q: torch.Tensor, k_cache: torch.Tensor,
                               v_cache: torch.Tensor, block_tables: torch.Tensor,
                               context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                               workspace: torch.Tensor, max_context_len_hint: int = 0,
                               stream=None) -> None:
    """q/out: [B][Hq][d]; block_tables int32 [B][MBS]; context_lens int32 [B]."""
    lib = load_library()
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    st = lib.pkv_paged_decode_attention(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(context_lens, "context_lens"), B, mbs, int(max_context_len_hint),
        float(scale), _dev_ptr(out, "out"), _DTYPE_CODE.get(q.dtype, -1),
        _DTYPE_CODE.get(out.dtype, -1), _dev_ptr(workspace, "workspace"),
        int(workspace.numel() * workspace.element_size()), _stream_handle(stream, q.device))
    _check(st, "pkv_paged_decode_attention")


def pkv_paged_decode_attention_multi(desc: CacheDesc, q: torch.Tensor, k_cache: torch.Tensor,
                                     v_cache: torch.Tensor, block_tables: torch.Tensor,
                                     context_lens: torch.Tensor, scale: float,
                                     out: torch.Tensor, workspace: torch.Tensor,
                                     max_context_len_hint: int = 0, stream=None) -> None:
    """q/out: [B][q_len][Hq][d], the last q_len tokens of each sequence, causal
    among themselves; block_tables int32 [B][MBS]; context_lens int32 [B]."""
    lib = load_library()
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if q.dim() != 4 or out.shape != q.shape:
        raise ValueError("q and out must be [B][q_len][Hq][d]")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    st = lib.pkv_paged_decode_attention_multi(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(context_lens, "context_lens"), B, int(q.shape[1]), mbs,
        int(max_context_len_hint), float(scale), _dev_ptr(out, "out"),
        _DTYPE_CODE.get(q.dtype, -1), _DTYPE_CODE.get(out.dtype, -1),
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _stream_handle(stream, q.device))
    _check(st, "pkv_paged_decode_attention_multi")


def pkv_paged_decode_attention_window(desc: CacheDesc, q: torch.Tensor, k_cache: torch.Tensor,
                                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                                      context_lens: torch.Tensor, window: int, sinks: int,
                                      scale: float, out: torch.Tensor, workspace: torch.Tensor,
                                      max_context_len_hint: int = 0, stream=None) -> None:
    """As pkv_paged_decode_attention_multi, token t seeing only positions
    t - window + 1 .. t and the first `sinks` positions (window 0: no window)."""
    lib = load_library()
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if q.dim() != 4 or out.shape != q.shape:
        raise ValueError("q and out must be [B][q_len][Hq][d]")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    st = lib.pkv_paged_decode_attention_window(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(context_lens, "context_lens"), B, int(q.shape[1]), int(window), int(sinks),
        mbs, int(max_context_len_hint), float(scale), _dev_ptr(out, "out"),
        _DTYPE_CODE.get(q.dtype, -1), _DTYPE_CODE.get(out.dtype, -1),
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _stream_handle(stream, q.device))
    _check(st, "pkv_paged_decode_attention_window")


def pkv_decode_step(desc: CacheDesc, q: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, slot_mapping: torch.Tensor, k: torch.Tensor,
                    v: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                    scale: float, out: torch.Tensor, workspace: torch.Tensor,
                    max_context_len_hint: int = 0, stream=None) -> None:
    """Append one token per sequence (k, v: [B][Hkv][d]) then attend."""
    lib = load_library()
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    if k.shape[0] != B or v.shape != k.shape or slot_mapping.shape[0] != B:
        raise ValueError("k, v and slot_mapping need one row per sequence")
    st = lib.pkv_decode_step(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(slot_mapping, "slot_mapping"),
        _dev_ptr(k, "k"), _dev_ptr(v, "v"), _DTYPE_CODE.get(k.dtype, -1),
        _dev_ptr(block_tables, "block_tables"), _dev_ptr(context_lens, "context_lens"),
        B, mbs, int(max_context_len_hint), float(scale), _dev_ptr(out, "out"),
        _DTYPE_CODE.get(q.dtype, -1), _DTYPE_CODE.get(out.dtype, -1),
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _stream_handle(stream, q.device))
    _check(st, "pkv_decode_step")


def pkv_paged_prefill_attention(desc: CacheDesc, q: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, block_tables: torch.Tensor,
                                context_lens: torch.Tensor, q_start: torch.Tensor,
                                max_q_len: int, scale: float, out: torch.Tensor,
                                stream=None) -> None:
    """q/out: [total_q][Hq][d]; sequence b's rows q_start[b] .. q_start[b+1]-1
    are its last positions, causal; q_start int32 [B+1] on the device."""
    lib = load_library()
    for t, n in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                 (q_start, "q_start")):
        if t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must be [total_q][Hq][d]")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    if q_start.numel() != B + 1:
        raise ValueError("q_start needs batch + 1 entries")
    st = lib.pkv_paged_prefill_attention(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(context_lens, "context_lens"), _dev_ptr(q_start, "q_start"), B,
        int(q.shape[0]), int(max_q_len), mbs, float(scale), _dev_ptr(out, "out"),
        _DTYPE_CODE.get(q.dtype, -1), _DTYPE_CODE.get(out.dtype, -1),
        _stream_handle(stream, q.device))
    _check(st, "pkv_paged_prefill_attention")


def pkv_decode_step_fused(desc: CacheDesc, q: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                          out: torch.Tensor, workspace: torch.Tensor,
                          max_context_len_hint: int = 0, stream=None,
                          overlap: bool = False) -> None:
    """One kernel: sequence b's new token (k[b], v[b]: [B][Hkv][d]) goes to its
    position context_lens[b] - 1, then every sequence attends.  overlap sets
    PKV_STEP_OVERLAP: context_lens and block_tables are not written by the
    kernel launched just before on the stream."""
    lib = load_library()
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    if k.shape[0] != B or v.shape != k.shape:
        raise ValueError("k and v need one row per sequence")
    st = lib.pkv_decode_step_fused(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
        _DTYPE_CODE.get(k.dtype, -1), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(context_lens, "context_lens"), B, mbs, int(max_context_len_hint),
        float(scale), _dev_ptr(out, "out"), _DTYPE_CODE.get(q.dtype, -1),
        _DTYPE_CODE.get(out.dtype, -1), _dev_ptr(workspace, "workspace"),
        int(workspace.numel() * workspace.element_size()), PKV_STEP_OVERLAP if overlap else 0,
        _stream_handle(stream, q.device))
    _check(st, "pkv_decode_step_fused")


def pkv_paged_decode_attention_noalloc(desc: CacheDesc, q: torch.Tensor,
                                       k_cache: torch.Tensor, v_cache: torch.Tensor,
                                       block_tables: torch.Tensor, context_lens: torch.Tensor,
                                       scale: float, out: torch.Tensor,
                                       max_context_len_hint: int = 0, stream=None) -> None:
    """Decode attention on the library's fixed device scratch (no workspace).

    For callers that cannot allocate device memory at call time.  Calls that
    overlap on the GPU share the scratch and race; the first call on a device
    should come before any stream capture."""
    lib = load_library()
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    B, mbs = int(block_tables.shape[0]), int(block_tables.shape[1])
    st = lib.pkv_paged_decode_attention_noalloc(
        ctypes.byref(desc), _dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(context_lens, "context_lens"), B, mbs, int(max_context_len_hint),
        float(scale), _dev_ptr(out, "out"), _DTYPE_CODE.get(q.dtype, -1),
        _DTYPE_CODE.get(out.dtype, -1), _stream_handle(stream, q.device))
    _check(st, "pkv_paged_decode_attention_noalloc")


def pkv_kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return int(load_library().pkv_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes))


def pkv_status_string(status: int) -> str:
    return load_library().pkv_status_string(int(status)).decode()


def pkv_version() -> int:
    return int(load_library().pkv_version())


@dataclass
class DecodeBuffers:
    """Zero-filled workspace sized for a launch shape (convenience for callers)."""
    workspace: torch.Tensor

    @staticmethod
    def allocate(desc: CacheDesc, batch: int, max_blocks_per_seq: int,
                 max_context_len_hint: int = 0, device="cuda") -> "DecodeBuffers":
        n = pkv_decode_workspace_bytes(desc, batch, max_blocks_per_seq, max_context_len_hint)
        if n == 0:
            raise PkvError(PKV_ERR_INVALID_ARG, "pkv_decode_workspace_bytes")
        return DecodeBuffers(torch.zeros(n, dtype=torch.uint8, device=device))
