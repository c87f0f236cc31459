"""Seeded synthetic decode-step workloads.

This module only draws inputs.  It holds none of the attention arithmetic and
none of the FP8 codec: both the CUDA path and the CPU oracle consume what it
produces.  The shapes, value distributions and table structure follow the
workloads the pages describe (Llama-3-8B / 70B-shaped GQA layers, an FP8
cache, a 32-KV-head 7B shape, long reasoning contexts) and the paged layout
of "KV Cache & Flash Attention." (kvcache-7e2.pages.dev), PagedAttention
section: 16-token blocks, a shared pool, one block table per sequence.

Recipe (per workload):
  * context lengths: fixed, or uniform integers in [lo, hi] (CPU generator);
  * the pool holds exactly the blocks the sequences need plus spares; block
    ids are a random permutation of the pool dealt out in sequence order
    (or the identity for the tiny case);
  * q, k, v ~ N(0, 1), rounded once to the stored dtype;
  * the cache holds every token but the newest of each sequence; the newest
    token's k/v rows and its slot are returned for the append step;
  * unused slots and spare blocks hold a poison value (NaN, or the E4M3 NaN
    code 0x7F), so a read outside the context shows up in the output;
  * FP8 cache: one fp32 scale per KV head for K and one for V, amax/448 over
    that head's drawn values; stored bytes are torch's float8_e4m3fn cast of
    value / scale (a library routine, used here only to draw input bytes);
  * FP8 cache with per-token scales ("e4m3tok"): the same, with one scale per
    (token, KV head) row, amax/448 over the row, held in one scale pool
    [NB][Hkv][2][P] (K scales, then V scales; NaN in unused slots).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple, Union

import torch

PAGE = 16
E4M3_MAX = 448.0
E4M3_NAN = 0x7F


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    cache: str                       # "f16" | "bf16" | "e4m3" | "e4m3tok"
    ctx: Union[int, Tuple[int, int]]  # fixed length or (lo, hi) uniform
    table: str = "permuted"          # "permuted" | "identity"
    seed: int = 0
    spare_blocks: int = 0
    q_dtype: str = ""                # default: cache dtype, bf16 for e4m3
    scale: Optional[float] = None    # default 1/sqrt(head_dim)
    description: str = ""

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def qdt(self) -> torch.dtype:
        name = self.q_dtype or ("bf16" if self.is_fp8 else self.cache)
        return {"f16": torch.float16, "bf16": torch.bfloat16}[name]

    @property
    def is_fp8(self) -> bool:
        return self.cache in ("e4m3", "e4m3tok")

    @property
    def cache_elem_bytes(self) -> int:
        return 1 if self.is_fp8 else 2


CONFIGS = {
    c.name: c
    for c in [
        DecodeConfig("tiny_b1_h4x1_d64_f16_ctx256", 1, 4, 1, 64, "f16", 256,
                     table="identity", seed=0, scale=1.0 / 8.0,
                     description="batch 1, 4 query heads on 1 KV head, d 64, fp16, "
                                 "context 256 (255 cached + 1 appended), identity table"),
        DecodeConfig("llama3_8b_b32_ctx1-4096_bf16", 32, 32, 8, 128, "bf16", (1, 4096),
                     seed=1, spare_blocks=64,
                     description="Llama-3-8B-shaped layer: batch 32, 32/8 heads, d 128, bf16, "
                                 "context uniform in [1, 4096], permuted shared pool"),
        DecodeConfig("llama3_8b_b8_ctx8192_bf16", 8, 32, 8, 128, "bf16", 8192, seed=5,
                     spare_blocks=64,
                     description="Llama-3-8B-shaped layer, 8 sequences of 8192 tokens (the "
                                 "prefill workload: each sequence's last 2048 positions are "
                                 "its new chunk)"),
        DecodeConfig("llama3_70b_b8_ctx32768_bf16", 8, 64, 8, 128, "bf16", 32768, seed=2,
                     spare_blocks=64,
                     description="Llama-3-70B-shaped layer: batch 8, 64/8 heads, d 128, bf16, "
                                 "context 32768, permuted tables"),
        DecodeConfig("fp8_8b_b64_ctx8192_e4m3", 64, 32, 8, 128, "e4m3", 8192, seed=3,
                     spare_blocks=64,
                     description="8B shape, batch 64, context 8192, E4M3 cache with per-head "
                                 "fp32 scales, bf16 q and output"),
        DecodeConfig("fp8tok_8b_b64_ctx8192_e4m3", 64, 32, 8, 128, "e4m3tok", 8192, seed=3,
                     spare_blocks=64,
                     description="8B shape, batch 64, context 8192, E4M3 cache with one fp32 "
                                 "scale per token and KV head, bf16 q and output"),
        DecodeConfig("mha_7b_b64_ctx8192_bf16", 64, 32, 32, 128, "bf16", 8192, seed=3,
                     spare_blocks=64,
                     description="7B MHA shape, 32/32 heads, batch 64, context 8192, bf16"),
        DecodeConfig("reasoning_b1_ctx131072_bf16", 1, 32, 8, 128, "bf16", 131072, seed=4,
                     spare_blocks=64,
                     description="single 131072-token sequence, 32/8 heads, bf16"),
        DecodeConfig("reasoning_b4_ctx131072_bf16", 4, 32, 8, 128, "bf16", 131072, seed=4,
                     spare_blocks=64,
                     description="4 sequences of 131072 tokens, 32/8 heads, bf16"),
    ]
}


def small_config(name: str, batch: int, q_heads: int, kv_heads: int, head_dim: int,
                 cache: str, ctx, seed: int = 7, table: str = "permuted",
                 spare_blocks: int = 5, q_dtype: str = "") -> DecodeConfig:
    return DecodeConfig(name, batch, q_heads, kv_heads, head_dim, cache, ctx, table=table,
                        seed=seed, spare_blocks=spare_blocks, q_dtype=q_dtype)


@dataclass
class DecodeWorkload:
    cfg: DecodeConfig
    ctx: torch.Tensor            # int32 [B] (cpu)
    block_tables: torch.Tensor   # int32 [B][MBS] (cpu); -1 past each sequence's pages
    slot_mapping: torch.Tensor   # int64 [B] (cpu): slot of each sequence's newest token
    num_blocks: int
    q: torch.Tensor              # [B][Hq][d]
    k_new: torch.Tensor          # [B][Hkv][d] input dtype (bf16 for e4m3)
    v_new: torch.Tensor
    K_log: torch.Tensor          # [B][T][Hkv][d] drawn values, input dtype
    V_log: torch.Tensor
    K_stored: torch.Tensor       # [B][T][Hkv][d] stored values (uint8 codes for e4m3)
    V_stored: torch.Tensor
    k_cache: torch.Tensor        # [NB][Hkv][P][d] stored dtype (uint8 for e4m3)
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None  # fp32 [Hkv] (e4m3); [NB][Hkv][2][P] (e4m3tok)
    v_scale: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def to(self, device) -> "DecodeWorkload":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return replace(self, q=mv(self.q), k_new=mv(self.k_new), v_new=mv(self.v_new),
                       k_cache=mv(self.k_cache), v_cache=mv(self.v_cache),
                       k_scale=mv(self.k_scale), v_scale=mv(self.v_scale))


def _store_dtype(cache: str) -> torch.dtype:
    return {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8,
            "e4m3tok": torch.uint8}[cache]


def draw_context_lengths(cfg: DecodeConfig, gen: torch.Generator) -> torch.Tensor:
    if isinstance(cfg.ctx, int):
        return torch.full((cfg.batch,), cfg.ctx, dtype=torch.int32)
    lo, hi = cfg.ctx
    return torch.randint(lo, hi + 1, (cfg.batch,), generator=gen, dtype=torch.int64).to(torch.int32)


def deal_block_tables(ctx: torch.Tensor, spare: int, table: str, gen: torch.Generator,
                      max_blocks: Optional[int] = None):
    """Pool of sum(ceil(ctx/P)) + spare blocks; ids dealt out in sequence order."""
    nblk = [(int(c) + PAGE - 1) // PAGE for c in ctx.tolist()]
    NB = max(1, sum(nblk) + spare)
    ids = torch.randperm(NB, generator=gen).to(torch.int32) if table == "permuted" \
        else torch.arange(NB, dtype=torch.int32)
    mbs = max_blocks if max_blocks is not None else max(1, max(nblk, default=1))
    tables = torch.full((len(nblk), mbs), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = ids[off:off + n]
        off += n
    return tables, NB


def generate(cfg: DecodeConfig, device: Union[str, torch.device] = "cpu",
             max_blocks: Optional[int] = None,
             ctx_override: Optional[torch.Tensor] = None) -> DecodeWorkload:
    """Draw one decode step's inputs.  Values are drawn on `device`."""
    device = torch.device(device)
    g_host = torch.Generator().manual_seed(cfg.seed)
    ctx = ctx_override.to(torch.int32).cpu() if ctx_override is not None \
        else draw_context_lengths(cfg, g_host)
    tables, NB = deal_block_tables(ctx, cfg.spare_blocks, cfg.table, g_host, max_blocks)
    B, Hq, Hkv, d = cfg.batch, cfg.q_heads, cfg.kv_heads, cfg.head_dim
    T = max(1, int(ctx.max()))
    g_dev = torch.Generator(device=device).manual_seed(cfg.seed + 1000)
    in_dt = cfg.qdt if not cfg.is_fp8 else torch.bfloat16
    q = torch.randn(B, Hq, d, generator=g_dev, device=device).to(cfg.qdt)
    K_log = torch.randn(B, T, Hkv, d, generator=g_dev, device=device).to(in_dt)
    V_log = torch.randn(B, T, Hkv, d, generator=g_dev, device=device).to(in_dt)

    ctx_d = ctx.to(device=device, dtype=torch.int64)
    last = (ctx_d - 1).clamp(min=0)
    ar = torch.arange(B, device=device)
    k_new = K_log[ar, last].contiguous()
    v_new = V_log[ar, last].contiguous()
    tab_d = tables.to(device=device, dtype=torch.int64)
    slot = (tab_d[ar, torch.div(last, PAGE, rounding_mode="floor")] * PAGE + last % PAGE)
    slot = torch.where(ctx_d > 0, slot, torch.full_like(slot, -1))

    k_scale = v_scale = None
    extra = {}
    if cfg.cache == "e4m3tok":
        ks_tok = K_log.float().abs().amax(dim=3) / E4M3_MAX  # [B][T][Hkv]
        vs_tok = V_log.float().abs().amax(dim=3) / E4M3_MAX
        ks_tok = torch.where(ks_tok > 0, ks_tok, torch.ones_like(ks_tok))
        vs_tok = torch.where(vs_tok > 0, vs_tok, torch.ones_like(vs_tok))
        K_st = (K_log.float() / ks_tok[..., None]).clamp(-E4M3_MAX, E4M3_MAX)
        V_st = (V_log.float() / vs_tok[..., None]).clamp(-E4M3_MAX, E4M3_MAX)
        K_stored = K_st.to(torch.float8_e4m3fn).view(torch.uint8)
        V_stored = V_st.to(torch.float8_e4m3fn).view(torch.uint8)
        del K_st, V_st
        poison = E4M3_NAN
        extra = {"k_tok_scale": ks_tok, "v_tok_scale": vs_tok}
        k_scale = torch.full((NB, Hkv, 2, PAGE), float("nan"), dtype=torch.float32,
                             device=device)
    elif cfg.cache == "e4m3":
        k_scale = (K_log.float().abs().amax(dim=(0, 1, 3)) / E4M3_MAX).clamp(min=1e-12)
        v_scale = (V_log.float().abs().amax(dim=(0, 1, 3)) / E4M3_MAX).clamp(min=1e-12)
        K_st = (K_log.float() / k_scale[None, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
        V_st = (V_log.float() / v_scale[None, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
        K_stored = K_st.to(torch.float8_e4m3fn).view(torch.uint8)
        V_stored = V_st.to(torch.float8_e4m3fn).view(torch.uint8)
        del K_st, V_st
        poison = E4M3_NAN
    else:
        K_stored, V_stored = K_log, V_log
        poison = float("nan")

    sdt = _store_dtype(cfg.cache)
    k_cache = torch.full((NB, Hkv, PAGE, d), poison, dtype=sdt, device=device)
    v_cache = torch.full((NB, Hkv, PAGE, d), poison, dtype=sdt, device=device)
    # the cache as a prefill would have left it: every token but the newest
    bi, ti = [], []
    for b, c in enumerate(ctx.tolist()):
        if c > 1:
            bi.append(torch.full((c - 1,), b, dtype=torch.int64))
            ti.append(torch.arange(c - 1, dtype=torch.int64))
    if bi:
        bi_t = torch.cat(bi).to(device)
        ti_t = torch.cat(ti).to(device)
        blk = tab_d[bi_t, torch.div(ti_t, PAGE, rounding_mode="floor")]
        off = ti_t % PAGE
        k_cache[blk, :, off, :] = K_stored[bi_t, ti_t]
        v_cache[blk, :, off, :] = V_stored[bi_t, ti_t]
        if cfg.cache == "e4m3tok":
            k_scale[blk, :, 0, off] = extra["k_tok_scale"][bi_t, ti_t]
            k_scale[blk, :, 1, off] = extra["v_tok_scale"][bi_t, ti_t]
    return DecodeWorkload(cfg=cfg, ctx=ctx, block_tables=tables, slot_mapping=slot.cpu(),
                          num_blocks=NB, q=q, k_new=k_new, v_new=v_new, K_log=K_log,
                          V_log=V_log, K_stored=K_stored, V_stored=V_stored,
                          k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                          extra=extra)


def cache_bytes_per_step(cfg: DecodeConfig, ctx: torch.Tensor) -> int:
    """Bytes of K and V the attention must read for one step (all contexts)."""
    return int(ctx.to(torch.int64).sum()) * cfg.kv_heads * cfg.head_dim * 2 * cfg.cache_elem_bytes
