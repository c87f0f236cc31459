"""The seeded input generator: structure of the tables, slots and pool
(host logic, no GPU)."""
import numpy as np
import torch

from paged_kv_cache_250_gb300 import workloads as wl


def _gather(w, b, what="K"):
    """Rebuild a sequence's cached rows from the pool through its table."""
    n = int(w.ctx[b])
    cache = w.k_cache if what == "K" else w.v_cache
    rows = []
    for t in range(n - 1):
        blk = int(w.block_tables[b, t // wl.PAGE])
        rows.append(cache[blk, :, t % wl.PAGE])
    return torch.stack(rows) if rows else None


def test_tables_are_a_permutation_of_the_pool():
    cfg = wl.small_config("t", 6, 8, 2, 64, "bf16", (1, 200), seed=3, spare_blocks=4)
    w = wl.generate(cfg)
    ids = w.block_tables[w.block_tables >= 0].numpy()
    assert len(set(ids.tolist())) == len(ids)  # no block shared
    assert ids.min() >= 0 and ids.max() < w.num_blocks
    need = [(int(c) + 15) // 16 for c in w.ctx]
    assert len(ids) == sum(need) and w.num_blocks == sum(need) + 4
    for b, n in enumerate(need):
        assert (w.block_tables[b, :n] >= 0).all() and (w.block_tables[b, n:] == -1).all()
        # waste inside a sequence's last block is at most P - 1 tokens
        assert n * 16 - int(w.ctx[b]) <= 15


def test_slot_mapping_points_at_the_newest_position():
    cfg = wl.small_config("s", 5, 4, 1, 64, "f16", (1, 100), seed=5)
    w = wl.generate(cfg)
    for b in range(cfg.batch):
        pos = int(w.ctx[b]) - 1
        blk = int(w.block_tables[b, pos // 16])
        assert int(w.slot_mapping[b]) == blk * 16 + pos % 16
        assert torch.equal(w.k_new[b], w.K_log[b, pos])


def test_pool_holds_the_logical_rows_and_poison_elsewhere():
    cfg = wl.small_config("p", 4, 8, 2, 64, "bf16", (1, 70), seed=6, spare_blocks=3)
    w = wl.generate(cfg)
    used = np.zeros((w.num_blocks, 16), bool)
    for b in range(cfg.batch):
        n = int(w.ctx[b])
        g = _gather(w, b, "K")
        if g is not None:
            assert torch.equal(g, w.K_log[b, :n - 1])
            assert torch.equal(_gather(w, b, "V"), w.V_log[b, :n - 1])
        for t in range(n - 1):
            used[int(w.block_tables[b, t // 16]), t % 16] = True
    kc = w.k_cache.float().permute(0, 2, 1, 3).numpy()  # [NB][P][Hkv][d]
    assert np.isnan(kc[~used]).all() and not np.isnan(kc[used]).any()


def test_fp8_inputs_are_codes_with_head_scales():
    cfg = wl.small_config("f", 3, 8, 2, 128, "e4m3", (2, 40), seed=9)
    w = wl.generate(cfg)
    assert w.k_cache.dtype == torch.uint8 and w.k_scale.shape == (2,)
    assert w.K_stored.dtype == torch.uint8
    # every finite drawn value fits the scale: codes never hit NaN
    assert ((w.K_stored & 0x7F) != 0x7F).all() and ((w.V_stored & 0x7F) != 0x7F).all()
    # at least one code per head reaches the top of the range
    top = (w.K_stored & 0x7F).amax(dim=(0, 1, 3))
    assert (top >= 0x7D).all()


def test_generation_is_seeded():
    cfg = wl.CONFIGS["tiny_b1_h4x1_d64_f16_ctx256"]
    a, b = wl.generate(cfg), wl.generate(cfg)
    assert torch.equal(a.q, b.q) and torch.equal(a.K_log, b.K_log)
    assert torch.equal(a.block_tables, torch.arange(16, dtype=torch.int32)[None])
    assert int(a.ctx[0]) == 256 and int(a.slot_mapping[0]) == 255
