"""Copy-on-write for shared prefixes on the GPU: pkv_copy_blocks against the
oracle's block copy (bit-exact), and a shared-prefix decode through the CUDA
path against the oracle's attention on the logical rows.

[AP] "Paged attention: stop reserving empty tables" (sequences share the
blocks of a common beginning, copying only a block one of them would change);
[KVFA] PagedAttention section (sharing a prefix shares ceil(prefix / P)
blocks, so the last may be partly filled).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_250_gb300 as pkv

P = 16


def _ids(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


@pytest.mark.gpu
@pytest.mark.parametrize("cache", ["bf16", "e4m3"])
def test_copy_blocks_bit_exact_and_bad_ids_reported(cache):
    g = torch.Generator().manual_seed(31)
    NB, Hkv, d = 13, 2, 128
    shape = (NB, Hkv, P, d)
    if cache == "bf16":
        k = torch.randn(shape, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, generator=g).to(torch.bfloat16)
        code, scales = pkv.PKV_BF16, (None, None)
    else:
        k = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
        v = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
        code = pkv.PKV_FP8_E4M3
        scales = (torch.ones(Hkv, device="cuda"), torch.ones(Hkv, device="cuda"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = pkv.make_desc(NB, P, Hkv, 8, d, code, scales[0], scales[1], err)
    src = [2, 9, 11, 5, 4]
    dst = [0, 7, 12, 10, 13]  # the last pair is outside the pool
    kc, vc = k.cuda(), v.cuda()
    pkv.pkv_copy_blocks(desc, kc, vc, _ids(src), _ids(dst))
    torch.cuda.synchronize()
    view = (lambda t: t.view(torch.int16)) if cache == "bf16" else (lambda t: t)
    want_k = oracle.copy_blocks(view(k).numpy(), src, dst)
    want_v = oracle.copy_blocks(view(v).numpy(), src, dst)
    assert np.array_equal(view(kc.cpu()).numpy(), want_k)
    assert np.array_equal(view(vc.cpu()).numpy(), want_v)
    assert int(err.item()) == pkv.PKV_ERR_BOUNDS
    # nothing to copy: no launch, no change
    pkv.pkv_copy_blocks(desc, kc, vc, _ids([]), _ids([]))


@pytest.mark.gpu
def test_shared_prefix_copy_on_write_decode():
    # A and B share a 40-token prefix in blocks 3, 8, 1 (block 1 holds 8
    # tokens); B's next token would change block 1, so B gets a copy (block 6)
    # first; then both append and attend over 41 tokens.
    g = torch.Generator().manual_seed(32)
    NB, Hkv, Hq, d = 12, 2, 8, 128
    grp = Hq // Hkv
    scale = d ** -0.5
    prefix_k = torch.randn(40, Hkv, d, generator=g).to(torch.bfloat16)
    prefix_v = torch.randn(40, Hkv, d, generator=g).to(torch.bfloat16)
    new_k = torch.randn(2, Hkv, d, generator=g).to(torch.bfloat16)  # rows of A, B
    new_v = torch.randn(2, Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(2, Hq, d, generator=g).to(torch.bfloat16)
    k_cache = torch.full((NB, Hkv, P, d), float("nan")).to(torch.bfloat16)
    v_cache = torch.full((NB, Hkv, P, d), float("nan")).to(torch.bfloat16)
    table_a = [3, 8, 1]
    for t in range(40):
        k_cache[table_a[t // P], :, t % P] = prefix_k[t]
        v_cache[table_a[t // P], :, t % P] = prefix_v[t]
    table_b = [3, 8, 6]
    kc, vc = k_cache.cuda(), v_cache.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = pkv.make_desc(NB, P, Hkv, Hq, d, pkv.PKV_BF16, None, None, err)
    pkv.pkv_copy_blocks(desc, kc, vc, _ids([1]), _ids([6]))
    slots = torch.tensor([1 * P + 8, 6 * P + 8], dtype=torch.int64, device="cuda")
    pkv.pkv_kv_append(desc, kc, vc, slots, new_k.cuda(), new_v.cuda())
    tables = _ids([table_a, table_b])
    ctx = _ids([41, 41])
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(desc, 2, 3, 0), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(2, Hq, d, dtype=torch.float32, device="cuda")
    pkv.pkv_paged_decode_attention(desc, q.cuda(), kc, vc, tables, ctx, scale, out, ws, 0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().double().numpy()
    for s in range(2):
        K = torch.cat([prefix_k, new_k[s:s + 1]]).double().numpy()
        V = torch.cat([prefix_v, new_v[s:s + 1]]).double().numpy()
        for hq in range(Hq):
            want = oracle.attend_row(q[s, hq].double().numpy(), K[:, hq // grp], V[:, hq // grp],
                                     scale)
            assert np.abs(got[s, hq] - want).max() <= 2e-3
    # the shared blocks are untouched apart from A's append into its own block
    assert torch.equal(kc[3].cpu().view(torch.int16), k_cache[3].view(torch.int16))
