"""Context-parallel split of long global sequences on the GPU, its ranks run
one after another on one GPU (separate launches; no kernel waits on another).

Each emulated rank holds a contiguous share of every sequence's pages
(cp.shard_pages) in a pool of its own, pages renumbered from 0, filled by
gw_kv_append at the tokens' absolute positions, and runs
gw_decode_attn_global_lse; gw_merge_lse merges the ranks' outputs by their
log-sum-exp.  The merged rows must match the float64 oracle over the whole
sequence and the unsplit call (attention tolerance), and the unsplit call's
log-sum-exp must match the oracle's.
"""

import numpy as np
import pytest
import torch

from oracle import attention
from paged_hybrid_attention_gb300 import cp, gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _layer():
    sp = synth.spec("long_global")
    lens = np.array([131072, 5000, 33], np.int32)
    return synth.Layer(synth.custom("cp", sp.seed, 32, lens, [1, 1, 1], sp.families, 0, 1), "global", layer=100)


def _rank_part(layer, table, world, rank, q):
    """This rank's pool, block table and key counts; returns (out, lse)."""
    sp = layer.spec
    shards = [cp.shard_pages(int(L), world, rank) for L in sp.lens]
    npages = [p1 - p0 for p0, p1, _, _ in shards]
    base = np.concatenate([[0], np.cumsum(npages)]).astype(np.int64)
    pool = gw.KVPool("folded", "bf16", max(1, int(base[-1])))
    bt = np.full((len(shards), max(1, max(npages))), -1, np.int32)
    for s, (p0, p1, k0, k1) in enumerate(shards):
        bt[s, :p1 - p0] = base[s] + np.arange(p1 - p0)
        if k1 == k0:
            continue
        pos, k, v = layer.kv(s)
        m = (pos >= k0) & (pos < k1)
        slot = ((base[s] + pos[m] // 16 - p0) * 16 + pos[m] % 16).astype(np.int32)
        gw.kv_append(pool, G.bits_to_cuda_bf16(k[m]), G.bits_to_cuda_bf16(v[m]), G.i32(slot), G.i32(pos[m]), table)
    n_keys = G.i32([k1 - k0 for _, _, k0, k1 in shards])
    ws = gw.alloc_workspace(pool, 32, len(shards), bt.shape[1], 1, 1)
    return cp.local_attention(pool, q, G.i32(bt), n_keys, ws)


@pytest.mark.parametrize("world", [2, 3])
def test_split_over_ranks_matches_oracle_and_unsplit(world):
    layer = _layer()
    sp = layer.spec
    table_np = G.oracle_table(1e6, 128, 512, int(sp.lens.max()) + 1)
    table = table_np.cuda()
    q = G.bits_to_cuda_bf16(layer.queries())
    parts = [_rank_part(layer, table, world, r, q) for r in range(world)]
    merged, lse = cp.merge([p[0] for p in parts], [p[1] for p in parts])
    # the unsplit call, with its log-sum-exp
    pool = G.new_pool(layer)
    G.append(layer, pool, table)
    ws = gw.alloc_workspace(pool, 32, layer.B, layer.block_table.shape[1], 1, 1)
    full = torch.empty_like(q)
    full_lse = torch.empty(layer.B, 32, dtype=torch.float32, device="cuda")
    gw.decode_attn_global_lse(pool, q, full, full_lse, G.i32(layer.cu_rows()), G.i32(sp.lens),
                              G.i32(layer.block_table), ws)
    torch.cuda.synchronize()
    ref = H.build_pool(layer, table_np.numpy())
    got, got_full = G.to_f64(merged), G.to_f64(full)
    for s in range(layer.B):
        want = H.oracle_rows(layer, ref, s)
        for x in (got[s:s + 1], got_full[s:s + 1]):
            mx, rl = G.errors(x, want)
            assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, mx, rl)
        # log-sum-exp of the oracle: ln sum_j exp(scale q.k_j)
        from oracle import pages
        rows = pages.read_global_rows(ref, "folded", layer.block_table[s], np.arange(int(sp.lens[s])))
        K, V = attention.rebuild_global_k(rows)
        m, l, _ = attention.partial(H.q64(layer, s)[0], K[:, None], V[:, None], 1.0 / np.sqrt(512))
        want_lse = m + np.log(l)
        for x in (lse[s].double().cpu().numpy(), full_lse[s].double().cpu().numpy()):
            assert np.max(np.abs(x - want_lse)) < 1e-3 * max(1.0, float(np.max(np.abs(want_lse))))


def test_merge_skips_empty_parts_and_keeps_one_part_exact():
    """A part whose keys are empty (lse -inf) is not read (its bytes may be
    NaN); a single part is returned unchanged."""
    rows, heads = 5, 8
    gen = torch.Generator(device="cuda").manual_seed(3)
    o = torch.randn(rows, heads, 512, generator=gen, device="cuda").to(torch.bfloat16)
    lse = torch.randn(rows, heads, generator=gen, device="cuda")
    nan = torch.full_like(o, float("nan"))
    empty = torch.full_like(lse, float("-inf"))
    out, l2 = cp.merge([o, nan], [lse, empty])
    one, l1 = cp.merge([o], [lse])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), o.view(torch.int16))
    assert torch.equal(one.view(torch.int16), o.view(torch.int16))
    assert torch.allclose(l2, lse) and torch.allclose(l1, lse)
