"""The split-KV combine on long sequences (many chunk groups) on the GPU.

The combine merges a sequence's chunks in groups of 16 (sums in chunk order
within a group, group sums in group order) and spreads the groups of one
sequence over 1, 4 or 8 warps, chosen from the call's bound on chunks per
sequence (the block table's width).  The output must agree with the float64
oracle and must not change, bit for bit, when a wider block table makes the
combine map the same sequence to other warps or more rounds.
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _widened(bt, width):
    wide = np.full((bt.shape[0], width), -1, dtype=np.int32)
    wide[:, :bt.shape[1]] = bt
    return wide


def _attend_with_table(layer, pool, bt):
    fam, sp = layer.fam, layer.spec
    q = G.bits_to_cuda_bf16(layer.queries())
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(sp.lens), bt.shape[1], 1, max(1, fam.window))
    args = (pool, q, out, G.i32(layer.cu_rows()), G.i32(sp.lens), G.i32(bt), ws)
    if fam.layout == "local":
        gw.decode_attn_local(*args, fam.window, None, 1, status)
    else:
        gw.decode_attn_global(*args, None, 1, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    return out


def _check(layer, widths):
    fam = layer.fam
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(layer.spec.lens)) + 1)
    pool = G.new_pool(layer)
    G.append(layer, pool, tab.cuda())
    outs = [_attend_with_table(layer, pool, _widened(layer.block_table, w)) for w in widths]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    ref = H.build_pool(layer, tab.numpy())
    got = G.to_f64(outs[0])
    cu = layer.cu_rows()
    for s in range(layer.B):
        mx, rl = G.errors(got[cu[s]:cu[s + 1]], H.oracle_rows(layer, ref, s))
        assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, mx, rl)


def test_local_many_groups_mapping_independent():
    # window 80000: 40000 keys = 313 chunks of 8 pages = 20 groups (8 warps,
    # 3 rounds); the wide table's bound is 40 groups (5 rounds).
    fam = synth.Family("local", "bf16", "local", 2, 256, 256, 1e4, 80000)
    layer = synth.Layer(synth.custom("cmbl", 71, 4, [40000, 100, 1100], [1, 1, 1], {"local": fam}), "local")
    _check(layer, [layer.block_table.shape[1], 6000])


def test_local_few_groups_mapping_independent():
    # window 8192: 500 pages = 63 chunks = 4 groups; the table's own width
    # gives 4 warps per task, the wide one 8.
    fam = synth.Family("local", "bf16", "local", 2, 256, 256, 1e4, 8192)
    layer = synth.Layer(synth.custom("cmbf", 72, 4, [8000, 3000], [1, 1], {"local": fam}), "local")
    _check(layer, [layer.block_table.shape[1], 2000])


def test_global_groups_mapping_independent():
    # 20000 tokens = 1250 pages = 40 chunks of 32 = 3 groups: 4 warps per task
    # from the table's own width, 8 from a 4096-page table.
    fam = synth.Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("cmbg", 73, 32, [20000, 700], [1, 1], {"global": fam}), "global")
    _check(layer, [layer.block_table.shape[1], 4096])
