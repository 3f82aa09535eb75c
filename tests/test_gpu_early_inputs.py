"""gw_set_early_inputs: the decode kernels read their plan inputs and first
page numbers before waiting on the previous kernel of their stream; the
results must not change.

Each case builds a pool, then captures a CUDA graph of the step as the
benchmark runs it: the append of this step's rows (which writes the pages the
decode then reads), then the attention call, launched with programmatic
dependent launch behind the append.  With early inputs on, the graph's
outputs and pool bytes must equal, bit for bit, eager calls with the
setting off; those pool bytes equal the oracle's page writer's, and those
outputs match the float64 oracle within the attention tolerance.
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _layer(kind, mixed):
    sp = synth.spec("serving")
    lens = list(sp.lens[:6]) + ([300, 700] if mixed else [])
    rows = [1] * 6 + ([300, 64] if mixed else [])
    fams = {"local": sp.families["local"], "global": sp.families["global"]}
    if kind == "e4m3":
        fams = {"local": synth.Family("local", "e4m3", "local", 16, 256, 256, 1e4, 1024, sigma=0.5)}
    elif kind == "full":
        fams = {"global": synth.Family("global", "bf16", "full", 1, 512, 128, 1e6, 0)}
    key = "global" if kind in ("global", "full") else "local"
    return synth.Layer(synth.custom("early", 1013, 32, lens, rows, fams), key, layer=0 if key == "local" else 100)


def _attend(layer, pool, q, out, cu, lens, bt, ws, mq, status):
    fam = layer.fam
    if fam.layout == "local":
        gw.decode_attn_local(pool, q, out, cu, lens, bt, ws, fam.window, max_q_rows=mq, dev_status=status)
    else:
        gw.decode_attn_global(pool, q, out, cu, lens, bt, ws, max_q_rows=mq, dev_status=status)


@pytest.mark.parametrize("kind,mixed", [("local", False), ("local", True), ("e4m3", False), ("e4m3", True),
                                        ("global", False), ("global", True), ("full", False), ("full", True)])
def test_early_inputs_same_bits(kind, mixed):
    layer = _layer(kind, mixed)
    fam, sp = layer.fam, layer.spec
    table_np = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sp.lens)) + 1)
    table = table_np.cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, table, part="history")
    torch.cuda.synchronize()
    snapshot = pool.data.clone()
    k, v, slot, pos = layer.gather(part="new")
    k, v, slot, pos = G.bits_to_cuda_bf16(k), G.bits_to_cuda_bf16(v), G.i32(slot), G.i32(pos)
    q = G.bits_to_cuda_bf16(layer.queries())
    cu, lens, bt = G.i32(layer.cu_rows()), G.i32(sp.lens), G.i32(layer.block_table)
    mq = int(np.max(sp.n_rows))
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(sp.lens), bt.shape[1], mq, max(1, fam.window))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)

    def step():
        gw.kv_append(pool, k, v, slot, pos, table, status)
        _attend(layer, pool, q, out, cu, lens, bt, ws, mq, status)

    gw.set_early_inputs(False)
    step()
    torch.cuda.synchronize()
    want, want_pool = out.clone(), pool.data.clone()
    ref_pool = H.build_pool(layer, table_np.numpy(), pool=np.zeros(pool.nbytes, np.uint8))
    assert np.array_equal(want_pool.cpu().numpy(), ref_pool)
    G.check_layer_vs_oracle(layer, want, ref_pool)
    try:
        gw.set_early_inputs(True)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
    finally:
        gw.set_early_inputs(False)
    for _ in range(3):
        pool.data.copy_(snapshot)
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0, int(status.item())
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))
        assert torch.equal(pool.data, want_pool)


def test_early_inputs_bad_length_still_reported():
    """A decode row longer than its block table is reported with early inputs
    too (the check moves after the wait) and is not read."""
    layer = _layer("local", False)
    fam, sp = layer.fam, layer.spec
    table = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sp.lens)) + 1).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, table)
    lens = sp.lens.copy()
    lens[2] = layer.block_table.shape[1] * 16 + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = G.bits_to_cuda_bf16(layer.queries())
    out = torch.zeros_like(q)
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(lens), layer.block_table.shape[1], 1, fam.window)
    try:
        gw.set_early_inputs(True)
        gw.decode_attn_local(pool, q, out, G.i32(layer.cu_rows()), G.i32(lens), G.i32(layer.block_table), ws,
                             fam.window, dev_status=status)
    finally:
        gw.set_early_inputs(False)
    torch.cuda.synchronize()
    assert int(status.item()) & 8  # GW_DEV_LEN_RANGE
    assert torch.isfinite(out.float()).all()
