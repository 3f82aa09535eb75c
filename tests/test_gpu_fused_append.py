"""gw_append_decode_attn_*: a decode step's append and attention in one call.

The fused call must leave the pool holding exactly the bytes that
gw_kv_append writes for the step's rows (slot and pos derived from the
sequence's length and block table) and produce exactly the output of
gw_decode_attn_* over that pool, bit for bit; both are also checked against
the float64 oracle.
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _fused(layer, pool, tab, status, early=False):
    """The step's rows appended and attended in one fused call; returns out."""
    fam, sp = layer.fam, layer.spec
    k, v, _, _ = layer.gather(part="new")
    q = G.bits_to_cuda_bf16(layer.queries())
    out = torch.full_like(q, float("nan"))
    cu, lens, bt = G.i32(layer.cu_rows()), G.i32(sp.lens), G.i32(layer.block_table)
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(sp.lens), bt.shape[1], 1, max(1, fam.window))
    gw.set_early_inputs(early)
    try:
        if fam.layout == "local":
            gw.append_decode_attn_local(pool, G.bits_to_cuda_bf16(k), G.bits_to_cuda_bf16(v), tab, q, out, cu, lens,
                                        bt, ws, fam.window, dev_status=status)
        else:
            gw.append_decode_attn_global(pool, G.bits_to_cuda_bf16(k), G.bits_to_cuda_bf16(v), tab, q, out, cu, lens,
                                         bt, ws, dev_status=status)
    finally:
        gw.set_early_inputs(False)
    return out


def _check(layer, early=False, oracle=True):
    fam = layer.fam
    max_pos = int(np.max(layer.spec.lens)) + 1
    tab_cpu = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, max_pos)
    tab = tab_cpu.cuda()
    # two calls: every row appended, then attention
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_pool = G.new_pool(layer, fill=0x3C)
    G.append(layer, ref_pool, tab, status=st_ref)
    ref_out = G.attend(layer, ref_pool, status=st_ref)
    # fused: history appended, then the step's rows inside the decode call
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer, fill=0x3C)
    G.append(layer, pool, tab, part="history", status=st)
    out = _fused(layer, pool, tab, st, early)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st_ref.item()) == 0
    assert torch.equal(pool.data, ref_pool.data)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    if oracle:
        G.check_layer_vs_oracle(layer, out, H.build_pool(layer, tab_cpu.numpy()))
    return pool


def test_fused_local_tiny():
    _check(synth.Layer(synth.spec("tiny"), "local"))


@pytest.mark.parametrize("early", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("kvh,hq", [(2, 2), (2, 4), (1, 4), (2, 16)])
def test_fused_local_groups_and_edges(kvh, hq, dtype, early):
    # lengths around page, chunk and window edges (first token, page ends,
    # one past a page, the window, a long tail); e4m3 draws N(0, 0.5) like the
    # fp8 workload
    W = 40
    lens = [1, 2, 15, 16, 17, 32, 33, W - 1, W, W + 1, W + 17, 128, 129, 300]
    fam = synth.Family("local", dtype, "local", kvh, 256, 256, 1e4, W, sigma=0.5 if dtype == "e4m3" else 1.0)
    layer = synth.Layer(synth.custom("fused", 41 + kvh + hq, hq, lens, [1] * len(lens), {"local": fam}), "local")
    _check(layer, early)


def test_fused_local_window_1024_many_sequences():
    # the served window over lengths that span 1..9 chunks per KV head, with
    # sequences that carry no row this step in between
    g = np.random.Generator(np.random.PCG64(77))
    lens = g.integers(1, 3000, size=40).astype(np.int32)
    rows = np.ones(40, np.int32)
    rows[::7] = 0
    fam = synth.Family("local", "bf16", "local", 4, 256, 256, 1e4, 1024)
    layer = synth.Layer(synth.custom("fused_w", 78, 8, lens, rows, {"local": fam}), "local")
    _check(layer, early=True)


@pytest.mark.slow
def test_fused_local_serving_full():
    _check(synth.Layer(synth.spec("serving"), "local"), early=True)


@pytest.mark.slow
def test_fused_local_fp8_full():
    # all 64 sequences of the fp8 workload, every output row against the oracle
    _check(synth.Layer(synth.spec("fp8_local"), "local"), early=True)


def test_fused_local_position_beyond_table_is_reported_not_written():
    fam = synth.Family("local", "bf16", "local", 2, 256, 256, 1e4, 64)
    layer = synth.Layer(synth.custom("fused_pos", 51, 4, [20, 90], [1, 1], {"local": fam}), "local")
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, 50).cuda()   # positions 0..49 only
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer, fill=0x3C)
    G.append(layer, pool, tab, seqs=[0], part="history", status=st)
    # sequence 1's history lies beyond the table too: write it with a larger one
    big = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, 100).cuda()
    G.append(layer, pool, big, seqs=[1], part="history", status=st)
    before = pool.data.clone()
    _fused(layer, pool, tab, st)
    torch.cuda.synchronize()
    assert int(st.item()) & gw.GW_DEV_POS_RANGE
    # sequence 0's row was written, sequence 1's (position 89) was not
    ref_pool = G.new_pool(layer)
    ref_pool.data.copy_(before)
    G.append(layer, ref_pool, tab, seqs=[0], part="new")
    assert torch.equal(pool.data, ref_pool.data)


@pytest.mark.parametrize("key", ["global", "global_full", "global_e4m3"])
def test_fused_global_tiny(key):
    _check(synth.Layer(synth.spec("tiny"), key))


@pytest.mark.parametrize("early", [False, True])
@pytest.mark.parametrize("layout,dtype", [("folded", "bf16"), ("full", "bf16"), ("folded_e4m3", "e4m3")])
@pytest.mark.parametrize("hq", [8, 32])
def test_fused_global_edges(layout, dtype, hq, early):
    # lengths around page, tile (4 pages) and chunk (32 pages) edges.  The
    # e4m3 pool draws N(0, 0.5) like the fp8 workload: at sigma 1 a two-token
    # softmax reaches max-abs 0.0102 against the oracle (outputs near 3, whose
    # bf16 rounding alone is up to 0.0078, and P carried as two e4m3 terms),
    # in the fused and the two-call path alike.
    lens = [1, 2, 16, 17, 63, 64, 65, 511, 512, 513, 1100]
    fam = synth.Family("global", dtype, layout, 1, 512, 128, 1e6, 0, sigma=0.5 if dtype == "e4m3" else 1.0)
    layer = synth.Layer(synth.custom("fused_g", 90 + hq, hq, lens, [1] * len(lens), {"global": fam}), "global")
    _check(layer, early)


@pytest.mark.slow
def test_fused_global_serving_full():
    _check(synth.Layer(synth.spec("serving"), "global"), early=True)
