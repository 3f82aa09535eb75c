"""The C-ABI calls captured in a CUDA graph (as the benchmark runs them)
give the same bits as eager calls, replay after replay, for decode and
mixed (prompt-row) steps on both families; the eager results match the
float64 oracle within the attention tolerance."""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _layer(key, mixed):
    sp = synth.spec("mixed" if mixed else "serving")
    n = 8 if mixed else 6
    lens = sp.lens[:n].copy()
    rows = np.ones(n, np.int32)
    if mixed:
        lens[-2:] = [300, 700]
        rows[-2:] = [300, 64]          # a new prompt and a continuation
    return synth.Layer(synth.custom("graph", sp.seed, 32, lens, rows, sp.families), key,
                       layer=0 if key == "local" else 100)


@pytest.mark.parametrize("mixed", [False, True])
@pytest.mark.parametrize("key", ["local", "global"])
def test_graph_replay_matches_eager_bitwise(key, mixed):
    layer = _layer(key, mixed)
    fam, sp = layer.fam, layer.spec
    tab_np = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sp.lens)) + 1)
    tab = tab_np.cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    q = G.bits_to_cuda_bf16(layer.queries())
    cu, lens, bt = G.i32(layer.cu_rows()), G.i32(sp.lens), G.i32(layer.block_table)
    mq = int(np.max(sp.n_rows))
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(sp.lens), bt.shape[1], mq, max(1, fam.window))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)

    def call():
        if fam.layout == "local":
            gw.decode_attn_local(pool, q, out, cu, lens, bt, ws, fam.window, max_q_rows=mq, dev_status=status)
        else:
            gw.decode_attn_global(pool, q, out, cu, lens, bt, ws, max_q_rows=mq, dev_status=status)

    call()
    torch.cuda.synchronize()
    want = out.clone()
    G.check_layer_vs_oracle(layer, want, H.build_pool(layer, tab_np.numpy()))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))
