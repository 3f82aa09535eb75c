"""Batch buckets: one CUDA graph, captured for a bucket of B sequence slots,
serves any batch of at most B sequences.

"Gemma 4" (pegainfer model page), "Serving path": decode steps replay graphs
captured for power-of-two batch sizes.  Here the split plan is computed in
the kernels from the device-side row offsets and lengths, so a bucket needs
no per-size plan: the unused slots get zero query rows (no units, no output)
and their append rows write a sink page that no sequence reads.  The live
rows of every replay must equal, bit for bit, unpadded eager calls over the
live sequences alone (append + attention), the pool bytes must match
everywhere but the sink page, and the live rows must match the float64
oracle (reading pools its own page writer filled) within the attention
tolerance.
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu

BUCKET = 8
LENS = [1500, 37, 1024, 3000, 900, 2049, 17, 5000]


def _layer(key):
    sp = synth.spec("serving")
    spec = synth.custom("bucket", 1011, 32, LENS, [1] * len(LENS), sp.families)
    return synth.Layer(spec, key, layer=0 if key == "local" else 100)


class BucketStep:
    """Device buffers of one bucket (append + attention of one layer)."""

    def __init__(self, layer, pool, table):
        fam, sp = layer.fam, layer.spec
        self.layer, self.pool, self.table = layer, pool, table
        B, dev = BUCKET, "cuda"
        self.cu = torch.zeros(B + 1, dtype=torch.int32, device=dev)
        self.lens = torch.zeros(B, dtype=torch.int32, device=dev)
        self.bt = torch.full((B, layer.block_table.shape[1]), -1, dtype=torch.int32, device=dev)
        self.q = torch.zeros(B, sp.num_q_heads, fam.head_dim, dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros_like(self.q)
        shape = (B, fam.kv_heads, 256) if fam.kind == "local" else (B, 512)
        self.k = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros_like(self.k)
        self.slot = torch.zeros(B, dtype=torch.int32, device=dev)
        self.pos = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = gw.alloc_workspace(pool, sp.num_q_heads, B, layer.block_table.shape[1], 1, max(1, fam.window))
        self.sink = int(layer.unused_pages[0])

    def fill(self, live):
        """Put the live sequences in slots 0..n-1 (in this order); pad the rest."""
        layer, n = self.layer, len(live)
        sp = layer.spec
        cu = np.concatenate([np.arange(n + 1), np.full(BUCKET - n, n)]).astype(np.int32)
        lens = np.zeros(BUCKET, np.int32)
        lens[:n] = sp.lens[live]
        bt = np.full(self.bt.shape, -1, np.int32)
        bt[:n] = layer.block_table[live]
        k, v, slot, pos = layer.gather(live, "new")
        assert len(slot) == n
        slot_all = np.concatenate([slot, self.sink * 16 + np.arange(BUCKET - n)]).astype(np.int32)
        pos_all = np.concatenate([pos, np.zeros(BUCKET - n, np.int32)]).astype(np.int32)
        pad = np.zeros((BUCKET - n,) + k.shape[1:], k.dtype)
        self.cu.copy_(G.i32(cu))
        self.lens.copy_(G.i32(lens))
        self.bt.copy_(G.i32(bt))
        self.slot.copy_(G.i32(slot_all))
        self.pos.copy_(G.i32(pos_all))
        self.k.copy_(G.bits_to_cuda_bf16(np.concatenate([k, pad])))
        self.v.copy_(G.bits_to_cuda_bf16(np.concatenate([v, pad])))
        q = layer.queries(live)
        qpad = np.zeros((BUCKET - n,) + q.shape[1:], q.dtype)
        self.q.copy_(G.bits_to_cuda_bf16(np.concatenate([q, qpad])))

    def step(self):
        gw.kv_append(self.pool, self.k, self.v, self.slot, self.pos, self.table, self.status)
        if self.layer.fam.layout == "local":
            gw.decode_attn_local(self.pool, self.q, self.out, self.cu, self.lens, self.bt, self.ws,
                                 self.layer.fam.window, dev_status=self.status)
        else:
            gw.decode_attn_global(self.pool, self.q, self.out, self.cu, self.lens, self.bt, self.ws,
                                  dev_status=self.status)


def _eager(layer, snapshot, table, live):
    """Unpadded eager append + attention over the live sequences alone."""
    fam, sp = layer.fam, layer.spec
    pool = G.new_pool(layer)
    pool.data.copy_(snapshot)
    G.append(layer, pool, table, seqs=live, part="new")
    q = G.bits_to_cuda_bf16(layer.queries(live))
    out = torch.zeros_like(q)
    cu = G.i32(np.arange(len(live) + 1))
    lens, bt = G.i32(sp.lens[live]), G.i32(layer.block_table[live])
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(live), bt.shape[1], 1, max(1, fam.window))
    if fam.layout == "local":
        gw.decode_attn_local(pool, q, out, cu, lens, bt, ws, fam.window)
    else:
        gw.decode_attn_global(pool, q, out, cu, lens, bt, ws)
    torch.cuda.synchronize()
    return out, pool


@pytest.mark.parametrize("key", ["local", "global"])
def test_one_bucket_graph_serves_smaller_batches_bitwise(key):
    layer = _layer(key)
    fam, sp = layer.fam, layer.spec
    table = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sp.lens)) + 1).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, table, part="history")
    torch.cuda.synchronize()
    snapshot = pool.data.clone()
    bs = BucketStep(layer, pool, table)
    bs.fill([0, 1, 2])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        bs.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bs.step()
    ref_pool = H.build_pool(layer, table.cpu().numpy())
    pb = pool.page_bytes
    keep = torch.ones(layer.num_pages, dtype=torch.bool, device="cuda")
    keep[bs.sink] = False
    for live in ([0, 1, 2, 3, 4], [7, 3, 5, 6, 1, 0, 2], list(range(BUCKET)), [6]):
        pool.data.copy_(snapshot)
        bs.status.zero_()
        bs.fill(live)
        graph.replay()
        torch.cuda.synchronize()
        assert int(bs.status.item()) == 0, (live, int(bs.status.item()))
        want, want_pool = _eager(layer, snapshot, table, live)
        n = len(live)
        assert torch.equal(bs.out[:n].view(torch.int16), want.view(torch.int16)), live
        got_pages = pool.data.view(layer.num_pages, pb)[keep]
        want_pages = want_pool.data.view(layer.num_pages, pb)[keep]
        assert torch.equal(got_pages, want_pages), live
        got = G.to_f64(bs.out[:n])
        for i, s in enumerate(live):
            G.assert_oracle_rows(layer, got[i:i + 1], s, ref_pool)
