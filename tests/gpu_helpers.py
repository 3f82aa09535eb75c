"""Test-side glue for the GPU path: build pools through gw_kv_append and run attention."""

import numpy as np
import torch

from oracle import rope
from paged_hybrid_attention_gb300 import gw


def bits_to_cuda_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def oracle_table(theta, rot_dim, head_dim, max_pos):
    """The oracle's own RoPE (cos, sin) table as a CPU float32 tensor.  Parity
    tests hand these bytes to both gw_kv_append and the oracle's page writer."""
    return torch.from_numpy(rope.rope_table(theta, rot_dim, head_dim, max_pos))


def table_for(fam, max_pos):
    return oracle_table(fam.theta, fam.rot_dim, fam.head_dim, max_pos).cuda()


def new_pool(layer, fill=0):
    fam = layer.fam
    pool = gw.KVPool(fam.layout, fam.dtype, layer.num_pages, fam.kv_heads)
    if fill:
        pool.data.fill_(fill)
    return pool


def append(layer, pool, table, seqs=None, part="all", status=None):
    k, v, slot, pos = layer.gather(seqs, part)
    if len(slot) == 0:
        return
    gw.kv_append(pool, bits_to_cuda_bf16(k), bits_to_cuda_bf16(v), i32(slot), i32(pos), table, status)


def attend(layer, pool, status=None, scale=None, q=None, out=None, stream=None):
    """Run the layer's attention for all sequences; returns the bf16 output tensor."""
    fam, sp = layer.fam, layer.spec
    if q is None:
        q = bits_to_cuda_bf16(layer.queries())
    if out is None:
        out = torch.full_like(q, float("nan"))
    cu = i32(layer.cu_rows())
    lens = i32(sp.lens)
    bt = i32(layer.block_table)
    mq = int(max(1, int(np.max(sp.n_rows)) if len(sp.n_rows) else 1))
    ws = gw.alloc_workspace(pool, sp.num_q_heads, len(sp.lens), bt.shape[1], mq, max(1, fam.window))
    if fam.layout == "local":
        gw.decode_attn_local(pool, q, out, cu, lens, bt, ws, fam.window, scale, mq, status, stream)
    else:
        gw.decode_attn_global(pool, q, out, cu, lens, bt, ws, scale, mq, status, stream)
    return out


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def errors(got, want):
    d = got - want
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / max(np.linalg.norm(want), 1e-30))


MAX_ABS, REL_L2 = 1e-2, 5e-3


def assert_oracle_rows(layer, got_rows, s, ref_pool, rows=None):
    """The GPU rows of sequence s (float64 [n, HQ, D], in row order) against
    the oracle on ref_pool, within the attention tolerance; `rows` restricts
    the check to a sample of row indices."""
    from tests import oracle_helpers as H
    want = H.oracle_rows(layer, ref_pool, s)
    if rows is not None:
        got_rows, want = got_rows[rows], want[rows]
    mx, rl = errors(got_rows, want)
    assert mx <= MAX_ABS and rl <= REL_L2, (s, mx, rl)


def check_layer_vs_oracle(layer, out, ref_pool, max_rows=8):
    """Every sequence's rows of `out` (layer.cu_rows() order) against the
    float64 oracle; prompt segments longer than max_rows are sampled at
    max_rows evenly spaced rows, first and last included."""
    got = to_f64(out)
    cu = layer.cu_rows()
    for s in range(layer.B):
        n = int(cu[s + 1] - cu[s])
        if n == 0:
            continue
        rows = None if n <= max_rows else np.unique(np.linspace(0, n - 1, max_rows).astype(int))
        assert_oracle_rows(layer, got[cu[s]:cu[s + 1]], s, ref_pool, rows)
