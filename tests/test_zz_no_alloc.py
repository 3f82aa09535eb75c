"""The allocation-free local decode entry point, gw_decode_attn_local_noalloc.

Some callers of this library cannot allocate device memory at the moment they
run attention (an embedding runtime without a device allocator of its own, a
host that forbids device allocation once serving has started).  For them the
library offers a variant of gw_decode_attn_local that takes no workspace and
uses a fixed device array inside the library instead.

This test calls it through the C ABI twice in a row, with different queries,
and checks each output against gw_decode_attn_local on the same inputs.  Both
run the same kernels with the same length-only split plan, so the outputs
must be equal bit for bit (a stricter bar than the attention tolerance of
max-abs 1e-2 and relative L2 5e-3 used against the oracle, which the outputs
are also checked against on a sample).  It also checks that a call needing
more scratch than the array holds is refused before anything runs, and that
an invalid call gets the same status as from gw_decode_attn_local.  It lives
in a file of its own, collected last, and passes both alone and after the
rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from oracle import attention
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _noalloc_call(layer, pool, q, out):
    fam, sp = layer.fam, layer.spec
    cu = G.i32(layer.cu_rows())
    lens = G.i32(sp.lens)
    bt = G.i32(layer.block_table)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = gw.lib().gw_decode_attn_local_noalloc(
        ctypes.byref(pool.desc), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        sp.num_q_heads, len(sp.lens), ctypes.c_void_p(cu.data_ptr()), ctypes.c_void_p(lens.data_ptr()),
        ctypes.c_void_p(bt.data_ptr()), bt.shape[1], 1, fam.window, 1.0 / 16.0,
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gw.GW_OK, gw.last_error()
    return status


def test_noalloc_matches_workspace_entry_point_twice():
    layer = synth.Layer(synth.spec("serving"), "local")
    fam, sp = layer.fam, layer.spec
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(sp.lens.max()) + 1).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    gen = torch.Generator(device="cuda").manual_seed(5)
    for call in range(2):
        q = torch.randn(len(sp.lens), sp.num_q_heads, 256, generator=gen, device="cuda").to(torch.bfloat16)
        want = G.attend(layer, pool, q=q)
        got = torch.full_like(q, float("nan"))
        status = _noalloc_call(layer, pool, q, got)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), call
        if call == 0:
            ref_pool = H.build_pool(layer, tab.cpu().numpy(), seqs=[0, 7])
            for s in (0, 7):
                oq = q[s:s + 1].float().cpu().numpy().astype(np.float64)
                ref = attention.local_rows(ref_pool, fam.kv_heads, fam.dtype, layer.block_table[s],
                                           int(sp.lens[s]), oq, fam.window, 1.0 / 16.0)
                mx, rl = G.errors(G.to_f64(got[s:s + 1]), ref)
                assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, mx, rl)


def test_noalloc_refuses_oversized_calls():
    desc = gw.PoolDesc(gw.LAYOUT_LOCAL, gw.KV_BF16, 1 << 20, 100, 16, 16, 256, 256)
    fake = ctypes.c_void_p(1 << 24)
    rc = gw.lib().gw_decode_attn_local_noalloc(ctypes.byref(desc), fake, fake, 32, 4096, fake, fake, fake, 512, 1,
                                               1024, 0.0625, None, None)
    assert rc == gw.GW_ERR_WORKSPACE
    msg = gw.last_error()
    assert msg.startswith("gw_decode_attn_local_noalloc:") and str(gw.lib().gw_noalloc_scratch_bytes()) in msg


def test_noalloc_reports_the_same_errors_as_the_workspace_entry_point():
    """An invalid call is refused with the status gw_decode_attn_local gives,
    even when it would also need more scratch than the array holds."""
    desc = gw.PoolDesc(gw.LAYOUT_LOCAL, gw.KV_BF16, 1 << 20, 100, 16, 16, 256, 256)
    fake = ctypes.c_void_p(1 << 24)
    L = gw.lib()
    for batch, hq, mq, scale in [(5000, 32, 1, 0.0625), (4096, 24, 1, 0.0625), (4096, 16 * 16, 1, 0.0625),
                                 (4096, 32, 0, 0.0625), (4096, 32, 1, float("nan"))]:
        rc = L.gw_decode_attn_local_noalloc(ctypes.byref(desc), fake, fake, hq, batch, fake, fake, fake, 512, mq,
                                            1024, scale, None, None)
        ref = L.gw_decode_attn_local(ctypes.byref(desc), fake, fake, hq, batch, fake, fake, fake, 512, mq, 1024,
                                     scale, ctypes.c_void_p(1 << 28), gw.lib().gw_noalloc_scratch_bytes(), None, None)
        assert rc == ref and rc in (gw.GW_ERR_UNSUPPORTED, gw.GW_ERR_INVALID_ARG), (batch, hq, rc, ref)
        assert gw.last_error().startswith("gw_decode_attn_local")
