"""Global decode attention (tcgen05 kernel) on the GPU against the oracle.

Folded V + k_rot pool and full K + V control pool; tolerance max-abs <= 1e-2
and relative L2 <= 5e-3 against the float64 oracle.  Bitwise invariants:
batch invariance, page permutation, and folded == full for tied K/V (the same
operand values reach the tensor core in the same order).
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _run(layer, seqs_for_oracle=None, status_ok=True):
    fam = layer.fam
    max_pos = int(np.max(layer.spec.lens)) + 1
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, max_pos)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer)
    G.append(layer, pool, tab.cuda(), status=status)
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    if status_ok:
        assert int(status.item()) == 0, int(status.item())
    seqs = range(layer.B) if seqs_for_oracle is None else seqs_for_oracle
    ref_pool = H.build_pool(layer, tab.numpy(), seqs=seqs)
    return out, ref_pool, pool


def _compare(layer, out, ref_pool, seqs):
    got_all = G.to_f64(out)
    cu = layer.cu_rows()
    worst = (0.0, 0.0)
    for s in seqs:
        want = H.oracle_rows(layer, ref_pool, s)
        got = got_all[cu[s]:cu[s + 1]]
        mx, rl = G.errors(got, want)
        worst = (max(worst[0], mx), max(worst[1], rl))
        assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, mx, rl)
    return worst


@pytest.mark.parametrize("key", ["global", "global_full", "global_e4m3"])
def test_global_tiny(key):
    layer = synth.Layer(synth.spec("tiny"), key)
    out, ref, _ = _run(layer)
    _compare(layer, out, ref, range(layer.B))


@pytest.mark.parametrize("layout", ["folded", "full", "folded_e4m3"])
@pytest.mark.parametrize("hq", [8, 16, 32])
def test_global_edges(layout, hq):
    lens = [1, 15, 16, 17, 63, 64, 65, 129, 300, 1000, 4100]
    fam = synth.Family("global", "e4m3" if layout == "folded_e4m3" else "bf16", layout, 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("gedges", 40 + hq, hq, lens, [1] * len(lens), {"global": fam}), "global")
    out, ref, _ = _run(layer)
    _compare(layer, out, ref, range(layer.B))


@pytest.mark.slow
def test_global_serving_full():
    layer = synth.Layer(synth.spec("serving"), "global")
    out, ref, _ = _run(layer)
    mx, rl = _compare(layer, out, ref, range(layer.B))
    print("serving global worst max-abs %.3g rel-l2 %.3g" % (mx, rl))


@pytest.mark.slow
@pytest.mark.parametrize("key,seqs", [("global", list(range(8))), ("global_full", [2, 7]),
                                      ("global_e4m3", [0, 3, 7])])
def test_global_long_context_sampled(key, seqs):
    layer = synth.Layer(synth.spec("long_global"), key)
    out, ref, _ = _run(layer, seqs)
    mx, rl = _compare(layer, out, ref, seqs)
    print("long_global %s worst max-abs %.3g rel-l2 %.3g" % (key, mx, rl))


def test_folded_equals_full_bitwise():
    """Compressed-K attention equals attention over the materialised full K
    (tied K/V): both layouts agree with the oracle, and with each other bit
    for bit."""
    lens = [5, 77, 1000, 2049]
    outs = []
    for layout in ["folded", "full"]:
        fam = synth.Family("global", "bf16", layout, 1, 512, 128, 1e6, 0)
        layer = synth.Layer(synth.custom("ff", 99, 32, lens, [1] * 4, {"global": fam}), "global")
        out, ref_pool, _ = _run(layer)
        _compare(layer, out, ref_pool, range(layer.B))
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_global_batch_invariance_bitwise():
    sp = synth.spec("serving")
    sub = synth.custom("ginv", sp.seed, 32, sp.lens[:5], sp.n_rows[:5], sp.families)
    layer = synth.Layer(sub, "global")
    fam = layer.fam
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sub.lens)) + 1).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    full = G.attend(layer, pool)
    cu = layer.cu_rows()
    for s in [0, 2, 4]:
        q = G.bits_to_cuda_bf16(layer.q(s))
        out1 = torch.empty_like(q)
        ws = gw.alloc_workspace(pool, 32, 1, layer.block_table.shape[1], 1, 1)
        gw.decode_attn_global(pool, q, out1, G.i32([0, 1]), G.i32(sub.lens[s:s + 1]),
                              G.i32(layer.block_table[s:s + 1]), ws)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), full[cu[s]:cu[s + 1]].view(torch.int16)), s


def test_global_page_permutation_bitwise():
    fam = synth.Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("gperm", 6, 32, [300, 1200, 45], [1, 1, 1], {"global": fam}), "global")
    tab = G.oracle_table(1e6, 128, 512, 1201).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    base = G.attend(layer, pool)
    perm = np.random.Generator(np.random.PCG64(4)).permutation(layer.num_pages)
    pb = pool.page_bytes
    pool2 = G.new_pool(layer)
    pool2.data.view(layer.num_pages, pb)[torch.from_numpy(perm).cuda()] = pool.data.view(layer.num_pages, pb)
    bt = layer.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    layer.block_table = bt
    out = G.attend(layer, pool2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_global_garbage_past_end_is_ignored():
    """Bytes of a partly filled last page that no append wrote (here NaN
    patterns) must not reach the output."""
    fam = synth.Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("gnan", 7, 32, [37, 100, 1001], [1, 1, 1], {"global": fam}), "global")
    tab = G.oracle_table(1e6, 128, 512, 1002)
    pool = G.new_pool(layer, fill=0xFF)        # 0xFFFF is a bf16 NaN
    G.append(layer, pool, tab.cuda())
    out = G.attend(layer, pool)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    ref = H.build_pool(layer, tab.numpy())
    _compare(layer, out, ref, range(layer.B))


def test_global_bad_page_reported():
    fam = synth.Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("gbad", 8, 32, [500, 200], [1, 1], {"global": fam}), "global")
    tab = G.oracle_table(1e6, 128, 512, 501).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    good = G.attend(layer, pool)
    bt = layer.block_table.copy()
    bt[0, 3] = -7
    layer.block_table = bt
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gw.GW_DEV_PAGE_RANGE
    assert torch.equal(out[1].view(torch.int16), good[1].view(torch.int16))
    assert torch.isfinite(out.float()).all()


def test_e4m3_global_batch_invariance_and_permutation_bitwise():
    """On the opt-in e4m3 folded pool too, a sequence's row is bit-identical
    alone or in a batch, and permuting physical pages changes nothing."""
    fam = synth.Family("global", "e4m3", "folded_e4m3", 1, 512, 128, 1e6, 0)
    lens = [300, 1200, 45, 4100, 17]
    layer = synth.Layer(synth.custom("g8inv", 16, 32, lens, [1] * 5, {"global": fam}), "global")
    tab = G.oracle_table(1e6, 128, 512, max(lens) + 1).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    full = G.attend(layer, pool)
    for s in [0, 3, 4]:
        q = G.bits_to_cuda_bf16(layer.q(s))
        out1 = torch.empty_like(q)
        ws = gw.alloc_workspace(pool, 32, 1, layer.block_table.shape[1], 1, 1)
        gw.decode_attn_global(pool, q, out1, G.i32([0, 1]), G.i32(layer.spec.lens[s:s + 1]),
                              G.i32(layer.block_table[s:s + 1]), ws)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), full[s:s + 1].view(torch.int16)), s
    perm = np.random.Generator(np.random.PCG64(5)).permutation(layer.num_pages)
    pb = pool.page_bytes
    pool2 = G.new_pool(layer)
    pool2.data.view(layer.num_pages, pb)[torch.from_numpy(perm).cuda()] = pool.data.view(layer.num_pages, pb)
    bt = layer.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    layer.block_table = bt
    out = G.attend(layer, pool2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))


def test_e4m3_global_garbage_past_end_and_large_q():
    """Unwritten bytes of a partly filled last page (0x7F / 0xFF are e4m3
    NaNs) never reach the output, and q far outside e4m3's range (|q| up to
    3e4, and tiny heads) is carried exactly enough by the per-head
    power-of-two scaling."""
    fam = synth.Family("global", "e4m3", "folded_e4m3", 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("g8nan", 17, 16, [37, 100, 1001], [1, 1, 1], {"global": fam}), "global")
    tab = G.oracle_table(1e6, 128, 512, 1002)
    pool = G.new_pool(layer, fill=0xFF)
    G.append(layer, pool, tab.cuda())
    q = layer.queries()
    qf = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).float()
    qf[:, 0] *= 3e4 / 4          # one head far above 448
    qf[:, 1] *= 1e-5             # one head far below e4m3's normal range
    qb = qf.to(torch.bfloat16)
    out = G.attend(layer, pool, q=qb.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    ref = H.build_pool(layer, tab.numpy())
    from oracle import attention
    got = G.to_f64(out)
    for s in range(layer.B):
        q64 = qb[s:s + 1].double().numpy()
        want = attention.global_rows(ref, "folded_e4m3", layer.block_table[s], int(layer.spec.lens[s]), q64,
                                     1.0 / np.sqrt(512))
        mx, rl = G.errors(got[s:s + 1], want)
        assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, mx, rl)
