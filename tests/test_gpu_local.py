"""Local (sliding-window) decode attention on the GPU against the oracle.

Tolerance for the attention output (bf16) against the float64 oracle:
max-abs <= 1e-2 and relative L2 <= 5e-3.  The e4m3 leg is compared with the
oracle reading the same e4m3 pool bytes.  Invariants that must hold bit for
bit on the GPU: a sequence's output does not depend on the rest of the batch,
and permuting physical pages changes nothing.
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _run(layer, seqs_for_oracle=None):
    fam = layer.fam
    max_pos = int(np.max(layer.spec.lens)) + 1
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, max_pos)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer)
    G.append(layer, pool, tab.cuda(), status=status)
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
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


def test_local_tiny():
    layer = synth.Layer(synth.spec("tiny"), "local")
    out, ref, _ = _run(layer)
    _compare(layer, out, ref, range(layer.B))


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("kvh,hq", [(2, 2), (2, 4), (1, 4), (2, 16)])
def test_local_groups_and_edges(dtype, kvh, hq):
    # lengths around page and window edges: 1, 15, 16, 17, W-1, W, W+1, W+17, long
    W = 40
    lens = [1, 15, 16, 17, W - 1, W, W + 1, W + 17, 300]
    fam = synth.Family("local", dtype, "local", kvh, 256, 256, 1e4, W, sigma=0.5 if dtype == "e4m3" else 1.0)
    layer = synth.Layer(synth.custom("edges", 31 + kvh + hq, hq, lens, [1] * len(lens), {"local": fam}), "local")
    out, ref, _ = _run(layer)
    _compare(layer, out, ref, range(layer.B))


@pytest.mark.slow
def test_local_serving_full():
    layer = synth.Layer(synth.spec("serving"), "local")
    out, ref, _ = _run(layer)
    mx, rl = _compare(layer, out, ref, range(layer.B))
    print("serving local worst max-abs %.3g rel-l2 %.3g" % (mx, rl))


@pytest.mark.slow
def test_local_fp8_full_size_sampled():
    sp = synth.spec("fp8_local")
    sample = list(range(64))                       # every sequence
    layer = synth.Layer(sp, "local")
    out8, ref8, _ = _run(layer, sample)
    mx, rl = _compare(layer, out8, ref8, sample)
    ctl = synth.Layer(sp, "local_bf16")
    out16, ref16, _ = _run(ctl, sample)
    _compare(ctl, out16, ref16, sample)
    d = G.to_f64(out8) - G.to_f64(out16)
    print("fp8 vs oracle-on-e4m3: max-abs %.3g rel-l2 %.3g; fp8 vs bf16 run (reported, not gated): max-abs %.3g"
          % (mx, rl, float(np.max(np.abs(d)))))


def test_batch_invariance_bitwise():
    """A sequence's output is bit-identical alone or inside a batch."""
    sp = synth.spec("serving")
    sub = synth.custom("inv", sp.seed, sp.num_q_heads, sp.lens[:6], sp.n_rows[:6], sp.families)
    layer = synth.Layer(sub, "local")
    fam = layer.fam
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sub.lens)) + 1).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    full = G.attend(layer, pool)
    cu = layer.cu_rows()
    for s in [0, 3, 5]:
        alone = synth.custom("one", sp.seed, sp.num_q_heads, sub.lens[s:s + 1], [1], sp.families)
        lay1 = synth.Layer(alone, "local")
        q = G.bits_to_cuda_bf16(layer.q(s))
        out1 = torch.empty_like(q)
        ws = gw.alloc_workspace(pool, sp.num_q_heads, 1, layer.block_table.shape[1], 1, fam.window)
        gw.decode_attn_local(pool, q, out1, G.i32([0, 1]), G.i32(sub.lens[s:s + 1]),
                             G.i32(layer.block_table[s:s + 1]), ws, fam.window)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), full[cu[s]:cu[s + 1]].view(torch.int16)), s


def test_page_permutation_bitwise():
    sp = synth.spec("tiny")
    fam = synth.Family("local", "bf16", "local", 4, 256, 256, 1e4, 64)
    layer = synth.Layer(synth.custom("perm", 5, 8, [90, 200, 33], [1, 1, 1], {"local": fam}), "local")
    tab = G.oracle_table(1e4, 256, 256, 201).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    base = G.attend(layer, pool)
    perm = np.random.Generator(np.random.PCG64(3)).permutation(layer.num_pages)
    pb = pool.page_bytes
    pool2 = G.new_pool(layer)
    src = pool.data.view(layer.num_pages, pb)
    pool2.data.view(layer.num_pages, pb)[torch.from_numpy(perm).cuda()] = src
    bt = layer.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    layer.block_table = bt
    out = G.attend(layer, pool2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_bad_page_and_length_are_reported_not_read():
    fam = synth.Family("local", "bf16", "local", 2, 256, 256, 1e4, 64)
    layer = synth.Layer(synth.custom("bad", 8, 4, [100, 50, 70], [1, 1, 1], {"local": fam}), "local")
    tab = G.oracle_table(1e4, 256, 256, 101).cuda()
    pool = G.new_pool(layer)
    G.append(layer, pool, tab)
    good = G.attend(layer, pool)
    bt = layer.block_table.copy()
    bt[1, 2] = layer.num_pages + 5          # page id out of range for sequence 1
    layer.block_table = bt
    lens = layer.spec.lens.copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gw.GW_DEV_PAGE_RANGE
    # the other sequences are unaffected, bit for bit
    assert torch.equal(out[0].view(torch.int16), good[0].view(torch.int16))
    assert torch.equal(out[2].view(torch.int16), good[2].view(torch.int16))
    # a length beyond the block table is refused on the device and yields zeros
    layer.spec.lens[0] = 10 ** 6
    status.zero_()
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    layer.spec.lens[:] = lens
    assert int(status.item()) & gw.GW_DEV_LEN_RANGE
    assert torch.count_nonzero(out[0].float()) == 0


def test_zero_row_sequences_are_skipped():
    fam = synth.Family("local", "bf16", "local", 2, 256, 256, 1e4, 64)
    sp = synth.custom("zr", 12, 4, [100, 0, 70], [1, 0, 1], {"local": fam})
    layer = synth.Layer(sp, "local")
    out, ref, _ = _run(layer)
    _compare(layer, out, ref, [0, 2])


def test_local_garbage_outside_window_is_ignored():
    """Unwritten bytes of the window's first and last pages (NaN patterns
    here) must not reach the output."""
    fam = synth.Family("local", "bf16", "local", 2, 256, 256, 1e4, 40)
    layer = synth.Layer(synth.custom("lnan", 13, 4, [100, 57, 333, 16], [1, 1, 1, 1], {"local": fam}), "local")
    tab = G.oracle_table(1e4, 256, 256, 334)
    pool = G.new_pool(layer, fill=0xFF)
    G.append(layer, pool, tab.cuda())
    out = G.attend(layer, pool)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    ref = H.build_pool(layer, tab.numpy())
    _compare(layer, out, ref, range(layer.B))


def test_workspace_shared_by_consecutive_calls_bitwise():
    """One workspace serves local, global and local calls in turn."""
    sp = synth.spec("serving")
    sub = synth.custom("ws", sp.seed, sp.num_q_heads, sp.lens[:5], sp.n_rows[:5], sp.families)
    loc = synth.Layer(sub, "local")
    glo = synth.Layer(sub, "global", layer=7)
    pools = []
    for layer in (loc, glo):
        fam = layer.fam
        tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sub.lens)) + 1).cuda()
        pool = G.new_pool(layer)
        G.append(layer, pool, tab)
        pools.append(pool)
    ref_l = G.attend(loc, pools[0])
    ref_g = G.attend(glo, pools[1])
    nbytes = max(gw.workspace_bytes(pools[0], 32, 5, loc.block_table.shape[1], 1, 1024),
                 gw.workspace_bytes(pools[1], 32, 5, glo.block_table.shape[1], 1, 1))
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda").fill_(0x77)   # no zero-fill needed
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    qs = [G.bits_to_cuda_bf16(l.queries()) for l in (loc, glo)]
    for it in range(3):
        for k, (layer, pool) in enumerate(zip((loc, glo), pools)):
            out = torch.empty_like(qs[k])
            args = (pool, qs[k], out, G.i32(layer.cu_rows()), G.i32(sub.lens), G.i32(layer.block_table), ws)
            if k == 0:
                gw.decode_attn_local(*args, 1024)
            else:
                gw.decode_attn_global(*args)
            torch.cuda.synchronize()
            ref = ref_l if k == 0 else ref_g
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (it, k)


def test_e4m3_decode_q_over_a_wide_range():
    """Decode rows on an e4m3 pool take q as two e4m3 terms after an exact
    power-of-two scaling per head, so a head holding one value far beyond
    f16's range (65536, -1e6), or only values near 1e-30, still matches the
    oracle and raises no status."""
    from oracle import attention
    fam = synth.Family("local", "e4m3", "local", 2, 256, 256, 1e4, 64, sigma=0.5)
    layer = synth.Layer(synth.custom("qr", 19, 4, [100, 70], [1, 1], {"local": fam}), "local")
    tab = G.oracle_table(1e4, 256, 256, 101)
    pool = G.new_pool(layer)
    G.append(layer, pool, tab.cuda())
    ref = H.build_pool(layer, tab.numpy())
    q = torch.from_numpy(layer.queries().view(np.int16)).view(torch.bfloat16).float() * 1e-3
    for big in [65280.0, 65536.0, -1e6, None]:
        qq = q.clone()
        if big is None:
            qq[1, 2] *= 1e-27
        else:
            qq[1, 2, 5] = big
        qb = qq.to(torch.bfloat16).cuda()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = G.attend(layer, pool, status=status, q=qb)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, big
        got = G.to_f64(out)
        for s in range(layer.B):
            want = attention.local_rows(ref, 2, "e4m3", layer.block_table[s], int(layer.spec.lens[s]),
                                        qb[s:s + 1].double().cpu().numpy(), 64, 1.0 / 16)
            mx, rl = G.errors(got[s:s + 1], want)
            assert mx <= G.MAX_ABS and rl <= G.REL_L2, (big, s, mx, rl)
