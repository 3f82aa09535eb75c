"""Mixed steps on the GPU: prompt rows (n > 1 query rows per sequence, causal)
computed in the same call as decode rows, against the oracle.

Covers new prompts (L == n) and continuations over cached history (L > n),
window edges on the local family, every GQA group and q-head count, folded
and full global pools, and the invariant that decode rows of a mixed call are
bit-identical to a decode-only call with the same rows.
"""

import numpy as np
import pytest
import torch

from oracle import attention, pages
from oracle.formats import bf16_bits_to_f64
from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _build(layer):
    fam = layer.fam
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(layer.spec.lens)) + 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer, fill=0xFF)           # unwritten bytes are NaN patterns
    G.append(layer, pool, tab.cuda(), status=status)
    return pool, tab, status


def _oracle_row(layer, ref_pool, s, r, scale):
    """Oracle output of row r of sequence s (float64 [HQ, D])."""
    fam, sp = layer.fam, layer.spec
    L, n = int(sp.lens[s]), int(sp.n_rows[s])
    p = L - n + r
    q = bf16_bits_to_f64(layer.q(s))[r]
    if fam.layout == "local":
        J = attention.local_keys(p, fam.window)
        K, V = pages.read_local(ref_pool, fam.kv_heads, fam.dtype, layer.block_table[s], J)
        return attention.attend(q, K, V, scale)
    rows = pages.read_global_rows(ref_pool, fam.layout, layer.block_table[s], np.arange(p + 1))
    K, V = attention.rebuild_global_k(rows) if fam.layout == "folded" else attention.split_full_rows(rows)
    return attention.attend(q, K[:, None], V[:, None], scale)


def _check(layer, out, tab, seq_rows):
    fam = layer.fam
    scale = 1.0 / np.sqrt(fam.head_dim)
    ref = H.build_pool(layer, tab.numpy(), seqs=list(seq_rows))
    got = G.to_f64(out)
    cu = layer.cu_rows()
    worst = (0.0, 0.0)
    for s, rows in seq_rows.items():
        for r in rows:
            want = _oracle_row(layer, ref, s, r, scale)
            mx, rl = G.errors(got[cu[s] + r], want)
            worst = (max(worst[0], mx), max(worst[1], rl))
            assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, r, mx, rl)
    return worst


def _check_whole_prompt(layer, out, tab, s):
    """Every row of sequence s's prompt segment against the oracle.  The
    segment's keys are read from the oracle pool once and each row attends
    over its own key range, as attention.local_rows / global_rows define it
    (they read the pool again for every row, which is too slow for 2048
    rows)."""
    fam, sp = layer.fam, layer.spec
    L, n = int(sp.lens[s]), int(sp.n_rows[s])
    scale = 1.0 / np.sqrt(fam.head_dim)
    ref = H.build_pool(layer, tab.numpy(), seqs=[s])
    q = bf16_bits_to_f64(layer.q(s))
    got = G.to_f64(out)[layer.cu_rows()[s]:layer.cu_rows()[s] + n]
    if fam.layout == "local":
        first = max(0, L - n - fam.window + 1)
        K, V = pages.read_local(ref, fam.kv_heads, fam.dtype, layer.block_table[s], np.arange(first, L))
    else:
        rows = pages.read_global_rows(ref, fam.layout, layer.block_table[s], np.arange(L))
        K, V = attention.rebuild_global_k(rows) if fam.layout == "folded" else attention.split_full_rows(rows)
        K, V, first = K[:, None], V[:, None], 0
    worst = (0.0, 0.0)
    for r in range(n):
        p = L - n + r
        J = (attention.local_keys(p, fam.window) if fam.layout == "local" else attention.global_keys(p)) - first
        sl = slice(int(J[0]), int(J[-1]) + 1)        # J is contiguous: a view, not a copy
        assert len(J) == sl.stop - sl.start
        want = attention.attend(q[r], K[sl], V[sl], scale)
        mx, rl = G.errors(got[r], want)
        worst = (max(worst[0], mx), max(worst[1], rl))
        assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, r, mx, rl)
    return worst


def _all_rows(sp):
    return {s: list(range(int(n))) for s, n in enumerate(sp.n_rows) if n > 0}


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("kvh,hq", [(4, 4), (4, 8), (2, 8), (1, 8)])
@pytest.mark.parametrize("window", [24, 1024])
def test_local_prompt_rows(kvh, hq, window, dtype):
    """Prompt rows on bf16 and on e4m3 local pools (the e4m3 leg against the
    oracle reading the same e4m3 bytes)."""
    lens = [40, 100, 300, 70, 9, 1]
    rows = [40, 1, 64, 5, 9, 1]          # new prompt, decode, continuation, short, new, decode
    fam = synth.Family("local", dtype, "local", kvh, 256, 256, 1e4, window, sigma=0.5 if dtype == "e4m3" else 1.0)
    layer = synth.Layer(synth.custom("lp", 61 + kvh + hq, hq, lens, rows, {"local": fam}), "local")
    pool, tab, status = _build(layer)
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(out.float()).all()
    _check(layer, out, tab, _all_rows(layer.spec))


@pytest.mark.parametrize("layout", ["folded", "full"])
@pytest.mark.parametrize("hq", [8, 16, 32])
def test_global_prompt_rows(layout, hq):
    lens = [40, 100, 300, 70, 33, 1]
    rows = [40, 1, 64, 5, 33, 1]
    fam = synth.Family("global", "bf16", layout, 1, 512, 128, 1e6, 0)
    layer = synth.Layer(synth.custom("gp", 71 + hq, hq, lens, rows, {"global": fam}), "global")
    pool, tab, status = _build(layer)
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(out.float()).all()
    _check(layer, out, tab, _all_rows(layer.spec))


@pytest.mark.parametrize("key", ["local", "global", "local_e4m3"])
def test_decode_rows_of_mixed_call_equal_decode_only_bitwise(key):
    """The mixed-step-against-serial gate: decode rows computed beside prompt
    rows are bit-identical to a decode-only call, on bf16 pools and on the
    e4m3 local pool."""
    sp = synth.spec("mixed")
    fams = dict(sp.families)
    if key == "local_e4m3":
        fams["local"] = synth.Family("local", "e4m3", "local", 16, 256, 256, 1e4, 1024, sigma=0.5)
        key = "local"
    # keep it small: 6 decode streams + 2 prompts of 300 rows
    lens = np.concatenate([sp.lens[:6], [300, 500]]).astype(np.int32)
    rows = np.concatenate([np.ones(6, np.int32), [300, 100]]).astype(np.int32)
    mixed = synth.custom("mx", sp.seed, 32, lens, rows, fams)
    layer = synth.Layer(mixed, key)
    pool, tab, _ = _build(layer)
    out_mixed = G.attend(layer, pool)
    # the same decode rows, prompts dropped (zero rows)
    dec_rows = rows.copy()
    dec_rows[6:] = 0
    dec = synth.custom("mx", sp.seed, 32, lens, dec_rows, fams)
    layer_d = synth.Layer(dec, key)
    layer_d.block_table = layer.block_table          # same pool, same pages
    q = G.bits_to_cuda_bf16(np.concatenate([layer.q(s) for s in range(6)]))
    out_dec = G.attend(layer_d, pool, q=q)
    torch.cuda.synchronize()
    assert torch.equal(out_mixed[:6].view(torch.int16), out_dec.view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("key", ["local", "global", "local_e4m3"])
def test_mixed_full_size_sampled(key):
    layer = synth.Layer(synth.spec("mixed_e4m3" if key == "local_e4m3" else "mixed"),
                        "local" if key == "local_e4m3" else key)
    pool, tab, status = _build(layer)
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.Generator(np.random.PCG64(3))
    sample = {s: [0] for s in range(48)}          # every decode row
    sample[51] = sorted(rng.choice(2048, 6, replace=False).tolist() + [2047])
    mx, rl = _check(layer, out, tab, sample)
    wm, wr = _check_whole_prompt(layer, out, tab, 48)   # one whole 2048-row prompt
    print("mixed %s: decode rows + sampled worst max-abs %.3g rel-l2 %.3g; whole prompt 48 max-abs %.3g "
          "rel-l2 %.3g" % (key, mx, rl, wm, wr))


@pytest.mark.slow
@pytest.mark.parametrize("key", ["local", "global"])
def test_chunked_continuation_full_size_sampled(key):
    """Prompt chunks of 1024 rows continuing over 4k-16k cached tokens (the
    chunked walk), next to 32 decode streams, sampled against the oracle."""
    layer = synth.Layer(synth.spec("chunked"), key)
    pool, tab, status = _build(layer)
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.Generator(np.random.PCG64(4))
    sample = {s: [0] for s in range(32)}          # every decode row
    sample[35] = sorted(rng.choice(1024, 4, replace=False).tolist() + [511])
    mx, rl = _check(layer, out, tab, sample)
    _check_whole_prompt(layer, out, tab, 32)      # one whole 1024-row chunk
    print("chunked %s sampled worst max-abs %.3g rel-l2 %.3g" % (key, mx, rl))


@pytest.mark.parametrize("key", ["local", "global"])
def test_prompt_rows_with_a_bad_page_are_reported_and_stay_finite(key):
    """A page id out of range inside a prompt's key range is reported and never
    read; rows of that prompt stay finite (the kernel substitutes zeros), the
    other sequences are bit-identical to a run with a valid table."""
    sp = synth.spec("mixed")
    lens = np.concatenate([sp.lens[:3], [200, 300]]).astype(np.int32)
    rows = np.array([1, 1, 1, 200, 150], np.int32)
    layer = synth.Layer(synth.custom("badp", sp.seed, 32, lens, rows, sp.families), key,
                        layer=0 if key == "local" else 100)
    pool, tab, status = _build(layer)
    good = G.attend(layer, pool)
    bt = layer.block_table.copy()
    bt[4, 5] = layer.num_pages + 7          # inside the continuation's key range
    layer.block_table = bt
    status.zero_()
    out = G.attend(layer, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gw.GW_DEV_PAGE_RANGE
    cu = layer.cu_rows()
    assert torch.isfinite(out[cu[4]:cu[5]].float()).all()
    assert torch.equal(out[:cu[4]].view(torch.int16), good[:cu[4]].view(torch.int16))
