"""Accuracy study for an e4m3 folded global pool (CPU, oracle only).

"feat(gemma4): the sliding family serves an opt in fp8 KV pool", "Description"
and "Verification": the pages store e4m3 at scale 1.0 for the sliding family
only and refuse it for global layers; the library refuses it too
(GW_ERR_UNSUPPORTED).  This study measures what an e4m3 global pool would
cost in accuracy, on the serving workload's global layer: attention over the
stored V || k_rot rows rounded once to e4m3 (round to nearest even,
saturating), against the same attention over the bf16 rows, both in float64.
The sliding family's e4m3 pool, which the pages do serve, is measured the
same way for comparison.  The errors are printed and bounded from the
format: e4m3 keeps 3 mantissa bits, so a stored element moves by at most
2^-4 of itself.
"""

import numpy as np

from oracle import attention, pages
from oracle.formats import bf16_bits_to_f64, e4m3_to_f64, f32_to_e4m3
from paged_hybrid_attention_gb300 import synth
from tests import oracle_helpers as H


def _e4m3(x64):
    return e4m3_to_f64(f32_to_e4m3(x64.astype(np.float32)))


def _errors(got, want):
    d = got - want
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / np.linalg.norm(want))


def test_e4m3_global_pool_error():
    sp = synth.spec("serving")
    lay = synth.Layer(sp, "global", layer=100)
    fam = lay.fam
    seqs = [0, 1, 2]
    tab = H.family_table(fam, int(np.max(sp.lens)) + 1)
    pool = H.build_pool(lay, tab, seqs=seqs)
    scale = 1.0 / np.sqrt(fam.head_dim)
    worst = (0.0, 0.0)
    for s in seqs:
        L = int(sp.lens[s])
        rows = pages.read_global_rows(pool, "folded", lay.block_table[s], np.arange(L))
        q = H.q64(lay, s)[0]
        K, V = attention.rebuild_global_k(rows)
        K8, V8 = attention.rebuild_global_k(_e4m3(rows))
        ref = attention.attend(q, K[:, None, :], V[:, None, :], scale)
        got = attention.attend(q, K8[:, None, :], V8[:, None, :], scale)
        mx, rl = _errors(got, ref)
        worst = (max(worst[0], mx), max(worst[1], rl))
    print("e4m3 global pool vs bf16: max-abs %.4g, rel-L2 %.4g" % worst)
    # each stored element moves by <= 2^-4 of itself, so no output can move by more
    assert 0.0 < worst[1] < 2.0 ** -4


def test_e4m3_local_pool_error_for_comparison():
    sp = synth.spec("serving")
    lay = synth.Layer(sp, "local", layer=0)
    fam = lay.fam
    seqs = [0, 1]
    tab = H.family_table(fam, int(np.max(sp.lens)) + 1)
    pool = H.build_pool(lay, tab, seqs=seqs)
    scale = 1.0 / np.sqrt(fam.head_dim)
    worst = (0.0, 0.0)
    for s in seqs:
        L = int(sp.lens[s])
        J = attention.local_keys(L - 1, fam.window)
        K, V = pages.read_local(pool, fam.kv_heads, "bf16", lay.block_table[s], J)
        q = H.q64(lay, s)[0]
        ref = attention.attend(q, K, V, scale)
        got = attention.attend(q, _e4m3(K), _e4m3(V), scale)
        mx, rl = _errors(got, ref)
        worst = (max(worst[0], mx), max(worst[1], rl))
    print("e4m3 local pool vs bf16: max-abs %.4g, rel-L2 %.4g" % worst)
    assert 0.0 < worst[1] < 2.0 ** -4
