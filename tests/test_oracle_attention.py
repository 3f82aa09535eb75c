"""Pins for the oracle's paged attention (CPU only).

Each check compares the paged oracle with something that is not itself:
  * brute force: plain Python loops over the logical (unpaged) tokens,
  * closed forms: L = 1, equal logits, a one-hot query, a designed softmax,
  * invariants: compressed-K global == attention over a materialised full K
    (with an arbitrary k_norm gain folded into q), page-table permutation,
    sliding window == full attention over the last W tokens, split-KV then
    combine == unsplit, window >= L == full attention.
"""

import math

import numpy as np
import pytest

from oracle import attention, formats, pages, rope
from paged_hybrid_attention_gb300 import synth
from tests import oracle_helpers as H


def _tiny(fam_key):
    sp = synth.spec("tiny")
    layer = synth.Layer(sp, fam_key)
    table = H.family_table(layer.fam, H.max_pos_of(sp))
    pool = H.build_pool(layer, table)
    return sp, layer, table, pool


def _brute(q_row, Ks, Vs, scale):
    """Plain-Python softmax attention of one head over lists of key/value rows."""
    logits = [scale * sum(a * b for a, b in zip(q_row, k)) for k in Ks]
    mx = max(logits)
    w = [math.exp(x - mx) for x in logits]
    den = sum(w)
    D = len(Vs[0])
    return [sum(w[j] * Vs[j][d] for j in range(len(Vs))) / den for d in range(D)]


def test_local_matches_brute_force_tiny():
    sp, layer, table, pool = _tiny("local")
    fam = layer.fam
    G = sp.num_q_heads // fam.kv_heads
    for s in range(layer.B):
        L = int(sp.lens[s])
        pos, k, v = layer.kv(s)
        kr = formats.bf16_bits_to_f64(formats.f32_to_bf16_bits(
            rope.rotate_half_f32(formats.bf16_bits_to_f32(k), table[pos][:, None])))
        vv = formats.bf16_bits_to_f64(v)
        got = H.oracle_rows(layer, pool, s)
        q = H.q64(layer, s)
        lo = max(0, L - fam.window)
        idx = [int(np.nonzero(pos == j)[0][0]) for j in range(lo, L)]
        for h in range(sp.num_q_heads):
            g = h // G
            want = _brute(list(q[0, h]), [list(kr[i, g]) for i in idx], [list(vv[i, g]) for i in idx],
                          1.0 / 16.0)
            assert np.max(np.abs(np.array(want) - got[0, h])) < 1e-12


@pytest.mark.parametrize("fam_key", ["global", "global_full"])
def test_global_matches_brute_force_tiny(fam_key):
    sp, layer, table, pool = _tiny(fam_key)
    for s in range(layer.B):
        L = int(sp.lens[s])
        pos, k, v = layer.kv(s)
        krot = formats.f32_to_bf16_bits(rope.rotate_half_f32(
            formats.bf16_bits_to_f32(k[:, :128]), table[pos]))
        K = formats.bf16_bits_to_f64(np.concatenate([krot, k[:, 128:]], axis=1))
        V = formats.bf16_bits_to_f64(v)
        got = H.oracle_rows(layer, pool, s)
        q = H.q64(layer, s)
        for h in range(0, sp.num_q_heads, 3):
            want = _brute(list(q[0, h]), [list(K[j]) for j in range(L)], [list(V[j]) for j in range(L)],
                          1.0 / math.sqrt(512))
            assert np.max(np.abs(np.array(want) - got[0, h])) < 1e-12


def _one_seq_local(L, window, kv_heads=2, hq=4, dtype="bf16", seed=5, n_rows=1):
    fam = synth.Family("local", dtype, "local", kv_heads, 256, 256, 1e4, window)
    sp = synth.custom("t", seed, hq, [L], [n_rows], {"local": fam})
    layer = synth.Layer(sp, "local")
    table = H.family_table(fam, L + 1)
    return sp, layer, table, H.build_pool(layer, table)


def test_length_one_returns_v0():
    sp, layer, table, pool = _one_seq_local(1, 1024)
    _, k, v = layer.kv(0)
    got = H.oracle_rows(layer, pool, 0)
    G = sp.num_q_heads // layer.fam.kv_heads
    for h in range(sp.num_q_heads):
        assert np.array_equal(got[0, h], formats.bf16_bits_to_f64(v[0, h // G]))


def test_equal_logits_give_window_mean():
    sp, layer, table, pool = _one_seq_local(70, 24)
    pos, k, v = layer.kv(0)
    q = np.zeros((1, sp.num_q_heads, 256))
    out = attention.local_rows(pool, 2, "bf16", layer.block_table[0], 70, q, 24, 1 / 16)
    V = formats.bf16_bits_to_f64(v)[pos >= 70 - 24]
    for h in range(sp.num_q_heads):
        assert np.allclose(out[0, h], V[:, h // 2].mean(axis=0), atol=1e-13)


def test_one_hot_query_selects_argmax_row():
    sp, layer, table, pool = _one_seq_local(50, 1024)
    K, V = pages.read_local(pool, 2, "bf16", layer.block_table[0], np.arange(50))
    q = np.zeros((1, sp.num_q_heads, 256))
    q[0, :, 7] = 1.0
    out = attention.local_rows(pool, 2, "bf16", layer.block_table[0], 50, q, 1024, 1e4)
    for h in range(sp.num_q_heads):
        j = int(np.argmax(K[:, h // 2, 7]))
        assert np.allclose(out[0, h], V[j, h // 2], atol=1e-12)


def test_designed_softmax_closed_form():
    # keys e_j * c_j on distinct axes, values one-hot rows: o = softmax(c)
    L = 9
    c = np.linspace(-2.0, 3.0, L)
    K = np.zeros((L, 1, 16))
    V = np.zeros((L, 1, L))
    for j in range(L):
        K[j, 0, j] = c[j]
        V[j, 0, j] = 1.0
    q = np.zeros((1, 16))
    q[0, :L] = 1.0
    o = attention.attend(q, K, V, 1.0)
    want = np.exp(c) / np.exp(c).sum()
    assert np.allclose(o[0], want, atol=1e-15)


def test_window_at_least_length_is_full_attention():
    sp, layer, table, pool = _one_seq_local(60, 60)
    K, V = pages.read_local(pool, 2, "bf16", layer.block_table[0], np.arange(60))
    q = H.q64(layer, 0)
    got = H.oracle_rows(layer, pool, 0)
    full = attention.attend(q[0], K, V, 1 / 16)
    assert np.allclose(got[0], full, atol=1e-13)


def test_sliding_equals_full_attention_over_last_w():
    sp, layer, table, pool = _one_seq_local(300, 64)
    got = H.oracle_rows(layer, pool, 0)
    K, V = pages.read_local(pool, 2, "bf16", layer.block_table[0], np.arange(300 - 64, 300))
    q = H.q64(layer, 0)
    assert np.allclose(got[0], attention.attend(q[0], K, V, 1 / 16), atol=1e-13)
    # and differs from attending one more token (window inclusivity is W tokens)
    K2, V2 = pages.read_local(pool, 2, "bf16", layer.block_table[0], np.arange(300 - 65, 300))
    assert not np.allclose(got[0], attention.attend(q[0], K2, V2, 1 / 16), atol=1e-6)


def test_page_permutation_invariance():
    sp, layer, table, pool = _one_seq_local(200, 1024, seed=9)
    base = H.oracle_rows(layer, pool, 0)
    # move every page to a new physical slot and rewrite the table
    g = np.random.Generator(np.random.PCG64(2))
    perm = g.permutation(layer.num_pages)
    pb = H.page_bytes(layer.fam)
    pool2 = np.zeros_like(pool)
    for old in range(layer.num_pages):
        pool2[perm[old] * pb:(perm[old] + 1) * pb] = pool[old * pb:(old + 1) * pb]
    bt = layer.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    q = H.q64(layer, 0)
    out = attention.local_rows(pool2, 2, "bf16", bt[0], 200, q, 1024, 1 / 16)
    assert np.array_equal(out, base)


def test_split_then_combine_equals_unsplit():
    g = np.random.Generator(np.random.PCG64(4))
    K = g.normal(size=(333, 2, 64))
    V = g.normal(size=(333, 2, 64))
    q = g.normal(size=(4, 64))
    full = attention.attend(q, K, V, 0.3)
    cuts = [0, 1, 17, 100, 101, 250, 333]
    parts = [attention.partial(q, K[a:b], V[a:b], 0.3) for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.allclose(attention.combine(parts), full, atol=1e-12)


def test_compressed_global_equals_materialised_full_k_with_gain():
    """K = k_norm gain g (x) V on the unrotated dims: folding g into q is exact."""
    sp = synth.spec("tiny")
    layer = synth.Layer(sp, "global")
    table = H.family_table(layer.fam, 100)
    pool = H.build_pool(layer, table)
    g = np.random.Generator(np.random.PCG64(8)).uniform(0.5, 1.5, 512)
    for s in range(layer.B):
        L = int(sp.lens[s])
        rows = pages.read_global_rows(pool, "folded", layer.block_table[s], np.arange(L))
        Kc, V = attention.rebuild_global_k(rows)
        Kfull = Kc.copy()
        Kfull[:, 128:] *= g[128:]          # materialised full K with a gain
        q = H.q64(layer, s)[0]
        qf = q.copy()
        qf[:, 128:] *= g[128:]             # gain folded into q
        a = attention.attend(q, Kfull[:, None], V[:, None], 1 / math.sqrt(512))
        b = attention.attend(qf, Kc[:, None], V[:, None], 1 / math.sqrt(512))
        assert np.allclose(a, b, atol=1e-12)


def test_folded_and_full_pools_agree_for_tied_kv():
    sp = synth.spec("tiny")
    for s in range(2):
        outs = []
        for key in ["global", "global_full"]:
            layer = synth.Layer(sp, key)
            table = H.family_table(layer.fam, 100)
            pool = H.build_pool(layer, table)
            outs.append(H.oracle_rows(layer, pool, s))
        assert np.allclose(outs[0], outs[1], atol=1e-12)


def test_prompt_rows_are_causal_and_windowed():
    sp, layer, table, pool = _one_seq_local(80, 16, n_rows=40)
    got = H.oracle_rows(layer, pool, 0)
    q = H.q64(layer, 0)
    for r in [0, 5, 39]:
        p = 80 - 40 + r
        K, V = pages.read_local(pool, 2, "bf16", layer.block_table[0], np.arange(p - 15, p + 1))
        assert np.allclose(got[r], attention.attend(q[r], K, V, 1 / 16), atol=1e-13)


def test_e4m3_pool_reads_back_rounded_values():
    sp, layer, table, pool = _one_seq_local(40, 1024, dtype="e4m3")
    pos, k, v = layer.kv(0)
    K, V = pages.read_local(pool, 2, "e4m3", layer.block_table[0], pos)
    want_v = formats.e4m3_to_f64(formats.bf16_bits_to_e4m3(v))
    assert np.array_equal(V, want_v)
    # |stored - exact| <= half an e4m3 ulp of the value (2^-4 relative for normals)
    exact = formats.bf16_bits_to_f64(v)
    big = np.abs(exact) >= 2.0 ** -6
    assert np.all(np.abs(V - exact)[big] <= np.abs(exact)[big] * 2.0 ** -4 + 1e-30)


@pytest.mark.parametrize("fam_key,layout", [("global", "folded"), ("global_full", "full")])
def test_global_prompt_rows_match_brute_force(fam_key, layout):
    """Global prompt rows (n > 1): row r of a segment of n rows sits at
    p = L - n + r and attends causally to keys [0, p], over a K rebuilt from
    the folded row (k_rot || V[128:]) or read from the full pool.  Checked
    against plain-Python loops over the unpaged tokens, and against the
    wrong reading that lets a row see one key past its own position."""
    fam = synth.Family("global", "bf16", layout, 1, 512, 128, 1e6, 0)
    L, n = 50, 20
    sp = synth.custom("gp", 21, 4, [L], [n], {fam_key: fam})
    layer = synth.Layer(sp, fam_key)
    table = H.family_table(fam, L + 1)
    pool = H.build_pool(layer, table)
    got = H.oracle_rows(layer, pool, 0)
    pos, k, v = layer.kv(0)
    assert np.array_equal(pos, np.arange(L))
    krot = formats.f32_to_bf16_bits(rope.rotate_half_f32(formats.bf16_bits_to_f32(k[:, :128]), table[pos]))
    K = formats.bf16_bits_to_f64(np.concatenate([krot, k[:, 128:]], axis=1))
    V = formats.bf16_bits_to_f64(v)
    q = H.q64(layer, 0)
    scale = 1.0 / math.sqrt(512)
    for r in [0, 1, 9, n - 1]:
        p = L - n + r
        for h in range(sp.num_q_heads):
            want = _brute(list(q[r, h]), [list(K[j]) for j in range(p + 1)], [list(V[j]) for j in range(p + 1)],
                          scale)
            assert np.max(np.abs(np.array(want) - got[r, h])) < 1e-12, (r, h)
        if p + 1 < L:
            wrong = _brute(list(q[r, 0]), [list(K[j]) for j in range(p + 2)], [list(V[j]) for j in range(p + 2)],
                           scale)
            assert np.max(np.abs(np.array(wrong) - got[r, 0])) > 1e-6


def test_folded_e4m3_pool_attention_matches_brute_force():
    """Global decode rows over the opt-in e4m3 folded pool: plain-Python
    attention over K = e4m3(k_rot) || e4m3(V)[128:] and V = e4m3(V), built
    directly from the unpaged tokens (each element rounded once: V from its
    bf16 value, k_rot from its float32 rotation)."""
    fam = synth.Family("global", "e4m3", "folded_e4m3", 1, 512, 128, 1e6, 0, sigma=0.5)
    sp = synth.custom("g8", 23, 8, [37, 100], [1, 1], {"global": fam})
    layer = synth.Layer(sp, "global")
    table = H.family_table(fam, 101)
    pool = H.build_pool(layer, table)
    for s in range(layer.B):
        L = int(sp.lens[s])
        pos, k, v = layer.kv(s)
        kr = formats.e4m3_to_f64(formats.f32_to_e4m3(rope.rotate_half_f32(
            formats.bf16_bits_to_f32(k[:, :128]), table[pos])))
        V = formats.e4m3_to_f64(formats.bf16_bits_to_e4m3(v))
        K = np.concatenate([kr, V[:, 128:]], axis=1)
        got = H.oracle_rows(layer, pool, s)
        q = H.q64(layer, s)
        for h in range(0, sp.num_q_heads, 3):
            want = _brute(list(q[0, h]), [list(K[j]) for j in range(L)], [list(V[j]) for j in range(L)],
                          1.0 / math.sqrt(512))
            assert np.max(np.abs(np.array(want) - got[0, h])) < 1e-12
