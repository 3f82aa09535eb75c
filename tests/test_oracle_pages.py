"""Pins for the oracle's pool layouts and page writer (CPU only)."""

import json
import os

import numpy as np

from oracle import formats, pages, rope

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_layout_offsets_golden():
    g = _gold("layout.json")
    for page, kvh, kind, o, d, want in g["local_kvh16"]:
        assert pages.local_offset(page, kvh, kind, o, d, 16) == want
    for page, o, e, want in g["folded"]:
        assert pages.tiled_offset(page, o, e, pages.FOLDED_ROW) == want
    for page, o, e, want in g["full"]:
        assert pages.tiled_offset(page, o, e, pages.FULL_ROW) == want
    for page, o, e, want in g["folded_e4m3"]:
        assert pages.tiled_offset(page, o, e, pages.FOLDED_ROW, 16) == want


def test_layouts_are_bijections():
    for row, blk in ((pages.FOLDED_ROW, 8), (pages.FULL_ROW, 8), (pages.FOLDED_ROW, 16)):
        o, e = np.meshgrid(np.arange(16), np.arange(row), indexing="ij")
        off = pages.tiled_offset(0, o, e, row, blk).ravel()
        assert np.array_equal(np.sort(off), np.arange(16 * row))
        # every 16-byte block row holds 16 bytes of one token, consecutive elements
        elem = 2 if blk == 8 else 1
        b = (off * elem) // 16
        assert np.all(np.bincount(b) == 16 // elem)
    p, g, k, o, d = np.meshgrid(np.arange(2), np.arange(4), np.arange(2), np.arange(16),
                                np.arange(256), indexing="ij")
    off = pages.local_offset(p, g, k, o, d, 4).ravel()
    assert np.array_equal(np.sort(off), np.arange(2 * pages.local_page_elems(4)))


def test_model_facts_byte_ratios():
    f = _gold("model_facts.json")
    assert pages.PAGE == f["page_tokens"]["value"]
    assert pages.LOCAL_D == f["local_head_dim"]["value"]
    assert pages.GLOBAL_D == f["global_head_dim"]["value"]
    assert pages.GLOBAL_ROT == f["global_rotated_dims"]["value"]
    assert pages.folded_page_bytes() / pages.full_page_bytes() == f["folded_over_full_bytes"]["value"]
    r = pages.local_page_bytes(16, "e4m3") / pages.local_page_bytes(16, "bf16")
    assert r == f["e4m3_over_bf16_local_bytes"]["value"]
    # the opt-in e4m3 folded pool: both savings at once
    assert pages.folded_e4m3_page_bytes() / pages.full_page_bytes() == \
        f["folded_over_full_bytes"]["value"] * f["e4m3_over_bf16_local_bytes"]["value"]


def test_unit_key_is_stored_as_rounded_cos_sin():
    tab = rope.rope_table(1e6, 128, 512, 300)
    pool = pages.new_pool(4, pages.folded_page_bytes())
    T = 3
    k = np.zeros((T, 512), np.uint16)
    v = np.zeros((T, 512), np.uint16)
    dims = [0, 17, 63]
    for t, i in enumerate(dims):
        k[t, i] = 0x3F80                       # 1.0
        v[t, :] = 0x4000                       # 2.0
    slot = np.array([2 * 16 + 5, 16 + 0, 3 * 16 + 15], np.int32)
    pos = np.array([0, 123, 299], np.int32)
    pages.write_global(pool, "folded", k, v, slot, pos, tab)
    table_row = np.arange(64)
    for t, i in enumerate(dims):
        bt = np.array([slot[t] // 16] * 20, np.int64)
        row = pages.read_global_rows(pool, "folded", bt, np.array([slot[t] % 16]))[0]
        assert np.all(row[:512] == 2.0)
        krot = row[512:]
        c, s = tab[pos[t], i]
        assert krot[i] == formats.bf16_bits_to_f64(formats.f32_to_bf16_bits(np.float32([c])))[0]
        assert krot[i + 64] == formats.bf16_bits_to_f64(formats.f32_to_bf16_bits(np.float32([s])))[0]
        others = np.delete(krot, [i, i + 64])
        assert np.all(others == 0.0)
    # pages never named by a slot stay untouched
    pb = pages.folded_page_bytes()
    assert not pool[0:pb].any()


def test_local_write_quantises_v_once_and_rotates_k():
    tab = rope.rope_table(1e4, 256, 256, 10)
    for dtype in ("bf16", "e4m3"):
        pool = pages.new_pool(2, pages.local_page_bytes(2, dtype), fill=0xA5)
        k = np.zeros((1, 2, 256), np.uint16)
        v = np.full((1, 2, 256), 0x3FC0, np.uint16)        # 1.5
        k[0, 1, 3] = 0x4040                                  # 3.0 on kv head 1, dim 3
        pages.write_local(pool, 2, dtype, k, v, np.array([16 + 4]), np.array([7]), tab)
        K, V = pages.read_local(pool, 2, dtype, np.array([1]), np.array([4]))
        assert np.all(V == 1.5)
        c, s = tab[7, 3]
        rq = formats.f32_to_bf16_bits if dtype == "bf16" else formats.f32_to_e4m3
        dq = formats.bf16_bits_to_f64 if dtype == "bf16" else formats.e4m3_to_f64
        assert K[0, 1, 3] == dq(rq(np.float32([np.float32(3.0) * c])))[0]
        assert K[0, 1, 3 + 128] == dq(rq(np.float32([np.float32(3.0) * s])))[0]
        assert np.count_nonzero(K[0, 0]) == 0
        # page 0 (not written) keeps its fill bytes
        assert np.all(pool[:pages.local_page_bytes(2, dtype)] == 0xA5)


def test_folded_e4m3_unit_key_is_stored_as_e4m3_cos_sin():
    """A unit key at dim i is stored, rotated, as the e4m3 roundings of the
    table's (cos, sin) at dims i and i + 64; V = 2.0 is stored exactly; every
    other element is zero; pages no slot names stay untouched."""
    tab = rope.rope_table(1e6, 128, 512, 300)
    pb = pages.folded_e4m3_page_bytes()
    pool = pages.new_pool(4, pb, fill=0xA5)
    k = np.zeros((3, 512), np.uint16)
    v = np.full((3, 512), 0x4000, np.uint16)                # 2.0
    dims = [0, 17, 63]
    for t, i in enumerate(dims):
        k[t, i] = 0x3F80                                      # 1.0
    slot = np.array([2 * 16 + 5, 16 + 0, 3 * 16 + 15], np.int32)
    pos = np.array([0, 123, 299], np.int32)
    pages.write_global(pool, "folded_e4m3", k, v, slot, pos, tab)
    for t, i in enumerate(dims):
        bt = np.array([slot[t] // 16] * 20, np.int64)
        row = pages.read_global_rows(pool, "folded_e4m3", bt, np.array([slot[t] % 16]))[0]
        assert np.all(row[:512] == 2.0)
        c, s = tab[pos[t], i]
        krot = row[512:]
        assert krot[i] == formats.e4m3_to_f64(formats.f32_to_e4m3(np.float32([c])))[0]
        assert krot[i + 64] == formats.e4m3_to_f64(formats.f32_to_e4m3(np.float32([s])))[0]
        assert np.all(np.delete(krot, [i, i + 64]) == 0.0)
        # the byte of V dim 0 of this token is at the documented offset: 0x40 is e4m3 2.0
        o = slot[t] % 16
        assert pool[(slot[t] // 16) * pb + (o // 8) * 40 * 128 + (o % 8) * 16] == 0x40
    assert np.all(pool[0:pb] == 0xA5)
