"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, and refuses bad arguments on the host before launching anything."""

import ctypes
import os
import re

import numpy as np
import pytest


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

gw = pytest.importorskip("paged_hybrid_attention_gb300.gw", reason="libgw.so not built")


def _declared():
    with open(os.path.join(ROOT, "include", "gw.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"^\s*(?:gw_status|size_t|const char\*|int32_t)\s+(gw_\w+)\s*\(", src, re.M)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 7
    for n in names:
        assert hasattr(gw.lib(), n), n
        assert n in gw.EXPORTS


def _desc(layout=gw.LAYOUT_LOCAL, dtype=gw.KV_BF16, page=16, kvh=16, hd=256, rd=256, base=1 << 20):
    return gw.PoolDesc(layout, dtype, base, 100, page, kvh, hd, rd)


def test_page_bytes_and_bad_descriptions():
    L = gw.lib()
    assert L.gw_pool_page_bytes(ctypes.byref(_desc())) == 16 * 16384
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(dtype=gw.KV_E4M3))) == 16 * 8192
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(gw.LAYOUT_GLOBAL_FOLDED, kvh=1, hd=512, rd=128))) == 20480
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(gw.LAYOUT_GLOBAL_FULL, kvh=1, hd=512, rd=128))) == 32768
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(page=32))) == 0
    assert "page_size" in gw.last_error()
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(base=0))) == 16 * 16384   # size query before allocation
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(gw.LAYOUT_GLOBAL_FOLDED, gw.KV_E4M3, kvh=1, hd=512, rd=128))) == 0
    assert "supports only local" in gw.last_error()
    # the opt-in e4m3 folded layout: 16 x 640 bytes, and only with dtype e4m3
    e8 = _desc(gw.LAYOUT_GLOBAL_FOLDED_E4M3, gw.KV_E4M3, kvh=1, hd=512, rd=128)
    assert L.gw_pool_page_bytes(ctypes.byref(e8)) == 10240
    assert L.gw_pool_page_bytes(ctypes.byref(_desc(gw.LAYOUT_GLOBAL_FOLDED_E4M3, kvh=1, hd=512, rd=128))) == 0
    assert "needs dtype e4m3" in gw.last_error()


def test_e4m3_global_opt_in_validation():
    L = gw.lib()
    f = _fake()
    e8 = _desc(gw.LAYOUT_GLOBAL_FOLDED_E4M3, gw.KV_E4M3, kvh=1, hd=512, rd=128)
    call = lambda mq: L.gw_decode_attn_global(ctypes.byref(e8), f, f, 32, 2, f, f, f, 64, mq, 0.04,
                                              _fake(1 << 28), 1 << 30, None, None)
    assert call(2) == gw.GW_ERR_UNSUPPORTED and "prompt rows" in gw.last_error()
    assert L.gw_attn_workspace_bytes(ctypes.byref(e8), 32, 8, 131072, 1, 0) == \
        L.gw_attn_workspace_bytes(ctypes.byref(_desc(gw.LAYOUT_GLOBAL_FOLDED, kvh=1, hd=512, rd=128)), 32, 8,
                                  131072, 1, 0)
    assert _local_call(e8) == gw.GW_ERR_INVALID_ARG               # a global pool on the local entry


def _fake(n=1 << 24):
    return ctypes.c_void_p(n)


def test_append_refuses_e4m3_global_and_bad_geometry():
    L = gw.lib()
    d = _desc(gw.LAYOUT_GLOBAL_FOLDED, gw.KV_E4M3, kvh=1, hd=512, rd=128)
    st = L.gw_kv_append(ctypes.byref(d), _fake(), _fake(), 4, _fake(), _fake(), _fake(), 10, None, None)
    assert st == gw.GW_ERR_UNSUPPORTED
    assert gw.last_error().startswith("gw_kv_append:") and "supports only local" in gw.last_error()
    d = _desc(hd=128)
    assert L.gw_kv_append(ctypes.byref(d), _fake(), _fake(), 4, _fake(), _fake(), _fake(), 10, None, None) == \
        gw.GW_ERR_INVALID_ARG
    d = _desc(base=(1 << 20) + 16)
    st = L.gw_kv_append(ctypes.byref(d), _fake(), _fake(), 4, _fake(), _fake(), _fake(), 10, None, None)
    assert st == gw.GW_ERR_INVALID_ARG and "256-byte" in gw.last_error()
    d = _desc()
    st = L.gw_kv_append(ctypes.byref(d), _fake((1 << 24) + 2), _fake(), 4, _fake(), _fake(), _fake(), 10, None, None)
    assert st == gw.GW_ERR_INVALID_ARG and "aligned" in gw.last_error()
    assert L.gw_kv_append(ctypes.byref(d), None, None, 0, None, None, None, 0, None, None) == gw.GW_OK


def _local_call(d, hq=32, batch=2, window=1024, ws_bytes=1 << 30, mq=1, scale=0.0625):
    L = gw.lib()
    f = _fake()
    return L.gw_decode_attn_local(ctypes.byref(d), f, f, hq, batch, f, f, f, 64, mq, window, scale, _fake(1 << 28),
                                  ws_bytes, None, None)


def test_attention_host_validation():
    d = _desc()
    assert _local_call(d, hq=24) == gw.GW_ERR_INVALID_ARG            # not a multiple of kv heads
    assert _local_call(d, hq=16 * 16) == gw.GW_ERR_UNSUPPORTED        # group 16
    assert _local_call(d, window=0) == gw.GW_ERR_INVALID_ARG
    assert _local_call(d, scale=float("nan")) == gw.GW_ERR_INVALID_ARG
    assert _local_call(d, ws_bytes=100) == gw.GW_ERR_WORKSPACE
    assert "workspace_bytes" in gw.last_error()
    assert _local_call(d, batch=0) == gw.GW_OK                        # empty batch: nothing to do
    assert _local_call(d, batch=4097) == gw.GW_ERR_UNSUPPORTED        # split plan lives in shared memory
    assert "4096" in gw.last_error()
    e8 = _desc(dtype=gw.KV_E4M3)
    assert _local_call(e8, mq=1) != gw.GW_ERR_UNSUPPORTED
    assert _local_call(e8, mq=2, ws_bytes=100) == gw.GW_ERR_WORKSPACE  # prompt rows on e4m3 local pools are served
    g = _desc(gw.LAYOUT_GLOBAL_FOLDED, kvh=1, hd=512, rd=128)
    assert _local_call(g) == gw.GW_ERR_INVALID_ARG                    # global pool on the local entry
    L = gw.lib()
    f = _fake()
    st = L.gw_decode_attn_global(ctypes.byref(g), f, f, 12, 2, f, f, f, 64, 1, 0.04, _fake(1 << 28), 1 << 30,
                                 None, None)
    assert st == gw.GW_ERR_UNSUPPORTED and gw.last_error().startswith("gw_decode_attn_global:")


def test_workspace_size_grows_with_batch_and_length():
    L = gw.lib()
    d = _desc()
    a = L.gw_attn_workspace_bytes(ctypes.byref(d), 32, 16, 8192, 1, 1024)
    b = L.gw_attn_workspace_bytes(ctypes.byref(d), 32, 32, 8192, 1, 1024)
    assert 0 < a < b
    g = _desc(gw.LAYOUT_GLOBAL_FOLDED, kvh=1, hd=512, rd=128)
    assert L.gw_attn_workspace_bytes(ctypes.byref(g), 32, 8, 131072, 1, 0) > \
        L.gw_attn_workspace_bytes(ctypes.byref(g), 32, 8, 8192, 1, 0)


def test_rope_cs_host_validation():
    L = gw.lib()
    f = _fake()
    assert L.gw_rope_cs(None, 1e4, 256, 256, 10, None) == gw.GW_ERR_INVALID_ARG
    assert gw.last_error().startswith("gw_rope_cs:")
    assert L.gw_rope_cs(_fake((1 << 24) + 4), 1e4, 256, 256, 10, None) == gw.GW_ERR_INVALID_ARG  # misaligned
    assert L.gw_rope_cs(f, 0.0, 256, 256, 10, None) == gw.GW_ERR_INVALID_ARG
    assert L.gw_rope_cs(f, float("inf"), 256, 256, 10, None) == gw.GW_ERR_INVALID_ARG
    assert L.gw_rope_cs(f, 1e6, 129, 512, 10, None) == gw.GW_ERR_INVALID_ARG                  # odd width
    assert L.gw_rope_cs(f, 1e6, 1024, 512, 10, None) == gw.GW_ERR_INVALID_ARG                 # wider than the head
    assert L.gw_rope_cs(f, 1e6, 128, 512, 0, None) == gw.GW_ERR_INVALID_ARG


def test_bw_probe_host_validation():
    L = gw.lib()
    assert L.gw_bw_probe(None, 1 << 20, None, None) == gw.GW_ERR_INVALID_ARG
    assert gw.last_error().startswith("gw_bw_probe:")
    assert L.gw_bw_probe(_fake((1 << 24) + 8), 1 << 20, None, None) == gw.GW_ERR_INVALID_ARG   # misaligned
    assert L.gw_bw_probe(_fake(), 4096, None, None) == gw.GW_ERR_INVALID_ARG                   # < one stage
    assert "8192" in gw.last_error()


def test_set_max_ctas_validation():
    L = gw.lib()
    assert L.gw_set_max_ctas(-1) == gw.GW_ERR_INVALID_ARG
    assert gw.last_error().startswith("gw_set_max_ctas:")
    assert L.gw_set_max_ctas(40) == gw.GW_OK
    assert L.gw_set_max_ctas(0) == gw.GW_OK
    assert L.gw_set_early_launch(0) == gw.GW_OK
    assert L.gw_set_early_launch(1) == gw.GW_OK
    assert L.gw_set_early_inputs(1) == gw.GW_OK
    assert L.gw_set_early_inputs(0) == gw.GW_OK


def test_wait_selftest_host_validation():
    L = gw.lib()
    f = _fake()
    assert L.gw_wait_selftest(None, f, 1_000_000, None) == gw.GW_ERR_INVALID_ARG
    assert gw.last_error().startswith("gw_wait_selftest:")
    assert L.gw_wait_selftest(f, None, 1_000_000, None) == gw.GW_ERR_INVALID_ARG
    assert L.gw_wait_selftest(f, f, 10, None) == gw.GW_ERR_INVALID_ARG               # below 1 us
    assert L.gw_wait_selftest(f, f, 5_000_000_000, None) == gw.GW_ERR_INVALID_ARG    # above 1 s


def test_noalloc_refusals_need_no_gpu():
    """gw_decode_attn_local_noalloc checks its arguments, scratch size
    included, before it touches the device: an oversized call is refused
    with the scratch size in the message, and an invalid one with the status
    gw_decode_attn_local gives."""
    L = gw.lib()
    d = _desc()
    f = _fake()
    rc = L.gw_decode_attn_local_noalloc(ctypes.byref(d), f, f, 32, 4096, f, f, f, 512, 1, 1024, 0.0625, None, None)
    assert rc == gw.GW_ERR_WORKSPACE
    msg = gw.last_error()
    assert msg.startswith("gw_decode_attn_local_noalloc:") and str(L.gw_noalloc_scratch_bytes()) in msg
    rc = L.gw_decode_attn_local_noalloc(ctypes.byref(d), f, f, 32, 5000, f, f, f, 512, 1, 1024, 0.0625, None, None)
    assert rc == gw.GW_ERR_UNSUPPORTED and "4096" in gw.last_error()
    assert L.gw_decode_attn_local_noalloc(ctypes.byref(d), f, f, 32, 0, f, f, f, 512, 1, 1024, 0.0625, None,
                                          None) == gw.GW_OK


def test_bw_probe_tma_host_validation():
    L = gw.lib()
    assert L.gw_bw_probe_tma(None, 1 << 20, None, None) == gw.GW_ERR_INVALID_ARG
    assert gw.last_error().startswith("gw_bw_probe_tma:")
    assert L.gw_bw_probe_tma(_fake((1 << 24) + 16), 1 << 20, None, None) == gw.GW_ERR_INVALID_ARG  # not 256-aligned
    assert L.gw_bw_probe_tma(_fake(), 8192, None, None) == gw.GW_ERR_INVALID_ARG                   # < one stage


def test_cp_entry_points_host_validation():
    L = gw.lib()
    f = _fake()
    g = _desc(gw.LAYOUT_GLOBAL_FOLDED, kvh=1, hd=512, rd=128)
    st = L.gw_decode_attn_global_lse(ctypes.byref(g), f, f, None, 32, 2, f, f, f, 64, 0.04, _fake(1 << 28), 1 << 30,
                                     None, None)
    assert st == gw.GW_ERR_INVALID_ARG and gw.last_error().startswith("gw_decode_attn_global_lse:")
    arr = (ctypes.c_void_p * 2)(1 << 24, 1 << 25)
    assert L.gw_merge_lse(0, arr, arr, f, None, 4, 8, 512, None) == gw.GW_ERR_INVALID_ARG      # no parts
    assert L.gw_merge_lse(17, arr, arr, f, None, 4, 8, 512, None) == gw.GW_ERR_INVALID_ARG     # above 16
    assert L.gw_merge_lse(2, arr, arr, f, None, 4, 8, 128, None) == gw.GW_ERR_INVALID_ARG      # head dim
    bad = (ctypes.c_void_p * 2)(1 << 24, (1 << 25) + 8)
    assert L.gw_merge_lse(2, bad, arr, f, None, 4, 8, 512, None) == gw.GW_ERR_INVALID_ARG      # misaligned part
    assert "part 1" in gw.last_error()
    assert L.gw_merge_lse(2, arr, arr, f, None, 0, 8, 512, None) == gw.GW_OK                   # no rows


def test_fused_append_entry_points_host_validation():
    """gw_append_decode_attn_local / _global refuse bad rows, RoPE tables and
    workspaces on the host, with the attention checks of their two-call
    counterparts; every refusal here comes before any launch."""
    L = gw.lib()
    f, ws = _fake(), _fake(1 << 28)
    d = _desc()

    def loc(desc=d, k=f, v=f, rope=f, max_pos=4096, hq=32, ws_bytes=1 << 30, window=1024):
        return L.gw_append_decode_attn_local(ctypes.byref(desc), k, v, rope, max_pos, f, f, hq, 2, f, f, f, 64,
                                             window, 0.0625, ws, ws_bytes, None, None)

    assert loc(k=None) == gw.GW_ERR_INVALID_ARG and "k/v" in gw.last_error()
    assert loc(v=_fake((1 << 24) + 8)) == gw.GW_ERR_INVALID_ARG              # v not 16-byte aligned
    assert loc(rope=None) == gw.GW_ERR_INVALID_ARG and "rope_cs" in gw.last_error()
    assert loc(max_pos=0) == gw.GW_ERR_INVALID_ARG and "max_pos" in gw.last_error()
    assert loc(hq=24) == gw.GW_ERR_INVALID_ARG                               # not a multiple of kv heads
    assert loc(window=0) == gw.GW_ERR_INVALID_ARG
    assert loc(ws_bytes=100) == gw.GW_ERR_WORKSPACE
    assert gw.last_error().startswith("gw_append_decode_attn_local:")
    assert loc(desc=_desc(dtype=gw.KV_E4M3), ws_bytes=100) == gw.GW_ERR_WORKSPACE   # e4m3 pools are served
    g = _desc(gw.LAYOUT_GLOBAL_FOLDED, kvh=1, hd=512, rd=128)
    assert loc(desc=g) == gw.GW_ERR_INVALID_ARG                              # global pool on the local entry

    def glo(desc=g, k=f, rope=f, max_pos=4096, hq=32, ws_bytes=1 << 30):
        return L.gw_append_decode_attn_global(ctypes.byref(desc), k, f, rope, max_pos, f, f, hq, 2, f, f, f, 64,
                                              0.04, ws, ws_bytes, None, None)

    assert glo(k=None) == gw.GW_ERR_INVALID_ARG
    assert glo(rope=_fake((1 << 24) + 4)) == gw.GW_ERR_INVALID_ARG           # rope_cs not 16-byte aligned
    assert glo(hq=12) == gw.GW_ERR_UNSUPPORTED
    assert glo(ws_bytes=100) == gw.GW_ERR_WORKSPACE
    assert gw.last_error().startswith("gw_append_decode_attn_global:")
    e8 = _desc(gw.LAYOUT_GLOBAL_FOLDED_E4M3, gw.KV_E4M3, kvh=1, hd=512, rd=128)
    assert glo(desc=e8, ws_bytes=100) == gw.GW_ERR_WORKSPACE                  # all three global layouts
    assert glo(desc=d) == gw.GW_ERR_INVALID_ARG                              # local pool on the global entry
