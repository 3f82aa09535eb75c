"""Python binding of the gw C ABI (include/gw.h) over ctypes.

Argument marshalling only: tensors are passed by ``data_ptr()`` and the
current CUDA stream; every step of the computation runs in libgw.so.  There
is no CPU path: if the library is missing this module raises ImportError.
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgw.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libgw.so is not built (%s); run `python -c 'import __graft_entry__ as g; g.build()'`"
                      % LIB_PATH)
_lib = ctypes.CDLL(LIB_PATH)

# ---- constants (mirror include/gw.h) -----------------------------------------
GW_OK, GW_ERR_INVALID_ARG, GW_ERR_UNSUPPORTED, GW_ERR_WORKSPACE, GW_ERR_CUDA = 0, 1, 2, 3, 4
GW_DEV_SLOT_RANGE, GW_DEV_POS_RANGE, GW_DEV_PAGE_RANGE, GW_DEV_LEN_RANGE = 1, 2, 4, 8
GW_DEV_TIMEOUT, GW_DEV_WORKSPACE = 16, 32
KV_BF16, KV_E4M3 = 0, 1
LAYOUT_LOCAL, LAYOUT_GLOBAL_FOLDED, LAYOUT_GLOBAL_FULL, LAYOUT_GLOBAL_FOLDED_E4M3 = 0, 1, 2, 3
LAYOUTS = {"local": LAYOUT_LOCAL, "folded": LAYOUT_GLOBAL_FOLDED, "full": LAYOUT_GLOBAL_FULL,
           "folded_e4m3": LAYOUT_GLOBAL_FOLDED_E4M3}
DTYPES = {"bf16": KV_BF16, "e4m3": KV_E4M3}
EXPORTS = ["gw_pool_page_bytes", "gw_kv_append", "gw_decode_attn_local", "gw_decode_attn_global",
           "gw_attn_workspace_bytes", "gw_last_error", "gw_version", "gw_decode_attn_local_noalloc",
           "gw_noalloc_scratch_bytes", "gw_bw_probe", "gw_set_max_ctas", "gw_set_early_launch",
           "gw_set_early_inputs", "gw_rope_cs", "gw_wait_selftest", "gw_bw_probe_tma",
           "gw_decode_attn_global_lse", "gw_merge_lse", "gw_append_decode_attn_local",
           "gw_append_decode_attn_global"]


class GwError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("gw status %d: %s" % (code, msg))
        self.code = code


class PoolDesc(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("dtype", ctypes.c_int32), ("base", ctypes.c_void_p),
                ("num_pages", ctypes.c_int64), ("page_size", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rot_dim", ctypes.c_int32)]


_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_P = ctypes.POINTER(PoolDesc)
_lib.gw_pool_page_bytes.argtypes = [_P]
_lib.gw_pool_page_bytes.restype = _sz
_lib.gw_kv_append.argtypes = [_P, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp]
_lib.gw_kv_append.restype = _i32
_lib.gw_decode_attn_local.argtypes = [_P, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _sz,
                                      _vp, _vp]
_lib.gw_decode_attn_local.restype = _i32
_lib.gw_append_decode_attn_local.argtypes = [_P, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32,
                                             _f32, _vp, _sz, _vp, _vp]
_lib.gw_append_decode_attn_local.restype = _i32
_lib.gw_append_decode_attn_global.argtypes = [_P, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32,
                                              _f32, _vp, _sz, _vp, _vp]
_lib.gw_append_decode_attn_global.restype = _i32
_lib.gw_decode_attn_global.argtypes = [_P, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _sz,
                                       _vp, _vp]
_lib.gw_decode_attn_global.restype = _i32
_lib.gw_decode_attn_global_lse.argtypes = [_P, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _f32, _vp, _sz,
                                           _vp, _vp]
_lib.gw_decode_attn_global_lse.restype = _i32
_lib.gw_merge_lse.argtypes = [_i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp]
_lib.gw_merge_lse.restype = _i32
_lib.gw_rope_cs.argtypes = [_vp, ctypes.c_double, _i32, _i32, _i32, _vp]
_lib.gw_rope_cs.restype = _i32
_lib.gw_attn_workspace_bytes.argtypes = [_P, _i32, _i32, _i32, _i32, _i32]
_lib.gw_attn_workspace_bytes.restype = _sz
_lib.gw_decode_attn_local_noalloc.argtypes = [_P, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _f32,
                                              _vp, _vp]
_lib.gw_decode_attn_local_noalloc.restype = _i32
_lib.gw_noalloc_scratch_bytes.argtypes = []
_lib.gw_noalloc_scratch_bytes.restype = _sz
_lib.gw_bw_probe.argtypes = [_vp, _sz, _vp, _vp]
_lib.gw_bw_probe.restype = _i32
_lib.gw_bw_probe_tma.argtypes = [_vp, _sz, _vp, _vp]
_lib.gw_bw_probe_tma.restype = _i32
_lib.gw_wait_selftest.argtypes = [_vp, _vp, _i64, _vp]
_lib.gw_wait_selftest.restype = _i32
_lib.gw_set_max_ctas.argtypes = [_i32]
_lib.gw_set_max_ctas.restype = _i32
_lib.gw_set_early_launch.argtypes = [_i32]
_lib.gw_set_early_launch.restype = _i32
_lib.gw_set_early_inputs.argtypes = [_i32]
_lib.gw_set_early_inputs.restype = _i32
_lib.gw_last_error.argtypes = []
_lib.gw_last_error.restype = ctypes.c_char_p
_lib.gw_version.argtypes = []
_lib.gw_version.restype = _i32


def lib():
    return _lib


def last_error():
    return _lib.gw_last_error().decode()


def version():
    return _lib.gw_version()


def _check(code):
    if code != GW_OK:
        raise GwError(code, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---- pools ---------------------------------------------------------------------
class KVPool:
    """A paged pool held in a torch uint8 device buffer plus its ABI descriptor."""

    def __init__(self, layout, dtype, num_pages, kv_heads=1, device="cuda", storage=None):
        self.layout, self.dtype = layout, dtype
        self.kv_heads = kv_heads if layout == "local" else 1
        head_dim, rot_dim = (256, 256) if layout == "local" else (512, 128)
        self.desc = PoolDesc(LAYOUTS[layout], DTYPES[dtype], None, num_pages, 16, self.kv_heads, head_dim, rot_dim)
        pb = _lib.gw_pool_page_bytes(ctypes.byref(self.desc))
        if pb == 0:
            raise GwError(GW_ERR_INVALID_ARG, last_error())
        self.page_bytes = pb
        self.num_pages = num_pages
        if storage is None:
            storage = torch.zeros(num_pages * pb + 256, dtype=torch.uint8, device=device)
        self._storage = storage
        off = (-storage.data_ptr()) % 256
        self.data = storage[off:off + num_pages * pb]
        self.desc.base = self.data.data_ptr()

    @property
    def nbytes(self):
        return self.num_pages * self.page_bytes


def rope_cs(theta, rot_dim, head_dim, max_pos, out=None, device="cuda", stream=None):
    """gw_rope_cs: the float32 [max_pos, rot_dim/2, 2] (cos, sin) table of
    gw_kv_append, computed by the library on the GPU (into `out` if given)."""
    if out is None:
        out = torch.empty((max_pos, rot_dim // 2, 2), dtype=torch.float32, device=device)
    _check(_lib.gw_rope_cs(_ptr(out), float(theta), int(rot_dim), int(head_dim), int(max_pos), _stream(stream)))
    return out


# ---- entry points ------------------------------------------------------------------
def kv_append(pool, k, v, slot, pos, rope_cs, dev_status=None, stream=None):
    """gw_kv_append: k, v bf16 CUDA tensors, slot/pos int32, rope_cs float32 [max_pos, R/2, 2]."""
    n = int(slot.numel())
    _check(_lib.gw_kv_append(ctypes.byref(pool.desc), _ptr(k), _ptr(v), n, _ptr(slot), _ptr(pos), _ptr(rope_cs),
                             int(rope_cs.shape[0]), _ptr(dev_status), _stream(stream)))


def workspace_bytes(pool, num_q_heads, batch, max_pages_per_seq, max_q_rows=1, window=1024):
    w = _lib.gw_attn_workspace_bytes(ctypes.byref(pool.desc), num_q_heads, batch, max_pages_per_seq * 16,
                                     max_q_rows, window)
    if w == 0 and batch > 0:
        raise GwError(GW_ERR_INVALID_ARG, last_error() or "invalid workspace request")
    return w


def alloc_workspace(pool, num_q_heads, batch, max_pages_per_seq, max_q_rows=1, window=1024, device="cuda"):
    n = workspace_bytes(pool, num_q_heads, batch, max_pages_per_seq, max_q_rows, window)
    buf = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def decode_attn_local(pool, q, out, cu_q_rows, seq_lens, block_table, workspace, window, scale=None,
                      max_q_rows=1, dev_status=None, stream=None):
    hq = int(q.shape[1])
    scale = 1.0 / math.sqrt(256) if scale is None else scale
    _check(_lib.gw_decode_attn_local(ctypes.byref(pool.desc), _ptr(q), _ptr(out), hq, int(seq_lens.numel()),
                                     _ptr(cu_q_rows), _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]),
                                     int(max_q_rows), int(window), float(scale), _ptr(workspace),
                                     int(workspace.numel()), _ptr(dev_status), _stream(stream)))


def append_decode_attn_local(pool, k, v, rope_cs, q, out, cu_q_rows, seq_lens, block_table, workspace, window,
                             scale=None, dev_status=None, stream=None):
    """gw_append_decode_attn_local: gw_kv_append of each decode row's k, v at
    position seq_len - 1, then its attention, in one call."""
    hq = int(q.shape[1])
    scale = 1.0 / math.sqrt(256) if scale is None else scale
    _check(_lib.gw_append_decode_attn_local(ctypes.byref(pool.desc), _ptr(k), _ptr(v), _ptr(rope_cs),
                                            int(rope_cs.shape[0]), _ptr(q), _ptr(out), hq, int(seq_lens.numel()),
                                            _ptr(cu_q_rows), _ptr(seq_lens), _ptr(block_table),
                                            int(block_table.shape[1]), int(window), float(scale), _ptr(workspace),
                                            int(workspace.numel()), _ptr(dev_status), _stream(stream)))


def append_decode_attn_global(pool, k, v, rope_cs, q, out, cu_q_rows, seq_lens, block_table, workspace, scale=None,
                              dev_status=None, stream=None):
    """gw_append_decode_attn_global: gw_kv_append of each decode row's k, v
    ([rows, 512]) at position seq_len - 1, then its attention, in one call."""
    hq = int(q.shape[1])
    scale = 1.0 / math.sqrt(512) if scale is None else scale
    _check(_lib.gw_append_decode_attn_global(ctypes.byref(pool.desc), _ptr(k), _ptr(v), _ptr(rope_cs),
                                             int(rope_cs.shape[0]), _ptr(q), _ptr(out), hq, int(seq_lens.numel()),
                                             _ptr(cu_q_rows), _ptr(seq_lens), _ptr(block_table),
                                             int(block_table.shape[1]), float(scale), _ptr(workspace),
                                             int(workspace.numel()), _ptr(dev_status), _stream(stream)))


def decode_attn_global(pool, q, out, cu_q_rows, seq_lens, block_table, workspace, scale=None, max_q_rows=1,
                       dev_status=None, stream=None):
    hq = int(q.shape[1])
    scale = 1.0 / math.sqrt(512) if scale is None else scale
    _check(_lib.gw_decode_attn_global(ctypes.byref(pool.desc), _ptr(q), _ptr(out), hq, int(seq_lens.numel()),
                                      _ptr(cu_q_rows), _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]),
                                      int(max_q_rows), float(scale), _ptr(workspace), int(workspace.numel()),
                                      _ptr(dev_status), _stream(stream)))


def decode_attn_global_lse(pool, q, out, lse, cu_q_rows, seq_lens, block_table, workspace, scale=None,
                           dev_status=None, stream=None):
    """gw_decode_attn_global_lse: decode rows, plus each row's log-sum-exp (float32 [rows, heads])."""
    hq = int(q.shape[1])
    scale = 1.0 / math.sqrt(512) if scale is None else scale
    _check(_lib.gw_decode_attn_global_lse(ctypes.byref(pool.desc), _ptr(q), _ptr(out), _ptr(lse), hq,
                                          int(seq_lens.numel()), _ptr(cu_q_rows), _ptr(seq_lens), _ptr(block_table),
                                          int(block_table.shape[1]), float(scale), _ptr(workspace),
                                          int(workspace.numel()), _ptr(dev_status), _stream(stream)))


def merge_lse(outs, lses, out, lse_out=None, stream=None):
    """gw_merge_lse: merge the parts (bf16 [rows, heads, D] outputs and their
    float32 [rows, heads] log-sum-exps) into `out`."""
    n = len(outs)
    o_arr = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    l_arr = (ctypes.c_void_p * n)(*[l.data_ptr() for l in lses])
    rows, heads, dim = (int(x) for x in out.shape)
    _check(_lib.gw_merge_lse(n, o_arr, l_arr, _ptr(out), _ptr(lse_out), rows, heads, dim, _stream(stream)))


def decode_attn_local_noalloc(pool, q, out, cu_q_rows, seq_lens, block_table, window, scale=None, max_q_rows=1,
                              dev_status=None, stream=None):
    """gw_decode_attn_local_noalloc: same as decode_attn_local, scratch from the library's static array."""
    hq = int(q.shape[1])
    scale = 1.0 / math.sqrt(256) if scale is None else scale
    _check(_lib.gw_decode_attn_local_noalloc(ctypes.byref(pool.desc), _ptr(q), _ptr(out), hq,
                                             int(seq_lens.numel()), _ptr(cu_q_rows), _ptr(seq_lens),
                                             _ptr(block_table), int(block_table.shape[1]), int(max_q_rows),
                                             int(window), float(scale), _ptr(dev_status), _stream(stream)))


def set_max_ctas(max_ctas):
    """gw_set_max_ctas: cap the CTAs (= SMs) of this thread's later attention
    calls; 0 restores one per SM."""
    _check(_lib.gw_set_max_ctas(int(max_ctas)))


def set_early_launch(on):
    """gw_set_early_launch: allow (True) or forbid programmatic early launch
    for this thread's later calls."""
    _check(_lib.gw_set_early_launch(1 if on else 0))


def set_early_inputs(on):
    """gw_set_early_inputs: let this thread's later decode calls read cu_q_rows,
    seq_lens and block_table, and its appends slot, pos and rope_cs, before
    the previous kernel of their stream ends (the caller guarantees that
    kernel does not write them)."""
    _check(_lib.gw_set_early_inputs(1 if on else 0))


def bw_probe(buf, dev_status=None, stream=None):
    """gw_bw_probe: stream `buf` (a CUDA tensor) through the decode kernels' copy pipeline."""
    _check(_lib.gw_bw_probe(_ptr(buf), int(buf.numel() * buf.element_size()), _ptr(dev_status), _stream(stream)))


def bw_probe_tma(buf, dev_status=None, stream=None):
    """gw_bw_probe_tma: stream `buf` through the bf16 decode kernel's tensor-map copy pipeline."""
    _check(_lib.gw_bw_probe_tma(_ptr(buf), int(buf.numel() * buf.element_size()), _ptr(dev_status),
                                _stream(stream)))


def wait_selftest(dev_status, result, limit_ns, stream=None):
    """gw_wait_selftest: run the kernels' bounded wait on a phase nothing
    completes, with a limit of limit_ns; result (int32[3] on the device)
    receives {first wait ok, second wait gave up, microseconds waited}."""
    _check(_lib.gw_wait_selftest(_ptr(dev_status), _ptr(result), int(limit_ns), _stream(stream)))
