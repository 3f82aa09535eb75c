"""Paged KV pools: byte layouts, page writer and gather reader (oracle; test only).

[pegainfer] "Scheduling" / intro: each attention kind has its own paged pool
with 16-token pages.  [pegainfer] "Architecture notes": local layers have KVH
KV heads of dim 256; global layers have one KV head of dim 512 whose K and V
come from one projection (K via k_norm + RoPE, V via a scale-free norm).
[Gewell] "the Why": because K and V are tied and RoPE rotates only 25% of K,
a global token can be stored as V plus the rotated 128-dim slice of K, which
is 0.625x of full K+V; the unrotated 384 dims of K are rebuilt from V.
[PR1012] "Description": the local (sliding) pool may store e4m3 at scale 1.0.

A pool is a flat byte buffer of ``num_pages`` pages.  A token lives at slot
``page * 16 + offset``.  Element layouts inside one page (this library's
storage format; the pages fix the content, not the order):

LOCAL, elements of 2 B (bf16) or 1 B (e4m3):
    [kv_head g][kind: 0=K, 1=V][token o (16)][dim d (256)]
    -> KVH * 16 KiB per page (bf16), KVH * 8 KiB (e4m3).

GLOBAL FOLDED, bf16, one token row is the 640-vector  V(512) || k_rot(128):
    [token block tb (2)][column block cb (80)][row r (8)][column c (8)]
    with token o = 8*tb + r and row element e = 8*cb + c.
    -> 20480 B per page; each 8x8 block is 128 contiguous bytes.

GLOBAL FULL (control), bf16, one token row is the 1024-vector K(512) || V(512):
    [tb (2)][cb (128)][r (8)][c (8)]  -> 32768 B per page.

GLOBAL FOLDED E4M3 (an opt-in the pages do not serve), e4m3, one token row is
the folded 640-vector V(512) || k_rot(128), each element rounded once to e4m3:
    [tb (2)][cb (40)][r (8)][c (16)]  with e = 16*cb + c
    -> 10240 B per page; each 8 x 16 block is 128 contiguous bytes.

Reading any element back is the inverse map; the reader below gathers the
tokens of one sequence through its block table.
"""

import numpy as np

from .formats import (f32_to_bf16_bits, f32_to_e4m3, bf16_bits_to_e4m3,
                      bf16_bits_to_f32, bf16_bits_to_f64, e4m3_to_f64)
from .rope import rotate_half_f32

PAGE = 16
LOCAL_D = 256
GLOBAL_D = 512
GLOBAL_ROT = 128
FOLDED_ROW = GLOBAL_D + GLOBAL_ROT        # 640 elements
FULL_ROW = 2 * GLOBAL_D                   # 1024 elements

BF16, E4M3 = "bf16", "e4m3"


def elem_bytes(dtype):
    return 2 if dtype == BF16 else 1


# ---------------------------------------------------------------- page sizes
def local_page_elems(kv_heads):
    return kv_heads * 2 * PAGE * LOCAL_D


def local_page_bytes(kv_heads, dtype):
    return local_page_elems(kv_heads) * elem_bytes(dtype)


def folded_page_bytes():
    return PAGE * FOLDED_ROW * 2


def full_page_bytes():
    return PAGE * FULL_ROW * 2


def folded_e4m3_page_bytes():
    return PAGE * FOLDED_ROW


def global_page_bytes(layout):
    return {"folded": folded_page_bytes(), "full": full_page_bytes(),
            "folded_e4m3": folded_e4m3_page_bytes()}[layout]


def global_row_len(layout):
    return FULL_ROW if layout == "full" else FOLDED_ROW


# ------------------------------------------------------------ element offsets
def local_offset(page, g, kind, o, d, kv_heads):
    """Element index of (page, kv head g, K/V kind, token offset o, dim d)."""
    page = np.asarray(page, dtype=np.int64)
    return ((((page * kv_heads + g) * 2 + kind) * PAGE + o) * LOCAL_D + d)


def tiled_offset(page, o, e, row_len, blk=8):
    """Element index in a GLOBAL page whose token rows have ``row_len``
    elements, in blocks of 8 tokens x ``blk`` elements (16 bytes per block
    row: blk = 8 for bf16, 16 for e4m3)."""
    page = np.asarray(page, dtype=np.int64)
    o = np.asarray(o, dtype=np.int64)
    e = np.asarray(e, dtype=np.int64)
    tb, r = o // 8, o % 8
    cb, c = e // blk, e % blk
    nblk = row_len // blk
    return page * (PAGE * row_len) + ((tb * nblk + cb) * 8 + r) * blk + c


# --------------------------------------------------------------- pool buffers
def new_pool(num_pages, page_bytes, fill=0):
    return np.full(num_pages * page_bytes, fill, dtype=np.uint8)


def _view(pool_u8, dtype):
    return pool_u8.view(np.uint16) if dtype == BF16 else pool_u8


# -------------------------------------------------------------------- writers
def write_local(pool_u8, kv_heads, dtype, k_bits, v_bits, slot, pos, table):
    """Append T local rows.

    k_bits, v_bits: bf16 bits [T, KVH, 256]; slot, pos: int [T]; table:
    float32 [max_pos, 128, 2].  K is rotated over all 256 dims at ``pos``; V is
    stored unchanged.  Both are then rounded once to the pool type.
    """
    k32 = bf16_bits_to_f32(k_bits)
    kr = rotate_half_f32(k32, table[np.asarray(pos)][:, None, :, :])
    if dtype == BF16:
        kq, vq = f32_to_bf16_bits(kr), np.asarray(v_bits, dtype=np.uint16)
    else:
        kq, vq = f32_to_e4m3(kr), bf16_bits_to_e4m3(v_bits)
    T = kq.shape[0]
    slot = np.asarray(slot, dtype=np.int64)
    page = (slot // PAGE)[:, None, None]
    o = (slot % PAGE)[:, None, None]
    g = np.arange(kv_heads)[None, :, None]
    d = np.arange(LOCAL_D)[None, None, :]
    view = _view(pool_u8, dtype)
    view[local_offset(page, g, 0, o, d, kv_heads)] = kq
    view[local_offset(page, g, 1, o, d, kv_heads)] = vq
    return T


def folded_rows(k_bits, v_bits, pos, table):
    """Token rows V || bf16(RoPE(k[:128])) as bf16 bits [T, 640]."""
    k32 = bf16_bits_to_f32(np.asarray(k_bits)[:, :GLOBAL_ROT])
    krot = f32_to_bf16_bits(rotate_half_f32(k32, table[np.asarray(pos)]))
    return np.concatenate([np.asarray(v_bits, dtype=np.uint16), krot], axis=1)


def full_rows(k_bits, v_bits, pos, table):
    """Token rows K || V as bf16 bits [T, 1024], K = RoPE(k[:128]) || k[128:]."""
    k_bits = np.asarray(k_bits, dtype=np.uint16)
    k32 = bf16_bits_to_f32(k_bits[:, :GLOBAL_ROT])
    krot = f32_to_bf16_bits(rotate_half_f32(k32, table[np.asarray(pos)]))
    K = np.concatenate([krot, k_bits[:, GLOBAL_ROT:]], axis=1)
    return np.concatenate([K, np.asarray(v_bits, dtype=np.uint16)], axis=1)


def folded_e4m3_rows(k_bits, v_bits, pos, table):
    """Token rows V || k_rot as e4m3 codes [T, 640]: V rounded once from bf16,
    the rotated slice rounded once from its float32 rotation (as the local
    e4m3 pool rounds its rotated K)."""
    k32 = bf16_bits_to_f32(np.asarray(k_bits)[:, :GLOBAL_ROT])
    krot = f32_to_e4m3(rotate_half_f32(k32, table[np.asarray(pos)]))
    return np.concatenate([bf16_bits_to_e4m3(v_bits), krot], axis=1)


def write_global(pool_u8, layout, k_bits, v_bits, slot, pos, table):
    """Append T global rows; layout is "folded", "full" or "folded_e4m3";
    k, v bf16 bits [T, 512]."""
    make = {"folded": folded_rows, "full": full_rows, "folded_e4m3": folded_e4m3_rows}[layout]
    rows = make(k_bits, v_bits, pos, table)
    row_len = rows.shape[1]
    slot = np.asarray(slot, dtype=np.int64)
    blk = 16 if layout == "folded_e4m3" else 8
    off = tiled_offset((slot // PAGE)[:, None], (slot % PAGE)[:, None],
                       np.arange(row_len)[None, :], row_len, blk)
    if layout == "folded_e4m3":
        pool_u8[off] = rows
    else:
        pool_u8.view(np.uint16)[off] = rows
    return rows.shape[0]


# -------------------------------------------------------------------- readers
def token_slots(block_row, positions):
    """Slots of logical positions through one sequence's block-table row."""
    positions = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(block_row, dtype=np.int64)[positions // PAGE]
    if (pages < 0).any():
        raise ValueError("position maps to an unassigned page")
    return pages * PAGE + positions % PAGE


def read_local(pool_u8, kv_heads, dtype, block_row, positions):
    """K, V float64 [n, KVH, 256] of the given logical positions."""
    slot = token_slots(block_row, positions)
    page = (slot // PAGE)[:, None, None]
    o = (slot % PAGE)[:, None, None]
    g = np.arange(kv_heads)[None, :, None]
    d = np.arange(LOCAL_D)[None, None, :]
    view = _view(pool_u8, dtype)
    dec = bf16_bits_to_f64 if dtype == BF16 else e4m3_to_f64
    K = dec(view[local_offset(page, g, 0, o, d, kv_heads)])
    V = dec(view[local_offset(page, g, 1, o, d, kv_heads)])
    return K, V


def read_global_rows(pool_u8, layout, block_row, positions):
    """Stored token rows (float64) [n, 640] folded (bf16 or e4m3) or [n, 1024] full."""
    row_len = global_row_len(layout)
    slot = token_slots(block_row, positions)
    blk = 16 if layout == "folded_e4m3" else 8
    off = tiled_offset((slot // PAGE)[:, None], (slot % PAGE)[:, None],
                       np.arange(row_len)[None, :], row_len, blk)
    if layout == "folded_e4m3":
        return e4m3_to_f64(pool_u8[off])
    return bf16_bits_to_f64(pool_u8.view(np.uint16)[off])
