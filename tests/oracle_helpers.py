"""Test-side glue: build oracle pools and oracle outputs for a synthetic layer."""

import numpy as np

from oracle import attention, pages, rope
from paged_hybrid_attention_gb300 import synth


def family_table(fam, max_pos):
    return rope.rope_table(fam.theta, fam.rot_dim, fam.head_dim, max_pos)


def page_bytes(fam):
    if fam.layout == "local":
        return pages.local_page_bytes(fam.kv_heads, fam.dtype)
    return pages.global_page_bytes(fam.layout)


def build_pool(layer, table, seqs=None, part="all", pool=None):
    """Oracle pool for ``layer`` holding the tokens of ``seqs`` (all by default)."""
    fam = layer.fam
    if pool is None:
        pool = pages.new_pool(layer.num_pages, page_bytes(fam))
    seqs = range(layer.B) if seqs is None else seqs
    for s in seqs:
        if layer.spec.lens[s] == 0:
            continue
        k, v, slot, pos = layer.gather([s], part=part)
        if len(pos) == 0:
            continue
        if fam.layout == "local":
            pages.write_local(pool, fam.kv_heads, fam.dtype, k, v, slot, pos, table)
        else:
            pages.write_global(pool, fam.layout, k, v, slot, pos, table)
    return pool


def q64(layer, s):
    from oracle.formats import bf16_bits_to_f64
    return bf16_bits_to_f64(layer.q(s))


def oracle_rows(layer, pool, s, scale=None):
    """float64 outputs [n_rows, HQ, D] of sequence s."""
    fam = layer.fam
    L = int(layer.spec.lens[s])
    scale = (1.0 / np.sqrt(fam.head_dim)) if scale is None else scale
    q = q64(layer, s)
    if q.shape[0] == 0:
        return q
    if fam.layout == "local":
        return attention.local_rows(pool, fam.kv_heads, fam.dtype, layer.block_table[s], L, q,
                                    fam.window, scale)
    return attention.global_rows(pool, fam.layout, layer.block_table[s], L, q, scale)


def max_pos_of(spec):
    return int(max(1, int(np.max(spec.lens)) if len(spec.lens) else 1))
