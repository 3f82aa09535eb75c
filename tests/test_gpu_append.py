"""gw_kv_append on the GPU against the oracle's page writer: bit-exact pools.

Both sides receive the same logical inputs (seeded k, v, slots, positions)
and the same RoPE table bytes; the GPU pool and the oracle pool, each
pre-filled with a sentinel byte, must agree byte for byte, including pages no
slot names.
"""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A


def _pools(layer, seqs=None, part="all"):
    fam = layer.fam
    max_pos = int(np.max(layer.spec.lens)) + 1
    tab_t = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, max_pos)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer, fill=SENTINEL)
    G.append(layer, pool, tab_t.cuda(), part=part, status=status)
    ref = H.build_pool(layer, tab_t.numpy(), seqs=seqs, part=part,
                       pool=np.full(pool.nbytes, SENTINEL, np.uint8))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return pool.data.cpu().numpy(), ref


@pytest.mark.parametrize("key", ["local", "global", "global_full", "global_e4m3"])
def test_append_tiny_bit_exact(key):
    layer = synth.Layer(synth.spec("tiny"), key)
    got, ref = _pools(layer)
    assert np.array_equal(got, ref)


def test_append_tiny_e4m3_bit_exact():
    sp = synth.spec("tiny")
    fam = synth.Family("local", "e4m3", "local", 4, 256, 256, 1e4, 32, sigma=0.5)
    layer = synth.Layer(synth.custom("tiny8", sp.seed, 8, sp.lens, sp.n_rows, {"local": fam}), "local")
    got, ref = _pools(layer)
    assert np.array_equal(got, ref)


def test_append_e4m3_saturates_and_rounds_ties():
    """Large and tie values: satfinite clamps to +-448, ties go to even."""
    fam = synth.Family("local", "e4m3", "local", 1, 256, 256, 1e4, 1024)
    layer = synth.Layer(synth.custom("sat", 77, 1, [16], [1], {"local": fam}), "local", spare_pages=0)
    vals = np.array([1000.0, -1000.0, 448.0, 464.0, 1.0625, 1.1875, 2.0 ** -10, -2.0 ** -11, 0.0, -0.0] * 26,
                    np.float32)[:256]
    v = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    k = v.copy()
    kk = np.broadcast_to(k, (16, 1, 256)).copy()
    vv = np.broadcast_to(v, (16, 1, 256)).copy()
    slot = layer.slots(0, np.arange(16))
    pos = np.zeros(16, np.int32)           # position 0: rotation is the identity
    tab = G.oracle_table(1e4, 256, 256, 1)
    pool = G.new_pool(layer, fill=SENTINEL)
    gw.kv_append(pool, G.bits_to_cuda_bf16(kk), G.bits_to_cuda_bf16(vv), G.i32(slot), G.i32(pos), tab.cuda())
    from oracle import pages
    ref = np.full(pool.nbytes, SENTINEL, np.uint8)
    pages.write_local(ref, 1, "e4m3", kk, vv, slot, pos, tab.numpy())
    got = pool.data.cpu().numpy()
    assert np.array_equal(got, ref)
    assert (got == 0x7E).any() and (got == 0xFE).any()


@pytest.mark.slow
@pytest.mark.parametrize("name,key,sample", [
    ("serving", "local", None), ("serving", "global", None),
    ("fp8_local", "local", [0, 17, 40, 63]), ("fp8_local", "local_bf16", [5, 33]),
    ("long_global", "global", [3]), ("long_global", "global_full", [6]), ("long_global", "global_e4m3", [1]),
    ("mixed", "local", list(range(44, 52))), ("mixed", "global", [0, 48, 51]),
])
def test_append_full_size_bit_exact(name, key, sample):
    layer = synth.Layer(synth.spec(name), key)
    got, ref = _pools(layer, seqs=sample)
    pb = H.page_bytes(layer.fam)
    seqs = range(layer.B) if sample is None else sample
    pages_used = np.unique(np.concatenate([layer.block_table[s][layer.block_table[s] >= 0] for s in seqs]))
    for p in pages_used:
        assert np.array_equal(got[p * pb:(p + 1) * pb], ref[p * pb:(p + 1) * pb]), (name, key, int(p))
    for p in layer.unused_pages:        # never written
        assert np.all(got[p * pb:(p + 1) * pb] == SENTINEL)


def test_append_out_of_range_rows_are_skipped_and_reported():
    layer = synth.Layer(synth.spec("tiny"), "local")
    fam = layer.fam
    k, v, slot, pos = layer.gather([0])
    slot = slot.copy()
    pos = pos.copy()
    slot[3] = layer.num_pages * 16        # one past the end
    pos[5] = 100000                        # beyond the table
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, 200)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = G.new_pool(layer, fill=SENTINEL)
    gw.kv_append(pool, G.bits_to_cuda_bf16(k), G.bits_to_cuda_bf16(v), G.i32(slot), G.i32(pos), tab.cuda(), status)
    keep = np.ones(len(slot), bool)
    keep[[3, 5]] = False
    from oracle import pages
    ref = np.full(pool.nbytes, SENTINEL, np.uint8)
    pages.write_local(ref, fam.kv_heads, "bf16", k[keep], v[keep], slot[keep], pos[keep], tab.numpy())
    assert np.array_equal(pool.data.cpu().numpy(), ref)
    assert int(status.item()) == (gw.GW_DEV_SLOT_RANGE | gw.GW_DEV_POS_RANGE)


@pytest.mark.parametrize("theta,R,D", [(1e4, 256, 256), (1e6, 128, 512), (1e4, 128, 512)])
def test_rope_cs_matches_oracle_table(theta, R, D):
    """gw_rope_cs (float64 on the GPU, rounded once) against the oracle's
    table (NumPy float64 with the host libm, rounded once), over 140000
    positions.  Both round float64 values of the same definition, so they
    agree to one float32 ulp (1e-10 absolute near zero, the float64 ulp of
    angles up to 1.4e5); they are not bit-identical, because a float64 ulp of
    difference between two pow/cos implementations moves the float32 rounding
    of values near a rounding boundary.  The parity tests therefore give the
    oracle's table to both sides."""
    from oracle import rope
    mine = gw.rope_cs(theta, R, D, 140000).cpu().numpy()
    ref = rope.rope_table(theta, R, D, 140000)
    tol = np.maximum(np.spacing(np.abs(ref)).astype(np.float64), 1e-10)
    assert np.all(np.abs(mine.astype(np.float64) - ref) <= tol)
    assert np.count_nonzero(mine.view(np.uint32) != ref.view(np.uint32)) < 1e-3 * ref.size
    assert np.array_equal(mine[0, :, 0], np.ones(R // 2, np.float32))     # position 0: cos 1, sin 0
    assert np.array_equal(mine[0, :, 1], np.zeros(R // 2, np.float32))
