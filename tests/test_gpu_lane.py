"""The CTA (SM) cap of a prefill lane: every call gives the same bits under
any cap as with one CTA per SM (a work unit's arithmetic never depends on
which CTA runs it), for decode rows and prompt rows on both families, and a
capped prompt lane without early launch on a second stream beside a decode
lane leaves both results unchanged.  The uncapped results themselves are
checked against the float64 oracle within the attention tolerance."""

import numpy as np
import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


def _layer(key, mixed, n=8):
    sp = synth.spec("mixed" if mixed else "serving")
    lens = sp.lens[:n].copy()
    rows = np.ones(n, np.int32)
    if mixed:
        lens[-2:] = [300, 700]
        rows[-2:] = [300, 64]          # a new prompt and a continuation
    return synth.Layer(synth.custom("lane", sp.seed, 32, lens, rows, sp.families), key,
                       layer=0 if key == "local" else 100)


def _setup(layer):
    fam, sp = layer.fam, layer.spec
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(np.max(sp.lens)) + 1)
    pool = G.new_pool(layer)
    G.append(layer, pool, tab.cuda())
    layer.ref_pool = H.build_pool(layer, tab.numpy())
    return pool


def _check_oracle(layer, out):
    G.check_layer_vs_oracle(layer, out, layer.ref_pool)


@pytest.mark.parametrize("mixed", [False, True])
@pytest.mark.parametrize("key", ["local", "global"])
def test_cap_gives_same_bits(key, mixed):
    layer = _layer(key, mixed)
    pool = _setup(layer)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = G.attend(layer, pool, status=status).clone()
    torch.cuda.synchronize()
    _check_oracle(layer, ref)
    try:
        for cap in (1, 7, 53, 99):
            gw.set_max_ctas(cap)
            got = G.attend(layer, pool, status=status)
            torch.cuda.synchronize()
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), cap
    finally:
        gw.set_max_ctas(0)
    assert int(status.item()) == 0


def test_capped_lane_beside_decode_lane():
    dec = _layer("local", False, n=16)
    pre = _layer("local", True)
    pool_d, pool_p = _setup(dec), _setup(pre)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_d = G.attend(dec, pool_d, status=status).clone()
    ref_p = G.attend(pre, pool_p, status=status).clone()
    torch.cuda.synchronize()
    _check_oracle(dec, ref_d)
    _check_oracle(pre, ref_p)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    n = torch.cuda.get_device_properties(0).multi_processor_count
    try:
        outs_d, outs_p = [], []
        for _ in range(3):
            gw.set_max_ctas(53)
            gw.set_early_launch(False)
            with torch.cuda.stream(sb):
                outs_p.append(G.attend(pre, pool_p, status=status, stream=sb).clone())
            gw.set_max_ctas(max(1, n - 53))
            gw.set_early_launch(True)
            with torch.cuda.stream(sa):
                outs_d.append(G.attend(dec, pool_d, status=status, stream=sa).clone())
        torch.cuda.synchronize()
    finally:
        gw.set_max_ctas(0)
        gw.set_early_launch(True)
    for o in outs_d:
        assert torch.equal(o.view(torch.int16), ref_d.view(torch.int16))
    for o in outs_p:
        assert torch.equal(o.view(torch.int16), ref_p.view(torch.int16))
    assert int(status.item()) == 0
