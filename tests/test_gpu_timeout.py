"""The kernels' bounded-wait path, made to run out on purpose, safely.

Every mbarrier wait in the library gives up after a time limit, ORs
GW_DEV_TIMEOUT into the caller's status word and lets the kernel return
instead of spinning forever.  gw_wait_selftest runs that same wait with a
1 ms limit on a phase that nothing ever completes: the kernel must end by
itself, report the timeout, and leave the context usable for the next call.
"""

import pytest
import torch

from paged_hybrid_attention_gb300 import gw, synth
from tests import gpu_helpers as G
from tests import oracle_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_bounded_wait_gives_up_and_reports(limit_ns):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    result = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    gw.wait_selftest(status, result, limit_ns)
    torch.cuda.synchronize()
    r = result.cpu().tolist()
    assert int(status.item()) == gw.GW_DEV_TIMEOUT
    assert r[0] == 1 and r[1] == 1, r
    assert limit_ns / 1000 <= r[2] < limit_ns / 1000 + 100_000, r     # gave up after the limit, not much later


def test_context_usable_after_a_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    result = torch.zeros(3, dtype=torch.int32, device="cuda")
    gw.wait_selftest(status, result, 1_000_000)
    layer = synth.Layer(synth.spec("tiny"), "local")
    fam = layer.fam
    tab = G.oracle_table(fam.theta, fam.rot_dim, fam.head_dim, int(layer.spec.lens.max()) + 1)
    pool = G.new_pool(layer)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.append(layer, pool, tab.cuda(), status=st2)
    out = G.attend(layer, pool, status=st2)
    torch.cuda.synchronize()
    assert int(status.item()) == gw.GW_DEV_TIMEOUT and int(st2.item()) == 0
    ref = H.build_pool(layer, tab.numpy())
    got = G.to_f64(out)
    for s in range(layer.B):
        mx, rl = G.errors(got[s:s + 1], H.oracle_rows(layer, ref, s))
        assert mx <= G.MAX_ABS and rl <= G.REL_L2, (s, mx, rl)
