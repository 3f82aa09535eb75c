"""gw_bw_probe: the read-bandwidth probe runs to completion through the C ABI
and rejects bad arguments on the host."""

import pytest
import torch

from paged_hybrid_attention_gb300 import gw

pytestmark = pytest.mark.gpu


def test_bw_probe_runs_and_reports_no_timeout():
    buf = torch.ones(64 << 20, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gw.bw_probe(buf, status)
    gw.bw_probe(buf[:8192 * 3 + 100], status)   # a ragged tail is ignored
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_bw_probe_rejects_bad_arguments():
    buf = torch.ones(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(gw.GwError) as e:
        gw.bw_probe(buf[:4096])
    assert e.value.code == gw.GW_ERR_INVALID_ARG and "8192" in str(e.value)
    with pytest.raises(gw.GwError):
        gw.bw_probe(buf[1:9000])


def test_bw_probe_tma_runs_and_reports_no_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf = torch.zeros((1 << 24) + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    gw.bw_probe_tma(buf[off:off + (1 << 24)], status)
    gw.bw_probe_tma(buf[off:off + 16384 * 5 + 300], status)   # a ragged tail is ignored
    torch.cuda.synchronize()
    assert int(status.item()) == 0
