"""Multi-rank host logic of the benchmark, run as two gloo ranks on the CPU.

The benchmark scales weakly: every rank serves its own batch of sequences and
the data path has no collective.  What the ranks share is host-side: the
barrier around the timed region, the max over ranks of the time per step and
the sum over ranks of the bytes read, and rank 0 alone printing the line.
"""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks("gloo")
    assert (r.world, r.rank) == (world, rank)
    r.barrier()
    ms = 2.0 + rank                      # the slower rank sets the step time
    step_bytes = 1e9 * (1 + rank)
    res = {"max": r.max(ms), "sum": r.sum(step_bytes), "gbs": r.throughput(step_bytes, ms)}
    sp, layers = bench.workload_layers("tiny", rank)
    res["lens"] = sp.lens.tolist()
    res["bytes"] = sum(bench.kv_bytes(l) for l in layers)
    res["q0"] = layers[0].q(0)[:8].tolist()
    res["pages"] = layers[0].block_table[0].tolist()
    r.close()
    with open(os.path.join(out, "rank%d.json" % rank), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_reduce_and_shard(tmp_path):
    mp.start_processes(_rank_main, args=(2, _port(), str(tmp_path)), nprocs=2, start_method="spawn")
    r0, r1 = (json.load(open(tmp_path / ("rank%d.json" % i))) for i in range(2))
    for r in (r0, r1):
        assert r["max"] == 3.0
        assert r["sum"] == 3e9
        assert r["gbs"] == pytest.approx(3e9 / 3e-3 / 1e9)
    # weak scaling: the same per-rank shape and bytes, independent data
    assert r0["lens"] == r1["lens"] and r0["bytes"] == r1["bytes"]
    assert r0["q0"] != r1["q0"]
    for r in (r0, r1):   # the first sequence's pages: ceil(37 / 16) valid entries, then -1 padding
        pages = np.array(r["pages"])
        assert np.all(pages[:3] >= 0) and np.all(pages[3:] == -1) and len(set(pages[:3])) == 3


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
