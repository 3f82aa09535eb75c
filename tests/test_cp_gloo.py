"""Context-parallel split of one long global sequence, as two gloo ranks on
the CPU: the host logic of paged_hybrid_attention_gb300.cp.

Each rank takes its contiguous share of the pages of a 131072-token
sequence (cp.shard_pages), computes with the oracle its rows' attention over
those keys and their log-sum-exp, and the ranks swap them through
cp.exchange (an all-gather over gloo).  Merged by the log-sum-exp rule in
rank order, the parts must equal the oracle's attention over the whole
sequence (to 1e-12).  The merge on the GPU (gw_merge_lse) is tested in
test_gpu_cp.py.
"""

import json
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from oracle import attention, pages
    from paged_hybrid_attention_gb300 import cp, synth
    from tests import oracle_helpers as H
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sp = synth.spec("long_global")
    one = synth.custom("cp", sp.seed, 8, sp.lens[:1], sp.n_rows[:1], sp.families, 0, 1)
    layer = synth.Layer(one, "global", layer=100)
    L = int(one.lens[0])
    table = H.family_table(layer.fam, L + 1)
    p0, p1, k0, k1 = cp.shard_pages(L, world, rank)
    # this rank's pool: its pages only, renumbered from 0
    pos, k, v = layer.kv(0)
    mine = (pos >= k0) & (pos < k1)
    slot = ((pos[mine] // 16 - p0) * 16 + pos[mine] % 16).astype(np.int32)
    pool = pages.new_pool(p1 - p0, pages.folded_page_bytes())
    pages.write_global(pool, "folded", k[mine], v[mine], slot, pos[mine], table)
    rows = pages.read_global_rows(pool, "folded", np.arange(p1 - p0), np.arange(k1 - k0))
    K, V = attention.rebuild_global_k(rows)
    q = H.q64(layer, 0)[0]
    m, l, o = attention.partial(q, K[:, None], V[:, None], 1.0 / np.sqrt(512))
    outs, lses = cp.exchange(torch.from_numpy(o / l[:, None]), torch.from_numpy(m + np.log(l)))
    res = {"range": [p0, p1, k0, k1]}
    if rank == 0:
        merged = attention.combine([(ls.numpy(), np.ones_like(ls.numpy()), ot.numpy()) for ot, ls in zip(outs, lses)])
        full_pool = H.build_pool(layer, table)
        want = H.oracle_rows(layer, full_pool, 0)[0]
        res["err"] = float(np.max(np.abs(merged - want)))
    dist.destroy_process_group()
    with open(os.path.join(out, "rank%d.json" % rank), "w") as f:
        json.dump(res, f)


def test_shard_pages_cover_the_sequence_once():
    sys.path.insert(0, ROOT)
    from paged_hybrid_attention_gb300 import cp
    for L in [1, 15, 16, 17, 1000, 131072, 131073]:
        for world in [1, 2, 3, 8, 16]:
            ranges = [cp.shard_pages(L, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == (L + 15) // 16
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))          # contiguous, disjoint
            assert ranges[0][2] == 0 and ranges[-1][3] == L
            assert all(a[3] == b[2] for a, b in zip(ranges, ranges[1:]))
            sizes = [p1 - p0 for p0, p1, _, _ in ranges]
            assert max(sizes) - min(sizes) <= 1                                    # balanced


def test_two_gloo_ranks_split_a_131072_token_sequence(tmp_path):
    mp.start_processes(_rank_main, args=(2, _port(), str(tmp_path)), nprocs=2, start_method="spawn")
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["range"] == [0, 4096, 0, 65536] and r1["range"] == [4096, 8192, 65536, 131072]
    assert r0["err"] < 1e-12
