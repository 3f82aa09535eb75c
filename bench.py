#!/usr/bin/env python
"""Decode-attention benchmark for the gw library on one GB300 (or N, weak scaling).

A step is one pass of the whole hot path over one batch: for every layer of a
5 local + 1 global group, append the step's K/V rows (gw_kv_append) and run
decode attention (gw_decode_attn_local / gw_decode_attn_global).  Each layer
has its own pools, so a step reads ~1.4 GB of KV (inputs larger than L2).

Default workload: 16 decode slots, lengths U[512, 8192], 32 q heads; local 16
KV heads hd256, window 1024, bf16; global one KV head hd512, folded V + k_rot.

Printed: ONE JSON line (rank 0) with value = algorithmic KV GB/s of the whole
step (KV bytes the method must read / device time), steps/s, a roofline
object for the dominant call (the local attention call), an e2e number through
the C ABI with host buffers (every step uploads its inputs from one pinned
host buffer and downloads its outputs into another, one copy each, on copy
streams that overlap the neighbouring steps' compute), the
oracle timed on host cores (cpu_baseline), clock samples and kernel launch
counts.

--impl reference times the float64 CPU oracle (the reference arm) on a
bounded sample of the same workload.
"""

import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_hybrid_attention_gb300 import synth  # noqa: E402

METRIC = "decode-attn KV GB/s (frac of HBM peak) & batched decode steps/s, 1×GB300"
UNIT = "GB/s"

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of the dominant kernel per workload, with the SHA-256 of the kernel source it
# was captured from; reported as null once the source no longer matches.
# workload: (bytes, source file under csrc/, sha256)
NCU_TRAFFIC = {
    "serving": (275954944, "attn_local.cu", "ee26d615efa09d7ee5b7523db126b699a96d1ae5a0bb0db87505374decd5af3e"),
    "fp8_local": (552621056, "attn_local_e4m3_tc.cu", "128157e7a4e08dd613ad92bbe60548ac553a2889bdd6734fc6befe95a6678dd9"),
    "long_global": (1354160896, "attn_global.cu", "cb628c3d09d39c1e5efd439f40f2a4ca9157ebad9077365c371ca8e1754ff163"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="serving",
                    help="serving (default), fp8_local, long_global, long_global_full, long_global_e4m3 (the "
                         "opt-in e4m3 folded global pool), mixed, chunked, stack48, prefill_lane (the serving step "
                         "beside an SM-capped prefill lane)")
    ap.add_argument("--lane-share", type=float, default=0.35,
                    help="prefill_lane: share of the SMs given to the prefill lane")
    ap.add_argument("--bucket", type=int, default=0,
                    help="pad every layer's step to this many sequence slots, as a CUDA graph captured for a "
                         "batch bucket runs a smaller batch (0: no padding)")
    ap.add_argument("--separate-append", action="store_true",
                    help="append each step's K/V rows with gw_kv_append before the decode call, instead of inside "
                         "it (gw_append_decode_attn_*, used where the layer's step has decode rows only)")
    ap.add_argument("--no-early-inputs", action="store_true",
                    help="decode kernels read their plan inputs only after the previous kernel has finished "
                         "(gw_set_early_inputs(0)); by default they read them while it runs, which holds here "
                         "because a step's row offsets, lengths and block tables are uploaded before its first "
                         "layer")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch every step eagerly instead of replaying a CUDA graph")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-probe", action="store_true", help="skip the gw_bw_probe read-ceiling measurement")
    return ap.parse_args()


# --------------------------------------------------------------------------- setup
def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, 'measured' | 'fallback')."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def workload_layers(name, rank):
    """[(Layer, family key)] of one step; each layer has its own page tables."""
    base = {"long_global_full": "long_global", "long_global_e4m3": "long_global", "prefill_lane": "serving"}.get(
        name, name)
    sp = synth.spec(base)
    if rank:
        sp = synth.custom(sp.name, sp.seed + 7919 * rank, sp.num_q_heads, sp.lens, sp.n_rows, sp.families,
                          sp.n_local_layers, sp.n_global_layers)
    layers = []
    lkey = "local"
    gkey = {"long_global_full": "global_full", "long_global_e4m3": "global_e4m3"}.get(name, "global")
    for i in range(sp.n_local_layers):
        layers.append(synth.Layer(sp, lkey, layer=i))
    for i in range(sp.n_global_layers):
        layers.append(synth.Layer(sp, gkey, layer=100 + i))
    return sp, layers


def kv_bytes(layer):
    """Algorithmic KV bytes one attention call must read (keys in range x bytes per token)."""
    fam, sp = layer.fam, layer.spec
    tot = 0
    for L, n in zip(sp.lens.astype(np.int64), sp.n_rows.astype(np.int64)):
        if n == 0:
            continue
        if fam.kind == "local":
            toks = min(int(L), int(n) - 1 + fam.window)
            per = fam.kv_heads * 2 * 256 * (2 if fam.dtype == "bf16" else 1)
        else:
            toks = int(L)
            per = {"folded": 1280, "full": 2048, "folded_e4m3": 640}[fam.layout]
        tot += toks * per
    return tot


def prompt_flops(layer):
    """Tensor FLOPs of the prompt rows (sequences with n > 1 query rows) of one
    attention call: 2 contractions (q.K, p.V) x 2 flops x heads x dim x keys."""
    fam, sp = layer.fam, layer.spec
    tot = 0
    for L, n in zip(sp.lens.astype(np.int64), sp.n_rows.astype(np.int64)):
        if n <= 1:
            continue
        p = np.arange(L - n, L, dtype=np.int64)
        keys = np.minimum(p + 1, fam.window) if fam.kind == "local" else p + 1
        tot += int(keys.sum())
    return 4 * sp.num_q_heads * fam.head_dim * tot


class GpuLayer:
    def __init__(self, layer, gw, gen, dev, bucket=0):
        fam, sp = layer.fam, layer.spec
        self.layer, self.fam = layer, fam
        self.pool = gw.KVPool(fam.layout, fam.dtype, layer.num_pages, fam.kv_heads, device=dev)
        max_pos = int(np.max(sp.lens)) + 1
        self.table = gw.rope_cs(fam.theta, fam.rot_dim, fam.head_dim, max_pos, device=dev)
        sig = fam.sigma
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # history: every token the step reads that was cached before it
        _, slot, pos = layer.index("history")
        self._append_random(gw, gen, dev, slot, pos, sig)
        # the step's own inputs
        _, slot, pos = layer.index("new")
        n = len(slot)
        shape = (n, fam.kv_heads, 256) if fam.kind == "local" else (n, 512)
        self.v_new = (torch.randn(*shape, generator=gen, device=dev) * sig).to(torch.bfloat16)
        self.k_new = (torch.randn(*shape, generator=gen, device=dev) * sig).to(torch.bfloat16) \
            if fam.kind == "local" else self.v_new.clone()
        self.slot_new = torch.from_numpy(slot).to(dev)
        self.pos_new = torch.from_numpy(pos).to(dev)
        rows = int(sp.n_rows.sum())
        self.q = torch.randn(rows, sp.num_q_heads, fam.head_dim, generator=gen, device=dev).to(torch.bfloat16)
        self.out = torch.empty_like(self.q)
        self.cu = torch.from_numpy(layer.cu_rows()).to(dev)
        self.lens = torch.from_numpy(sp.lens.astype(np.int32)).to(dev)
        self.bt = torch.from_numpy(layer.block_table).to(dev)
        self.max_q_rows = int(max(1, sp.n_rows.max()))
        self.ws = gw.alloc_workspace(self.pool, sp.num_q_heads, len(sp.lens), self.bt.shape[1], self.max_q_rows,
                                     max(1, fam.window), device=dev)
        self.kv_bytes = kv_bytes(layer)
        self.prompt_flops = prompt_flops(layer)
        self.fused = False
        if bucket > len(sp.lens):
            self._pad_to_bucket(gw, bucket, dev)

    def _pad_to_bucket(self, gw, bucket, dev):
        """Pad the step to `bucket` sequence slots, as a graph captured for a
        batch bucket runs a smaller batch: the extra slots get zero query rows
        (the decode kernels plan no work for them) and append rows that write
        a sink page no sequence reads."""
        fam, sp = self.fam, self.layer.spec
        extra = bucket - len(sp.lens)
        sink = int(self.layer.unused_pages[0])
        i32 = dict(dtype=torch.int32, device=dev)
        self.cu = torch.cat([self.cu, self.cu[-1:].repeat(extra)])
        self.lens = torch.cat([self.lens, torch.zeros(extra, **i32)])
        self.bt = torch.cat([self.bt, torch.full((extra, self.bt.shape[1]), -1, **i32)])
        self.slot_new = torch.cat([self.slot_new, sink * 16 + torch.arange(extra, **i32) % 16])
        self.pos_new = torch.cat([self.pos_new, torch.zeros(extra, **i32)])
        self.k_new = torch.cat([self.k_new, torch.zeros((extra,) + tuple(self.k_new.shape[1:]), dtype=torch.bfloat16,
                                                        device=dev)])
        self.v_new = torch.cat([self.v_new, torch.zeros((extra,) + tuple(self.v_new.shape[1:]), dtype=torch.bfloat16,
                                                        device=dev)])
        self.ws = gw.alloc_workspace(self.pool, sp.num_q_heads, bucket, self.bt.shape[1], self.max_q_rows,
                                     max(1, fam.window), device=dev)

    def _append_random(self, gw, gen, dev, slot, pos, sig, chunk=1 << 18):
        fam = self.fam
        for a in range(0, len(slot), chunk):
            s_ = torch.from_numpy(slot[a:a + chunk]).to(dev)
            p_ = torch.from_numpy(pos[a:a + chunk]).to(dev)
            n = len(s_)
            shape = (n, fam.kv_heads, 256) if fam.kind == "local" else (n, 512)
            v = (torch.randn(*shape, generator=gen, device=dev) * sig).to(torch.bfloat16)
            k = (torch.randn(*shape, generator=gen, device=dev) * sig).to(torch.bfloat16) \
                if fam.kind == "local" else v
            gw.kv_append(self.pool, k, v, s_, p_, self.table, self.status)

    def can_fuse(self, gw):
        """Whether this layer's step appends inside its decode call
        (gw_append_decode_attn_*): decode rows only, on the bf16 local and
        bf16 folded global pools, where the fused call measured faster (one
        box: serving step 259.7 vs 275.0 us, long-context folded call 238.6
        vs 239.0 us).  On the e4m3 local pool (98.8 vs 94.6 us per fp8
        call), the full control (410.9 vs 406.7 us) and the e4m3 folded pool
        (200.9 vs 198.0 us) the two calls measured faster."""
        return self.max_q_rows == 1 and self.fam.dtype == "bf16" and self.fam.layout in ("local", "folded")

    def attend(self, gw, stream):
        if self.fused:
            # the step's rows appended by the decode call itself (re-appending
            # the same bytes when the call is replayed)
            if self.fam.kind == "local":
                gw.append_decode_attn_local(self.pool, self.k_new, self.v_new, self.table, self.q, self.out, self.cu,
                                            self.lens, self.bt, self.ws, self.fam.window, dev_status=self.status,
                                            stream=stream)
            else:
                gw.append_decode_attn_global(self.pool, self.k_new, self.v_new, self.table, self.q, self.out,
                                             self.cu, self.lens, self.bt, self.ws, dev_status=self.status,
                                             stream=stream)
            return
        if self.fam.kind == "local":
            gw.decode_attn_local(self.pool, self.q, self.out, self.cu, self.lens, self.bt, self.ws, self.fam.window,
                                 max_q_rows=self.max_q_rows, dev_status=self.status, stream=stream)
        else:
            gw.decode_attn_global(self.pool, self.q, self.out, self.cu, self.lens, self.bt, self.ws,
                                  max_q_rows=self.max_q_rows, dev_status=self.status, stream=stream)

    def prompt_view(self, dev):
        """Inputs of a call over this layer's prompt sequences alone (same
        pool and pages): its time is the prompt-row kernel's, the decode
        kernel finding no decode rows."""
        sp = self.layer.spec
        cu = self.layer.cu_rows()
        idx = [i for i, n in enumerate(sp.n_rows) if n > 1]
        if not idx:
            return None
        rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in idx])
        ridx = torch.from_numpy(rows).to(dev)
        n = sp.n_rows[idx].astype(np.int32)
        self.pv_q = self.q.index_select(0, ridx).contiguous()
        self.pv_out = torch.empty_like(self.pv_q)
        self.pv_cu = torch.from_numpy(np.concatenate([[0], np.cumsum(n)]).astype(np.int32)).to(dev)
        self.pv_lens = torch.from_numpy(sp.lens[idx].astype(np.int32)).to(dev)
        self.pv_bt = self.bt.index_select(0, torch.tensor(idx, device=dev)).contiguous()
        return len(idx)

    def attend_prompt(self, gw, stream):
        if self.fam.kind == "local":
            gw.decode_attn_local(self.pool, self.pv_q, self.pv_out, self.pv_cu, self.pv_lens, self.pv_bt, self.ws,
                                 self.fam.window, max_q_rows=self.max_q_rows, dev_status=self.status, stream=stream)
        else:
            gw.decode_attn_global(self.pool, self.pv_q, self.pv_out, self.pv_cu, self.pv_lens, self.pv_bt, self.ws,
                                  max_q_rows=self.max_q_rows, dev_status=self.status, stream=stream)

    def run(self, gw, stream, ev=None):
        if not self.fused:
            gw.kv_append(self.pool, self.k_new, self.v_new, self.slot_new, self.pos_new, self.table, self.status,
                         stream)
        if ev is not None:
            ev[0].record(stream)
        self.attend(gw, stream)
        if ev is not None:
            ev[1].record(stream)

    INPUTS = ("q", "k_new", "v_new", "slot_new", "pos_new", "cu", "lens", "bt")


class Arena:
    """One device buffer holding the named tensors of every layer (256-byte
    aligned views), mirrored by one pinned host buffer: a step's inputs go up
    in one copy and its outputs come back in one.  With bind=True the layers'
    tensors become views of this arena; bind() re-points them later."""

    def __init__(self, glayers, names, dev, bind=True, host=None):
        items, off = [], 0
        for g in glayers:
            for n in names:
                t = getattr(g, n)
                items.append((g, n, t, off))
                off += -(-t.numel() * t.element_size() // 256) * 256
        self.nbytes = off
        self.dev = torch.empty(off, dtype=torch.uint8, device=dev)
        self.views = []
        for g, n, t, o in items:
            view = self.dev[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            view.copy_(t)
            self.views.append((g, n, view))
        if bind:
            self.bind()
        self.host = host if host is not None else self.dev.cpu().pin_memory()

    def bind(self):
        for g, n, view in self.views:
            setattr(g, n, view)

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)

    def download(self):
        self.host.copy_(self.dev, non_blocking=True)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "samples": len(sms),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- oracle legs
_ORACLE_CACHE = {}


def _oracle_one(job):
    """The float64 oracle (append + attention) on one (layer, sequence) pair
    of a workload: returns (algorithmic KV bytes, seconds).  Each pair gets a
    pool of its own pages only (its block-table row renumbered 0..n-1), so a
    worker process holds one sequence's pages at a time."""
    from oracle import attention, pages, rope  # test infrastructure: CPU baseline leg only
    from oracle.formats import bf16_bits_to_f64
    name, li, s = job
    if name not in _ORACLE_CACHE:
        sp, layers = workload_layers(name, 0)
        _ORACLE_CACHE.clear()
        _ORACLE_CACHE[name] = (sp, layers, {})
    sp, layers, tables = _ORACLE_CACHE[name]
    layer = layers[li]
    fam = layer.fam
    key = (fam.theta, fam.rot_dim, fam.head_dim)
    if key not in tables:
        tables[key] = rope.rope_table(fam.theta, fam.rot_dim, fam.head_dim, int(sp.lens.max()) + 1)
    table = tables[key]
    k, v, _, pos = layer.gather([s])
    q = bf16_bits_to_f64(layer.q(s))
    L = int(sp.lens[s])
    row = layer.block_table[s]
    n_log = (L + 15) // 16
    bt = np.where(row[:n_log] >= 0, np.arange(n_log), -1)
    slot = (bt[pos // 16] * 16 + pos % 16).astype(np.int32)
    pb = pages.local_page_bytes(fam.kv_heads, fam.dtype) if fam.layout == "local" else \
        pages.global_page_bytes(fam.layout)
    pool = np.zeros(n_log * pb, np.uint8)
    t0 = time.perf_counter()
    if fam.layout == "local":
        pages.write_local(pool, fam.kv_heads, fam.dtype, k, v, slot, pos, table)
        attention.local_rows(pool, fam.kv_heads, fam.dtype, bt, L, q, fam.window, 1.0 / math.sqrt(256))
    else:
        pages.write_global(pool, fam.layout, k, v, slot, pos, table)
        attention.global_rows(pool, fam.layout, bt, L, q, 1.0 / math.sqrt(512))
    dt = time.perf_counter() - t0
    one = synth.custom("one", 0, sp.num_q_heads, sp.lens[s:s + 1], sp.n_rows[s:s + 1], sp.families)
    return kv_bytes(synth.Layer(one, layer.fam_key, layer=layer.layer)), dt


def _oracle_init(name):
    """Pool worker start-up: imports and the workload's page tables, outside
    the timed region."""
    import oracle  # noqa: F401  (test infrastructure: CPU baseline leg only)
    sp, layers = workload_layers(name, 0)
    _ORACLE_CACHE.clear()
    _ORACLE_CACHE[name] = (sp, layers, {})


def _oracle_order(name):
    sp, layers = workload_layers(name, 0)
    order = [(name, li, s) for s in range(len(sp.lens)) for li in range(len(layers)) if sp.n_rows[s] > 0]
    rng = np.random.Generator(np.random.PCG64(17))
    rng.shuffle(order)
    return order


def oracle_sample(name, budget_s):
    """The oracle on one host thread, whole (layer, sequence) pairs in a
    seeded order until about budget_s seconds of oracle time; returns
    (GB/s, description, seconds)."""
    done_bytes, t_used, n = 0, 0.0, 0
    for job in _oracle_order(name):
        b, dt = _oracle_one(job)
        done_bytes += b
        t_used += dt
        n += 1
        if t_used >= budget_s:
            break
    desc = "%d (layer, sequence) pairs of the %s step (append + attention per pair), float64 NumPy, 1 thread" % (
        n, name)
    return done_bytes / t_used / 1e9, desc, t_used


def oracle_pool_sample(name, budget_s):
    """The oracle on every host core this process may use: a process pool
    (spawned, one BLAS thread per worker) over the same seeded (layer,
    sequence) pairs, in waves of one pair per worker until about budget_s
    seconds of wall time; returns (GB/s over the wall time, cores,
    description, seconds)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    order = _oracle_order(name)
    done_bytes, n = 0, 0
    with mp.get_context("spawn").Pool(cores, initializer=_oracle_init, initargs=(name,)) as pool:
        pool.map(_oracle_one, [order[x % len(order)] for x in range(cores)], chunksize=1)   # warm-up wave
        t0 = time.perf_counter()
        i = cores
        while time.perf_counter() - t0 < budget_s:
            wave = [order[x % len(order)] for x in range(i, i + cores)]
            i += cores
            for b, _ in pool.map(_oracle_one, wave, chunksize=1):
                done_bytes += b
                n += 1
        wall = time.perf_counter() - t0
    desc = ("%d (layer, sequence) pairs of the %s step (append + attention per pair), float64 NumPy, %d worker "
            "processes x 1 thread, throughput over wall time" % (n, name, cores))
    return done_bytes / wall / 1e9, cores, desc, wall


def cpu_baseline(name, pool_budget_s, single_budget_s):
    gbs, cores, desc, _ = oracle_pool_sample(name, pool_budget_s)
    one, desc1, _ = oracle_sample(name, single_budget_s)
    return {"value": gbs, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
            "single_thread": {"value": one, "unit": UNIT, "cores": 1, "sample": desc1}}


# --------------------------------------------------------------------------- main
class Ranks:
    """The ranks of one run (torchrun environment: RANK, LOCAL_RANK,
    WORLD_SIZE, MASTER_ADDR/PORT).  Weak scaling: every rank serves its own
    independent batch of sequences, so the data path has no collective; the
    process group only brackets the timed region (barrier) and reduces the
    per-rank figures on the host side of the measurement."""

    def __init__(self, backend):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.backend = backend
        self.device = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)

    def barrier(self):
        if self.world > 1:
            torch.distributed.barrier()

    def _reduce(self, x, op):
        if self.world == 1:
            return float(x)
        dev = self.device if self.backend == "nccl" else torch.device("cpu")
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=op)
        return float(t.item())

    def max(self, x):
        return self._reduce(x, torch.distributed.ReduceOp.MAX if self.world > 1 else None)

    def sum(self, x):
        return self._reduce(x, torch.distributed.ReduceOp.SUM if self.world > 1 else None)

    def throughput(self, step_bytes, ms):
        """Whole-job GB/s: the bytes every rank's step read, over the slowest
        rank's time per step."""
        return self.sum(step_bytes) / (self.max(ms) * 1e-3) / 1e9

    def close(self):
        if self.world > 1:
            torch.distributed.destroy_process_group()


def prefill_lane_main(args, peak, peak_kind):
    """NEXT-4: the serving decode step with an async prefill lane beside it.

    The decode lane replays the serving step (5 local + 1 global layers, one
    decode row per sequence) on one stream; the prefill lane replays the
    appends and prompt rows of 4 new 2048-token prompts on the same six
    layer shapes on a second stream, its attention kernels capped at a share
    of the SMs (gw_set_max_ctas: these kernels run one CTA per SM, so a CTA
    cap is an SM cap) and the decode lane's at the rest.  Reported: the
    decode step alone, beside the capped lane and beside the uncapped lane,
    and the prefill step alone and in each lane.  `value` is the decode KV
    GB/s beside the capped lane."""
    ranks = Ranks("nccl")
    world, rank = ranks.world, ranks.rank
    dev = torch.device("cuda", ranks.local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    ranks.device = dev
    from paged_hybrid_attention_gb300 import gw
    gw.set_early_inputs(not args.no_early_inputs)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    share = args.lane_share
    cap_pre = max(1, int(round(share * sms)))
    cap_dec = max(1, sms - cap_pre)
    sp_d, layers_d = workload_layers("serving", rank)
    sp_p, layers_p = workload_layers("prefill", rank)
    gen = torch.Generator(device=dev).manual_seed(sp_d.seed + 17 * rank)
    dec = [GpuLayer(l, gw, gen, dev) for l in layers_d]
    pre = [GpuLayer(l, gw, gen, dev) for l in layers_p]
    torch.cuda.synchronize()
    dec_bytes = sum(g.kv_bytes for g in dec)
    pre_flops = sum(g.prompt_flops for g in pre)

    def capture(gls, cap, early=True):
        gw.set_max_ctas(cap)
        gw.set_early_launch(early)
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(2):
                    for g in gls:
                        g.run(gw, side)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for g in gls:
                    g.run(gw, torch.cuda.current_stream())
        finally:
            gw.set_max_ctas(0)
            gw.set_early_launch(True)
        return gr

    # the capped prefill lane launches each kernel only once its predecessor
    # has finished: early (programmatic) launches would park its CTAs on the
    # decode lane's SMs while they wait out a prompt kernel
    g_dec, g_pre = capture(dec, 0), capture(pre, 0)
    g_dec_c, g_pre_c = capture(dec, cap_dec), capture(pre, cap_pre, early=False)
    g_pre_ce = capture(pre, cap_pre)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(gr, st, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record(st)
            for _ in range(n):
                gr.replay()
            e1.record(st)
        return e0, e1

    for gr in (g_dec, g_pre, g_dec_c, g_pre_c, g_pre_ce):
        for _ in range(max(3, args.warmup)):
            gr.replay()
    torch.cuda.synchronize()
    ranks.barrier()
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    K = max(3, args.steps)
    a0, a1 = timed(g_dec, sa, K)
    torch.cuda.synchronize()
    dec_alone = a0.elapsed_time(a1) / K
    a0, a1 = timed(g_dec_c, sa, K)
    torch.cuda.synchronize()
    dec_capped_alone = a0.elapsed_time(a1) / K
    KP = max(2, min(K, 20))
    b0, b1 = timed(g_pre, sb, KP)
    torch.cuda.synchronize()
    pre_alone = b0.elapsed_time(b1) / KP
    b0, b1 = timed(g_pre_c, sb, 2)
    torch.cuda.synchronize()
    pre_capped_alone = b0.elapsed_time(b1) / 2

    def lanes(gd, gp):
        # the prefill lane runs M steps; the decode lane runs N steps inside
        # them, an event after each (the worst step is the longest gap
        # between two tokens of a decode stream)
        M = 3
        N = max(3, int(0.5 * M * pre_alone * (sms / cap_pre) / dec_alone))
        p0, p1 = timed(gp, sb, M)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(N + 1)]
        with torch.cuda.stream(sa):
            evs[0].record(sa)
            for i in range(N):
                gd.replay()
                evs[i + 1].record(sa)
        torch.cuda.synchronize()
        steps = [evs[i].elapsed_time(evs[i + 1]) for i in range(N)]
        worst = {"ms": max(steps), "step": int(np.argmax(steps)), "median_ms": statistics.median(steps)}
        return evs[0].elapsed_time(evs[N]) / N, worst, p0.elapsed_time(p1) / M, N, M

    dec_cap, dec_cap_worst, pre_cap, n_cap, m_cap = lanes(g_dec_c, g_pre_c)
    dec_cape, dec_cape_worst, pre_cape, _, _ = lanes(g_dec_c, g_pre_ce)
    dec_unc, dec_unc_worst, pre_unc, n_unc, m_unc = lanes(g_dec, g_pre)
    clk = clocks.stop()
    ranks.barrier()
    dec_cap_max = ranks.max(dec_cap)
    status = int(sum(int(g.status.item()) for g in dec + pre))
    if rank != 0:
        ranks.close()
        return
    gbs = lambda ms: dec_bytes / (ms * 1e-3) / 1e9
    value = ranks.throughput(dec_bytes, dec_cap)
    lane = {
        "sms": sms, "prefill_ctas": cap_pre, "decode_ctas": cap_dec, "share": share,
        "decode_step_alone_ms": dec_alone, "decode_gbs_alone": gbs(dec_alone),
        "decode_step_capped_alone_ms": dec_capped_alone, "prefill_step_capped_alone_ms": pre_capped_alone,
        "decode_step_capped_lane_ms": dec_cap, "decode_steps_capped_lane": dec_cap_worst,
        "decode_steps_uncapped_lane": dec_unc_worst,
        "capped_lane_with_early_launch": {"decode_step_ms": dec_cape, "decode_steps": dec_cape_worst,
                                          "prefill_step_ms": pre_cape}, "decode_gbs_capped_lane": gbs(dec_cap),
        "decode_step_uncapped_lane_ms": dec_unc, "decode_gbs_uncapped_lane": gbs(dec_unc),
        "prefill_step_alone_ms": pre_alone, "prefill_step_capped_ms": pre_cap, "prefill_step_uncapped_ms": pre_unc,
        "prefill_tflops_alone": pre_flops / (pre_alone * 1e-3) / 1e12,
        "prefill_tflops_capped": pre_flops / (pre_cap * 1e-3) / 1e12,
        "decode_steps_measured": {"capped": n_cap, "uncapped": n_unc},
        "prefill_steps_measured": {"capped": m_cap, "uncapped": m_unc},
        "how": "decode lane: CUDA graph of the serving step replayed on one stream; prefill lane: CUDA graph of the "
               "appends + prompt rows of 4 x 2048-token prompts replayed on a second stream, enqueued first; the "
               "decode steps timed with events on their stream while the prefill lane runs",
    }
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n_cap,
        "warmup": args.warmup, "ms_per_step": dec_cap_max, "steps_per_s": 1000.0 / dec_cap_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill_lane", "launch": "cuda_graph", "early_inputs": not args.no_early_inputs, "decode": "serving step (5 local + 1 global)",
                   "prefill": "4 prompts x 2048 rows, same layer shapes",
                   "l2": "inputs larger than L2: 1.43 GB of decode KV per step",
                   "parallelism": "dp%d (sequences sharded, no collective)" % world},
        "roofline": {"kernel": "serving decode step beside the capped prefill lane (all its kernels)", "bound": "hbm",
                     "achieved": gbs(dec_cap), "peak": peak, "unit": "GB/s", "frac": gbs(dec_cap) / peak,
                     "peak_kind": peak_kind, "traffic": None, "algorithmic_bytes_per_launch": dec_bytes,
                     "ms_per_launch": dec_cap},
        "lane": lane, "cpu_baseline": None, "e2e": None,
        "gpu_launches": (3 * len(dec)) * n_cap,
        "clocks": clk, "device_status": status,
    }
    print(json.dumps(line))
    ranks.close()


def main():
    args = parse()
    peak, peak_tf, peak_kind = peaks()

    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        ref_steps, ref_secs = [], []
        desc, cores = "", 1
        for _ in range(args.warmup + args.steps):
            gbs, cores, desc, secs = oracle_pool_sample(args.workload,
                                                        budget_s=max(1.0, 90.0 / max(1, args.steps + args.warmup)))
            ref_steps.append(gbs)
            ref_secs.append(secs)
        val = statistics.median(ref_steps[args.warmup:]) if args.steps else ref_steps[-1]
        ms = 1000.0 * (statistics.median(ref_secs[args.warmup:]) if args.steps else ref_secs[-1])
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, "l2": "n/a (CPU)",
                           "step": "one bounded sample of the workload (see cpu_baseline.sample)"},
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.workload == "prefill_lane":
        prefill_lane_main(args, peak, peak_kind)
        return

    ranks = Ranks("nccl")
    world, rank = ranks.world, ranks.rank
    dev = torch.device("cuda", ranks.local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    ranks.device = dev
    from paged_hybrid_attention_gb300 import gw
    gw.set_early_inputs(not args.no_early_inputs)

    sp, layers = workload_layers(args.workload, rank)
    gen = torch.Generator(device=dev).manual_seed(sp.seed + 17 * rank)
    glayers = [GpuLayer(l, gw, gen, dev, bucket=args.bucket) for l in layers]
    for g in glayers:
        g.fused = not args.separate_append and g.can_fuse(gw)
    arena_in = Arena(glayers, GpuLayer.INPUTS, dev)   # the step's inputs, one upload
    arena_out = Arena(glayers, ("out",), dev)         # the step's outputs, one download
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    step_bytes = sum(g.kv_bytes for g in glayers)
    locals_ = [g for g in glayers if g.fam.kind == "local"]
    dom = locals_ if locals_ else glayers
    dom_name = ("local decode attention call (%ssplit-KV decode + combine)"
                % ("the step's append inside the decode kernel, " if any(g.fused for g in dom) else "")) if locals_ else \
        "global decode attention call (tcgen05 decode with in-kernel plan + combine)"
    dom_bytes = statistics.mean(g.kv_bytes for g in dom)

    def step():
        for g in glayers:
            g.run(gw, torch.cuda.current_stream())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
    for g in glayers:
        g.status.zero_()

    # ---- device-timed region: K steps (CUDA-graph replays unless --eager)
    K = args.steps
    clocks = ClockSampler(dev.index)
    ranks.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(K):
        if graph is not None:
            graph.replay()
        else:
            step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms_rank = t0.elapsed_time(t1) / K
    # a sustained loop of at least one second right after, inside the same
    # clock-sampling window, so that the clock record has many samples under
    # load and a sustained rate stands beside the K-step figure
    n_sus = max(K, int(math.ceil(1.0 / max(ms_rank * 1e-3, 1e-6))))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for k in range(n_sus):
        if graph is not None:
            graph.replay()
        else:
            step()
    s1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ranks.barrier()
    sus_ms = s0.elapsed_time(s1) / n_sus
    ms = ranks.max(ms_rank)
    value = ranks.throughput(step_bytes, ms_rank)
    status = int(sum(int(g.status.item()) for g in glayers))

    # ---- dominant call, steady state: a CUDA graph of consecutive calls over
    # the dominant layers (each its own pool, so every call reads its KV from
    # HBM), replayed R times between CUDA events on the launching stream
    reps_in_graph = max(1, 20 // len(dom))
    n_calls = reps_in_graph * len(dom)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for g in dom:
            g.attend(gw, side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    gdom = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gdom):
        for _ in range(reps_in_graph):
            for g in dom:
                g.attend(gw, torch.cuda.current_stream())
    for _ in range(3):
        gdom.replay()
    torch.cuda.synchronize()
    R = 20
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(R):
        gdom.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    dom_ms = d0.elapsed_time(d1) / (R * n_calls)
    # the same call timed eagerly (events around each call of 50 eager steps)
    K2 = min(K, 50)
    evs = {id(g): [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K2)]
           for g in dom}
    for k in range(K2):
        for g in glayers:
            g.run(gw, stream, evs[id(g)][k] if id(g) in evs else None)
    torch.cuda.synchronize()
    dom_ms_eager = statistics.mean(e0.elapsed_time(e1) for g in dom for e0, e1 in evs[id(g)])

    # ---- the global call of a decode step with local layers too: its own
    # roofline, timed like the dominant call over enough global pools (extra
    # ones built for the purpose) that the calls' KV exceeds L2 twice over
    roof_global = None
    glob = [g for g in glayers if g.fam.kind == "global"]
    if locals_ and glob and all(g.max_q_rows == 1 for g in glob):
        gl = list(glob)
        gbytes = statistics.mean(g.kv_bytes for g in glob)
        need = int(math.ceil(2 * 129e6 / max(gbytes, 1)))
        for i in range(max(0, need - len(gl))):
            gl.append(GpuLayer(synth.Layer(sp, glob[0].layer.fam_key, layer=200 + i), gw, gen, dev))
        torch.cuda.synchronize()
        reps_g = max(1, 20 // len(gl))
        with torch.cuda.stream(side):
            for g in gl:
                g.attend(gw, side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg):
            for _ in range(reps_g):
                for g in gl:
                    g.attend(gw, torch.cuda.current_stream())
        for _ in range(3):
            gg.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(R):
            gg.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        g_ms = g0.elapsed_time(g1) / (R * reps_g * len(gl))
        g_ach = gbytes / (g_ms * 1e-3) / 1e9
        roof_global = {"kernel": "global decode attention call (tcgen05 decode with in-kernel plan + combine), "
                                 "CUDA-graph replay of %d consecutive calls over %d pools x %d, events on the "
                                 "launching stream" % (reps_g * len(gl), len(gl), R),
                       "bound": "hbm", "achieved": g_ach, "peak": peak, "unit": "GB/s", "frac": g_ach / peak,
                       "peak_kind": peak_kind, "frac_of_nominal_8000": g_ach / 8000.0,
                       "algorithmic_bytes_per_launch": gbytes, "ms_per_launch": g_ms}
        status += int(sum(int(g.status.item()) for g in gl[len(glob):]))

    # ---- the prompt-row kernel on its own: the same layers' prompt sequences
    # alone (same pools and pages), CUDA-graph replay as above
    prompt_ms = None
    pdom = [g for g in dom if g.prompt_flops > 0 and g.prompt_view(dev)]
    if pdom:
        with torch.cuda.stream(side):
            for g in pdom:
                g.attend_prompt(gw, side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp):
            for _ in range(reps_in_graph):
                for g in pdom:
                    g.attend_prompt(gw, torch.cuda.current_stream())
        for _ in range(3):
            gp.replay()
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(R):
            gp.replay()
        p1.record(stream)
        torch.cuda.synchronize()
        prompt_ms = p0.elapsed_time(p1) / (R * reps_in_graph * len(pdom))

    # ---- read ceiling of the decode kernels' copy pipeline (gw_bw_probe, 4 GiB)
    read_gbs = read_gbs_tma = None
    if not args.no_probe:
        probe_buf = torch.ones(4 << 30, dtype=torch.uint8, device=dev)   # 4 GiB, 256-byte aligned

        def probe_rate(fn):
            for _ in range(3):
                fn(probe_buf, stream=stream)
            best = []
            for _ in range(5):
                p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                p0.record(stream)
                fn(probe_buf, stream=stream)
                p1.record(stream)
                torch.cuda.synchronize()
                best.append(p0.elapsed_time(p1))
            return probe_buf.numel() / (min(best) * 1e-3) / 1e9

        read_gbs = probe_rate(gw.bw_probe)
        read_gbs_tma = probe_rate(gw.bw_probe_tma)
        del probe_buf

    # ---- end to end through the C ABI with host buffers: every step uploads
    # its inputs from pinned host memory and downloads its outputs, on their
    # own streams with two device buffer sets, so the copies of one step
    # overlap the computation of its neighbours (all inside the timed region)
    e2e = None
    if not args.no_e2e:
        h2d, d2h = arena_in.nbytes, arena_out.nbytes
        ins = [arena_in, Arena(glayers, GpuLayer.INPUTS, dev, bind=False, host=arena_in.host)]
        outs = [arena_out, Arena(glayers, ("out",), dev, bind=False)]
        up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(k):
            b = k % 2
            if k >= 2:
                up_s.wait_event(ev_comp[b])          # inputs[b] consumed by step k - 2
            with torch.cuda.stream(up_s):
                ins[b].upload()
                ev_up[b].record(up_s)
            stream.wait_event(ev_up[b])
            if k >= 2:
                stream.wait_event(ev_down[b])        # outputs[b] of step k - 2 are home
            ins[b].bind()
            outs[b].bind()
            for g in glayers:
                g.run(gw, stream)
            ev_comp[b].record(stream)
            down_s.wait_event(ev_comp[b])
            with torch.cuda.stream(down_s):
                outs[b].download()
                ev_down[b].record(down_s)

        for k in range(4):
            e2e_step(k)
        torch.cuda.synchronize()
        ranks.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_s.wait_event(e0)
        for k in range(K):
            e2e_step(k)
        stream.wait_stream(down_s)
        e1.record(stream)
        torch.cuda.synchronize()
        ins[0].bind()
        outs[0].bind()
        e2e_rank = e0.elapsed_time(e1) / K
        e2e_ms = ranks.max(e2e_rank)
        e2e = {"value": ranks.throughput(step_bytes, e2e_rank), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "how": "inputs up and outputs down every step from pinned host memory, copies on two streams "
                      "overlapping the neighbouring steps' compute (two device buffer sets)"}

    if rank != 0:
        ranks.close()
        return
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    dom_flops = statistics.mean(g.prompt_flops for g in dom)
    traffic = None
    if args.workload in NCU_TRAFFIC:
        tb, fname, sha = NCU_TRAFFIC[args.workload]
        with open(os.path.join(ROOT, "paged_hybrid_attention_gb300", "csrc", fname), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() == sha:
                traffic = tb
    how = dom_name + ", CUDA-graph replay of %d consecutive calls x %d, events on the launching stream" % (n_calls, R)
    if dom_flops > 0:
        # prompt rows are a dense contraction: tensor roofline of the prompt
        # kernel, timed on the layers' prompt sequences alone; the whole call
        # (decode rows too) is reported beside it
        tflops = dom_flops / (prompt_ms * 1e-3) / 1e12
        roofline = {"kernel": "prompt-row kernel: calls over the dominant layers' prompt sequences alone "
                              "(the decode kernel finds no decode rows), CUDA-graph replay of %d calls x %d, "
                              "events on the launching stream" % (reps_in_graph * len(pdom), R),
                    "bound": "tensor", "achieved": tflops, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": tflops / peak_tf, "peak_kind": peak_kind, "traffic": None,
                    "algorithmic_flops_per_launch": dom_flops, "ms_per_launch": prompt_ms,
                    "whole_call": {"what": how + " (decode rows + causal prompt rows)", "ms_per_launch": dom_ms,
                                   "ms_per_launch_eager": dom_ms_eager, "kv_gbs": achieved,
                                   "prompt_tflops": dom_flops / (dom_ms * 1e-3) / 1e12}}
    else:
        # the probe whose copy pipeline the dominant kernel uses: tensor-map
        # boxes for the local kernels (4 KB for bf16; the e4m3 kernel's 2 KB
        # boxes stream no faster), bulk copies for the global kernel
        tma_pipe = bool(locals_)
        probe = read_gbs_tma if tma_pipe else read_gbs
        roofline = {"kernel": how, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                    "frac_of_read_probe": achieved / probe if probe else None,
                    "read_probe": "gw_bw_probe_tma" if tma_pipe else "gw_bw_probe",
                    "frac_of_nominal_8000": achieved / 8000.0,
                    "algorithmic_bytes_per_launch": dom_bytes, "ms_per_launch": dom_ms,
                    "ms_per_launch_eager": dom_ms_eager}
    cpu = None
    if not args.no_cpu:
        cpu = cpu_baseline(args.workload, pool_budget_s=12.0, single_budget_s=8.0)
    # gw kernels per layer: append (unless the decode kernel appends), decode
    # (split plan computed in-kernel) and combine; prompt rows add a tile plan
    # and the prompt kernel
    launches_per_step = sum((0 if g.fused else 1) + 2 + (2 if g.max_q_rows > 1 else 0) for g in glayers)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "steps_per_s": 1000.0 / ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if any(g.fam.dtype == "e4m3" for g in glayers) else "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "launch": "eager" if graph is None else "cuda_graph",
                   "layers": "%d local + %d global" % (sp.n_local_layers,
                                                                                   sp.n_global_layers),
                   "batch": int(len(sp.lens)), "kv_bytes_per_step": step_bytes, "q_heads": sp.num_q_heads,
                   "bucket": args.bucket if args.bucket > len(sp.lens) else None,
                   "early_inputs": not args.no_early_inputs,
                   "append": ("inside the decode call (%d of %d layers)" % (sum(g.fused for g in glayers), len(glayers))
                              if any(g.fused for g in glayers) else "gw_kv_append before each decode call"),
                   "l2": "inputs larger than L2: %.2f GB of KV read per step" % (step_bytes / 1e9),
                   "parallelism": "dp%d (sequences sharded, no collective)" % world},
        "roofline": roofline,
        "roofline_global": roof_global,
        "sustained": {"steps": n_sus, "seconds": sus_ms * n_sus * 1e-3, "ms_per_step": sus_ms,
                      "value": ranks.throughput(step_bytes, sus_ms),
                      "what": "the same step replayed for at least 1 s right after the timed steps, inside the "
                              "clock-sampling window"},
        "bw_probe": None if read_gbs is None else {
            "read_gbs": read_gbs, "read_gbs_tma": read_gbs_tma, "bytes": 4 << 30,
            "what": "4 GiB streamed with no arithmetic, best of 5: gw_bw_probe through a bulk-copy pipeline "
                    "(8 warps x 2-stage 8 KiB rings per SM; the global decode copies whole pages in bulk), "
                    "gw_bw_probe_tma through the tensor-map pipeline (6 warps x 2-stage 16 KiB page-head rings "
                    "per SM of 4 KB boxes, as the bf16 local decode kernel)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": None if clk is None else dict(clk, window="the K timed steps and the sustained loop after them"),
        "device_status": status,
    }
    print(json.dumps(line))
    ranks.close()


if __name__ == "__main__":
    main()
