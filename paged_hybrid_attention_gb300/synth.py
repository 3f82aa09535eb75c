"""Seeded synthetic workloads shared by the tests and the benchmark.

This module draws random numbers and lays out page tables; it holds none of
the attention, RoPE or rounding arithmetic.  Values are drawn in float32 with
``torch.Generator`` on the CPU and cast to bf16 by torch; callers receive the
bf16 bit patterns as ``numpy.uint16``.

Workloads (sizes from the decode shapes the pages serve: 16-token pages,
window 1024, local hd256 with GQA, global hd512 with one KV head, 5 local
layers per global layer):

  tiny        2 sequences (L = 37, 100), 8 q heads; local 4 KV heads, window
              32; global rotated slice 128 dims, RoPE base 10000 for both.
  serving     16 decode slots, L ~ U[512, 8192], 32 q heads; local 16 KV
              heads, window 1024, bf16; global folded; 5 local + 1 global.
  fp8_local   64 sequences, L ~ U[4096, 32768], local only, e4m3 pool, values
              N(0, 0.5) (the clip at +-448 never binds); bf16 control.
  long_global 8 slots at L = 131072, global only, folded vs full control,
              and the opt-in e4m3 folded pool of the same tokens.
  mixed       48 decode streams, L ~ U[1024, 16384], plus 4 new prompts of 2048
              rows appended and attended in the same step; both families.
  mixed_e4m3  the mixed step with the local family on an e4m3 pool (N(0, 0.5)).
  chunked     32 decode streams, L ~ U[1024, 16384], plus 4 prompts continuing
              with a 1024-row chunk over U[4096, 16384] cached tokens (the
              chunked walk); both families.
  stack48     the serving shapes over a 48-layer stack (40 local + 8 global
              layers, each with its own pools).
  prefill     4 new prompts of 2048 rows with the serving families (5 local
              + 1 global layers): the work of an async prefill lane that runs
              beside the serving decode step.

Every sequence's tensors come from their own generator seed, so one sequence
can be regenerated alone (the oracle checks samples of the big workloads).
Physical pages are a seeded permutation of the pool, so a sequence's pages
are scattered.  Global K is tied to V before RoPE (k_pre = v), which is the
tied-KV structure the folded layout relies on.
"""

from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 16


@dataclass
class Family:
    kind: str            # "local" or "global"
    dtype: str           # "bf16" or "e4m3"
    layout: str          # "local", "folded", "full" or "folded_e4m3"
    kv_heads: int
    head_dim: int
    rot_dim: int
    theta: float
    window: int          # 0 for global
    sigma: float = 1.0


@dataclass
class Spec:
    name: str
    seed: int
    num_q_heads: int
    lens: np.ndarray                 # int32 [B], length after this step's append
    n_rows: np.ndarray               # int32 [B], query rows this step
    families: dict = field(default_factory=dict)
    n_local_layers: int = 0
    n_global_layers: int = 0


def _draw_lens(seed, B, lo, hi):
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(lo, hi + 1, size=B).astype(np.int32)


def spec(name):
    """Workload spec by name (see module docstring)."""
    if name == "tiny":
        loc = Family("local", "bf16", "local", 4, 256, 256, 1e4, 32)
        glo = Family("global", "bf16", "folded", 1, 512, 128, 1e4, 0)
        return Spec(name, 1001, 8, np.array([37, 100], np.int32), np.ones(2, np.int32),
                    {"local": loc, "global": glo, "global_full": _full(glo), "global_e4m3": _e4m3(glo)}, 1, 1)
    if name == "serving":
        lens = _draw_lens(1002, 16, 512, 8192)
        loc = Family("local", "bf16", "local", 16, 256, 256, 1e4, 1024)
        glo = Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
        return Spec(name, 1002, 32, lens, np.ones(16, np.int32),
                    {"local": loc, "global": glo}, 5, 1)
    if name == "fp8_local":
        lens = _draw_lens(1003, 64, 4096, 32768)
        loc = Family("local", "e4m3", "local", 16, 256, 256, 1e4, 1024, sigma=0.5)
        ctl = Family("local", "bf16", "local", 16, 256, 256, 1e4, 1024, sigma=0.5)
        return Spec(name, 1003, 32, lens, np.ones(64, np.int32),
                    {"local": loc, "local_bf16": ctl}, 1, 0)
    if name == "long_global":
        lens = np.full(8, 131072, np.int32)
        glo = Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
        return Spec(name, 1004, 32, lens, np.ones(8, np.int32),
                    {"global": glo, "global_full": _full(glo), "global_e4m3": _e4m3(glo)}, 0, 1)
    if name == "mixed":
        dec = _draw_lens(1005, 48, 1024, 16384)
        lens = np.concatenate([dec, np.full(4, 2048, np.int32)]).astype(np.int32)
        rows = np.concatenate([np.ones(48, np.int32), np.full(4, 2048, np.int32)])
        loc = Family("local", "bf16", "local", 16, 256, 256, 1e4, 1024)
        glo = Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
        return Spec(name, 1005, 32, lens, rows, {"local": loc, "global": glo}, 5, 1)
    if name == "mixed_e4m3":
        # the mixed step with the sliding family on its opt-in e4m3 pool
        base = spec("mixed")
        loc = Family("local", "e4m3", "local", 16, 256, 256, 1e4, 1024, sigma=0.5)
        return Spec(name, base.seed, base.num_q_heads, base.lens, base.n_rows,
                    {"local": loc, "global": base.families["global"]}, 5, 1)
    if name == "chunked":
        dec = _draw_lens(1006, 32, 1024, 16384)
        hist = _draw_lens(1106, 4, 4096, 16384)
        lens = np.concatenate([dec, hist + 1024]).astype(np.int32)
        rows = np.concatenate([np.ones(32, np.int32), np.full(4, 1024, np.int32)])
        loc = Family("local", "bf16", "local", 16, 256, 256, 1e4, 1024)
        glo = Family("global", "bf16", "folded", 1, 512, 128, 1e6, 0)
        return Spec(name, 1006, 32, lens, rows, {"local": loc, "global": glo}, 5, 1)
    if name == "prefill":
        base = spec("serving")
        return Spec(name, 1007, base.num_q_heads, np.full(4, 2048, np.int32), np.full(4, 2048, np.int32),
                    base.families, 5, 1)
    if name == "stack48":
        base = spec("serving")
        return Spec(name, base.seed, base.num_q_heads, base.lens, base.n_rows, base.families, 40, 8)
    raise KeyError(name)


def _full(fam):
    return Family(fam.kind, fam.dtype, "full", fam.kv_heads, fam.head_dim, fam.rot_dim,
                  fam.theta, fam.window, fam.sigma)


def _e4m3(fam):
    """The opt-in e4m3 folded pool of a global family (same tokens)."""
    return Family(fam.kind, "e4m3", "folded_e4m3", fam.kv_heads, fam.head_dim, fam.rot_dim,
                  fam.theta, fam.window, fam.sigma)


def custom(name, seed, num_q_heads, lens, n_rows, families, n_local=1, n_global=1):
    """A spec built by hand (edge-case tests)."""
    return Spec(name, seed, num_q_heads, np.asarray(lens, np.int32),
                np.asarray(n_rows, np.int32), families, n_local, n_global)


# ------------------------------------------------------------------ helpers
def _gen(*key):
    seed = 0
    for k in key:
        seed = (seed * 1_000_003 + int(k)) % (2 ** 62)
    return torch.Generator().manual_seed(seed)


def randn_bf16_bits(shape, sigma, *key):
    x = torch.randn(*shape, generator=_gen(*key), dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def first_position(L, n, fam):
    """Earliest logical position the step's rows read on this family."""
    if fam.kind == "local":
        return max(0, (L - n) - fam.window + 1)
    return 0


class Layer:
    """One layer's paged inputs: page table, pool size and per-sequence tensors."""

    def __init__(self, sp, fam_key, layer=0, spare_pages=3):
        self.spec = sp
        self.fam = sp.families[fam_key]
        self.fam_key = fam_key
        self.layer = layer
        fam = self.fam
        B = len(sp.lens)
        self.B = B
        first = [first_position(int(L), int(n), fam) // PAGE for L, n in zip(sp.lens, sp.n_rows)]
        last = [(int(L) - 1) // PAGE if L > 0 else -1 for L in sp.lens]
        self.max_pages = max([1] + [(int(L) + PAGE - 1) // PAGE for L in sp.lens])
        need = sum(max(0, b - a + 1) for a, b in zip(first, last))
        self.num_pages = need + spare_pages
        g = np.random.Generator(np.random.PCG64(sp.seed * 7919 + layer * 31 + _fam_id(fam_key)))
        perm = g.permutation(self.num_pages).astype(np.int32)
        bt = np.full((B, self.max_pages), -1, np.int32)
        k = 0
        for s in range(B):
            for lp in range(first[s], last[s] + 1):
                bt[s, lp] = perm[k]
                k += 1
        self.block_table = bt
        self.unused_pages = np.sort(perm[k:])      # never written: sentinel pages
        self.first_pos = np.array([first_position(int(L), int(n), fam)
                                   for L, n in zip(sp.lens, sp.n_rows)], np.int64)

    # -- per-sequence tensors -------------------------------------------------
    def kv(self, s):
        """(positions, k_bits, v_bits) of every cached token of sequence s this step reads."""
        fam, sp = self.fam, self.spec
        L = int(sp.lens[s])
        pos = np.arange(self.first_pos[s], L, dtype=np.int32)
        n = len(pos)
        seed = (sp.seed, self.layer, _fam_id(self.fam_key), s)
        if fam.kind == "local":
            k = randn_bf16_bits((n, fam.kv_heads, fam.head_dim), fam.sigma, *seed, 1)
            v = randn_bf16_bits((n, fam.kv_heads, fam.head_dim), fam.sigma, *seed, 2)
        else:
            v = randn_bf16_bits((n, fam.head_dim), fam.sigma, *seed, 2)
            k = v.copy()       # tied K and V before RoPE: k_pre = v
        return pos, k, v

    def q(self, s):
        fam, sp = self.fam, self.spec
        n = int(sp.n_rows[s])
        return randn_bf16_bits((n, sp.num_q_heads, fam.head_dim), 1.0,
                               sp.seed, self.layer, _fam_id(self.fam_key), s, 3)

    def slots(self, s, pos):
        pos = np.asarray(pos, np.int64)
        return (self.block_table[s][pos // PAGE].astype(np.int64) * PAGE + pos % PAGE).astype(np.int32)

    def new_mask(self, s, pos):
        """True for positions appended in this step (the sequence's last n_rows)."""
        L, n = int(self.spec.lens[s]), int(self.spec.n_rows[s])
        return np.asarray(pos) >= L - n

    def gather(self, seqs=None, part="all"):
        """Concatenated append batch (k, v, slot, pos) over sequences.

        part: "history" (tokens already cached before the step), "new" (the
        step's own rows) or "all".
        """
        seqs = range(self.B) if seqs is None else seqs
        ks, vs, ss, ps = [], [], [], []
        for s in seqs:
            pos, k, v = self.kv(s)
            m = self.new_mask(s, pos)
            sel = m if part == "new" else (~m if part == "history" else np.ones_like(m))
            ks.append(k[sel]); vs.append(v[sel]); ps.append(pos[sel]); ss.append(self.slots(s, pos[sel]))
        return (np.concatenate(ks), np.concatenate(vs),
                np.concatenate(ss).astype(np.int32), np.concatenate(ps).astype(np.int32))

    def index(self, part="all"):
        """(seq, slot, pos) int arrays of the tokens gather() would return, without values."""
        ss, sl, ps = [], [], []
        for s in range(self.B):
            L, n = int(self.spec.lens[s]), int(self.spec.n_rows[s])
            lo = int(self.first_pos[s]) if part != "new" else L - n
            hi = L - n if part == "history" else L
            pos = np.arange(lo, hi, dtype=np.int64)
            ss.append(np.full(len(pos), s, np.int32))
            ps.append(pos)
            sl.append(self.slots(s, pos) if len(pos) else np.zeros(0, np.int32))
        return (np.concatenate(ss), np.concatenate(sl).astype(np.int32), np.concatenate(ps).astype(np.int32))

    def queries(self, seqs=None):
        seqs = range(self.B) if seqs is None else seqs
        return np.concatenate([self.q(s) for s in seqs])

    def cu_rows(self):
        return np.concatenate([[0], np.cumsum(self.spec.n_rows)]).astype(np.int32)


def _fam_id(key):
    return {"local": 1, "global": 2, "global_full": 2, "local_bf16": 1, "global_e4m3": 2}[key]
