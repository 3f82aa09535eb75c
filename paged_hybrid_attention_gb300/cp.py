"""Context parallelism for one long global sequence across ranks.

"Gemma 4" (pegainfer model page), "Raised ceiling" and "Limits": a global
layer attends over the whole history (contexts up to 262144 tokens) and the
pages' engine runs one GPU per sequence.  The decode kernels already split a
long sequence into chunks of pages and merge the chunks' partial results by
their log-sum-exp; this module spreads the same split over ranks:

* rank r holds a contiguous range of the sequence's pages (``shard_pages``),
  in a pool of its own with the pages renumbered from 0, and runs
  ``gw_decode_attn_global_lse`` over them: attention over its keys plus the
  rows' log-sum-exp;
* one exchange step gathers every rank's (output, log-sum-exp) to all ranks
  (``exchange``: an all-gather through torch.distributed, NCCL or gloo);
* ``gw_merge_lse`` merges them, in rank order, into the rows' outputs.

Only decode rows (one query row per sequence) are split this way.  The
module is host-side plumbing over the C ABI: every step of the arithmetic
runs in libgw.so.
"""

import torch

PAGE = 16


def _gw():
    from . import gw   # the C library; importing it fails loudly if it is not built
    return gw


def shard_pages(seq_len, world, rank):
    """(first page, end page, first key, end key) of `rank`'s contiguous share
    of a sequence of `seq_len` tokens split over `world` ranks.  Pages are
    dealt in equal contiguous runs (the last ranks may get one page fewer, or
    none); the keys are the tokens of those pages that exist."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d outside a world of %d" % (rank, world))
    pages = (seq_len + PAGE - 1) // PAGE
    base, extra = divmod(pages, world)
    p0 = rank * base + min(rank, extra)
    p1 = p0 + base + (1 if rank < extra else 0)
    return p0, p1, min(seq_len, p0 * PAGE), min(seq_len, p1 * PAGE)


def local_attention(pool, q, block_table, n_keys, workspace, scale=None, stream=None):
    """This rank's part: attention of the decode rows `q` ([rows, heads, 512]
    bf16, one row per sequence) over its `n_keys` keys (int32 tensor [rows]) in
    `pool` through `block_table` (its own pages, renumbered from 0).  Returns
    (output bf16, log-sum-exp float32 [rows, heads])."""
    rows, heads = int(q.shape[0]), int(q.shape[1])
    out = torch.empty_like(q)
    lse = torch.empty(rows, heads, dtype=torch.float32, device=q.device)
    cu = torch.arange(rows + 1, dtype=torch.int32, device=q.device)
    _gw().decode_attn_global_lse(pool, q, out, lse, cu, n_keys, block_table, workspace, scale=scale, stream=stream)
    return out, lse


def exchange(out, lse, group=None):
    """The split's one exchange step: every rank's (output, log-sum-exp),
    gathered on every rank in rank order."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    outs = [torch.empty_like(out) for _ in range(world)]
    lses = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(outs, out.contiguous(), group=group)
    dist.all_gather(lses, lse.contiguous(), group=group)
    return outs, lses


def merge(outs, lses, stream=None):
    """gw_merge_lse of the gathered parts: the rows' attention over all keys
    (bf16) and their overall log-sum-exp (float32)."""
    out = torch.empty_like(outs[0])
    lse = torch.empty_like(lses[0])
    _gw().merge_lse(outs, lses, out, lse, stream=stream)
    return out, lse
