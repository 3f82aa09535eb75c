"""Decode / prompt-row attention over the paged pools in float64 (oracle; test only).

Definitions, for one sequence whose cache holds positions [0, L) after the
append, one query row at position p and q head h (HQ heads, KVH KV heads,
group G = HQ / KVH, KV head of h is h // G):

    logits_j = scale * sum_d q[h, d] * K[j, h // G, d]        j in J(p)
    o[h]     = sum_j softmax(logits)_j * V[j, h // G, :]

* Local (sliding) layers  [pegainfer] "Architecture notes", "Scheduling":
  window W = 1024; J(p) = [max(0, p - W + 1), p], i.e. the last W positions
  including the row's own token.
* Global layers  [pegainfer] "Architecture notes", [Gewell] "the Why":
  J(p) = [0, p]; one KV head; K is rebuilt from the folded row as
  K_j = k_rot_j || V_j[128:512] (the oracle materialises it explicitly).
* Decode rows: a sequence contributing one row has p = L - 1.  A sequence
  contributing n rows (a prompt segment computed in the same step,
  [pegainfer] "Scheduling") has rows at p = L - n, ..., L - 1 (causal).
* scale = 1 / sqrt(head dim); the pages give none, the synthetic workloads fix
  this one.

Softmax is max-subtracted in float64.  Split-KV: ``partial`` gives
(m, l, o) = (max logit, sum exp(logit - m), sum exp(logit - m) V) over a
subset of J and ``combine`` merges them by the log-sum-exp rule
o = sum_c e^{m_c - M} o_c / sum_c e^{m_c - M} l_c.
"""

import numpy as np

from . import pages


def attend(q64, K64, V64, scale):
    """One query row, all heads. q64 [HQ, D]; K64, V64 [n, KVH, D] -> [HQ, D]."""
    HQ = q64.shape[0]
    KVH = K64.shape[1]
    G = HQ // KVH
    out = np.empty((HQ, V64.shape[2]), dtype=np.float64)
    for h in range(HQ):
        g = h // G
        s = scale * (K64[:, g, :] @ q64[h])
        w = np.exp(s - s.max())
        out[h] = (w @ V64[:, g, :]) / w.sum()
    return out


def partial(q64, K64, V64, scale):
    """Unnormalised split-KV partial over the given keys: (m [HQ], l [HQ], o [HQ, D])."""
    HQ = q64.shape[0]
    G = HQ // K64.shape[1]
    m = np.empty(HQ)
    l = np.empty(HQ)
    o = np.empty((HQ, V64.shape[2]))
    for h in range(HQ):
        g = h // G
        s = scale * (K64[:, g, :] @ q64[h])
        m[h] = s.max()
        w = np.exp(s - m[h])
        l[h] = w.sum()
        o[h] = w @ V64[:, g, :]
    return m, l, o


def combine(parts):
    """Merge a list of (m, l, o) partials of the same rows."""
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    num = sum(np.exp(p[0] - M)[:, None] * p[2] for p in parts)
    den = sum(np.exp(p[0] - M) * p[1] for p in parts)
    return num / den[:, None]


def local_keys(p, window):
    return np.arange(max(0, p - window + 1), p + 1)


def global_keys(p):
    return np.arange(0, p + 1)


def rebuild_global_k(rows64):
    """Folded rows [n, 640] = V || k_rot  ->  (K [n, 512], V [n, 512])."""
    V = rows64[:, :pages.GLOBAL_D]
    krot = rows64[:, pages.GLOBAL_D:]
    K = np.concatenate([krot, V[:, pages.GLOBAL_ROT:]], axis=1)
    return K, V


def split_full_rows(rows64):
    """Full rows [n, 1024] = K || V -> (K, V)."""
    return rows64[:, :pages.GLOBAL_D], rows64[:, pages.GLOBAL_D:]


def local_rows(pool_u8, kv_heads, dtype, block_row, L, q64, window, scale):
    """Outputs for the n = q64.shape[0] rows of one sequence on a local layer."""
    n = q64.shape[0]
    out = np.empty_like(q64)
    for r in range(n):
        p = L - n + r
        J = local_keys(p, window)
        K, V = pages.read_local(pool_u8, kv_heads, dtype, block_row, J)
        out[r] = attend(q64[r], K, V, scale)
    return out


def global_rows(pool_u8, layout, block_row, L, q64, scale):
    """Outputs for the rows of one sequence on a global layer (folded, full or
    folded_e4m3 pool)."""
    n = q64.shape[0]
    rows = pages.read_global_rows(pool_u8, layout, block_row, np.arange(L))
    K, V = split_full_rows(rows) if layout == "full" else rebuild_global_k(rows)
    out = np.empty_like(q64)
    for r in range(n):
        p = L - n + r
        J = global_keys(p)
        out[r] = attend(q64[r], K[J][:, None, :], V[J][:, None, :], scale)
    return out
