"""Rotary position embedding as the KV append applies it (oracle; test only).

[pegainfer] "Architecture notes": local layers rotate the full 256-dim head
with theta = 10k; global layers use a *proportional* RoPE in which only 128 of
the 512 head dims rotate while the frequency denominator stays the full head
dim (512), theta = 1M.  [Gewell] "the Why": RoPE touches only 25% of global K.

Readings fixed here (the pages do not spell them out):
  * The rotated slice is dims [0, R) of the head and pairs are "rotate-half":
    (i, i + R/2) for i in [0, R/2).
  * Frequency i is inv_f_i = theta^(-2 i / D_full) with D_full the full head
    dim (256 local, 512 global); so the global slice uses the R/2 = 64
    highest frequencies of a 512-dim spectrum.
  * The table entry for position p is (cos, sin) of p * inv_f_i computed in
    float64 and rounded once to float32.
  * The rotation is evaluated in binary32 with a fixed operation order and no
    fused multiply-add:
        r0 = fl(fl(x0 * c) - fl(x1 * s))
        r1 = fl(fl(x1 * c) + fl(x0 * s))
    where x0 = x[i], x1 = x[i + R/2] are the exact float32 values of the bf16
    inputs.  NumPy float32 arithmetic rounds every operation, which is this.
"""

import numpy as np


def inv_freq(theta, rot_dim, d_full):
    i = np.arange(rot_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / np.float64(d_full))


def rope_table(theta, rot_dim, d_full, max_pos):
    """float32 [max_pos, rot_dim // 2, 2] table of (cos, sin)."""
    pos = np.arange(max_pos, dtype=np.float64)
    ang = pos[:, None] * inv_freq(theta, rot_dim, d_full)[None, :]
    tab = np.empty((max_pos, rot_dim // 2, 2), dtype=np.float32)
    tab[..., 0] = np.cos(ang)   # float64 -> float32 assignment rounds to nearest
    tab[..., 1] = np.sin(ang)
    return tab


def rotate_half_f32(x32, cs):
    """Rotate float32 x[..., R] by table rows cs[..., R/2, 2] (float32)."""
    x32 = np.asarray(x32, dtype=np.float32)
    h = x32.shape[-1] // 2
    x0, x1 = x32[..., :h], x32[..., h:]
    c, s = cs[..., 0].astype(np.float32), cs[..., 1].astype(np.float32)
    r0 = (x0 * c) - (x1 * s)
    r1 = (x1 * c) + (x0 * s)
    assert r0.dtype == np.float32 and r1.dtype == np.float32
    return np.concatenate([r0, r1], axis=-1)
