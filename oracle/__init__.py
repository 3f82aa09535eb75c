"""CPU oracle for paged hybrid decode attention (TEST INFRASTRUCTURE ONLY).

This package is a plain, slow, float64 NumPy statement of what the GPU path
computes.  It exists to check the CUDA library and nothing else: only the test
suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference legs of
``bench.py`` may import it.  The product path (``paged_hybrid_attention_gb300``)
never imports it and has no CPU fallback.

It shares no code with the CUDA path: no kernels, headers, tables, helpers or
pre/post-processing.  Its parts:

* ``formats``   - bf16 and OCP e4m3 ("e4m3fn") encode/decode from the format
                  definitions, by integer bit operations.
* ``rope``      - the fp32 cos/sin table and the fixed-order fp32 rotate-half.
* ``pages``     - the three paged pool layouts (local, global folded V+k_rot,
                  global full K+V) with a page writer and a gather reader.
* ``attention`` - windowed / causal softmax attention in float64, the
                  compressed-K rebuild, and the split / log-sum-exp combine.

Sources (cited by page title and section):
  [Gewell]    "Gewell - Gemma4 inference engine", section "the Why".
  [pegainfer] "Gemma 4" (pegainfer model page): "Scheduling",
              "Architecture notes", "Reproducibility under concurrency".
  [PR1012]    "feat(gemma4): the sliding family serves an opt in fp8 KV pool",
              "Description" and "Verification".

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, library routines or the format standards;
none is "parity unpinned".
"""

from . import formats, rope, pages, attention  # noqa: F401
