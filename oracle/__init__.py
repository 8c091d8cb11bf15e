"""Float64 CPU oracle for paged split-KV decode, log2-LSE merge and the two-level
cascade.  TEST INFRASTRUCTURE ONLY.

This package is the independent definition the CUDA library is checked against.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import it.  It shares no code with the CUDA library
(``paged_split_kv_decode_gb300``) and imports nothing from it.

Modules
-------
attention  gather pages into contiguous K/V and run plain softmax attention in
           float64; per-chunk partials; the log2-LSE merge; fp8-e4m3 decoding.
planner    split-KV work list, shared-prefix detection, cascade plan, head
           stacking index maps (pure Python integers).
cascade    the two-level cascade evaluated level by level in float64, for
           diagnosis and for the invariants the pages state.
rope_append  rotary embedding of the new token's query and key rows and their
           append into the paged pools (bf16 or fp8-e4m3 codes).  The rotation runs
           in float32, since its roundings decide bit patterns; tests pin it to the
           exact float64 rotation.

Every numeric function is pinned by ``tests/test_oracle_*.py`` against brute force,
closed forms, library routines or the pages' invariants.  Parity is pinned for all
functions here; the planner's tie-break and cap-before-threshold ordering are
readings of the pages (see the planner docstrings), pinned by hand-made cases.
"""
from . import attention, planner, cascade, rope_append  # noqa: F401
