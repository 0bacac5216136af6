"""CPU oracle for layer-streamed execution — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or run anything in this package. The product path (the
C-ABI library and its Python binding) never calls it, and this package imports
nothing from the product: the two share only the seeded input generator in
``synth``.

Contents:
  * ``forward``  — the plain fp64 forward of every segment kind, with all weights
                   resident (layer streaming moves weights, it does not change
                   the arithmetic).
  * ``policy``   — an event-level simulator of the slot / residency / prefetch
                   policy that produces the exact schedule the runtime must
                   execute.
  * ``brute``    — brute-force enumeration of feasible plans and an occupancy
                   replay used to pin ``policy``.

Every function cites the page passage it follows. Pins: ``tests/test_oracle_pins.py``
and ``tests/test_policy_oracle.py`` (closed forms, page rows and worked numbers,
brute force). Parity-unpinned items are listed in the module docstrings.
"""
