"""CPU oracle for the int4 weight-only group-wise decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (``int4_weight_only_group_gb300``) never imports it and shares no code
with it; the two meet only in the seeded input generators of ``workloads``.

Contents:
  decoder.py   the decode step in numpy float64, written from the pages'
               description of the method (see the module docstring);
  packspec.py  the packed int4 byte layout written from its specification in
               the C header, in plain Python loops, for bit-exact pack checks.

Pinning: every function is checked in ``tests/test_oracle_*.py`` against
closed forms, invariants, special cases, hand-worked values under
``tests/golden/`` or library routines on tiny inputs.  End-to-end text
agreement with the pages' own engine cannot be pinned (no code or weights are
published): parity unpinned for that, and only for that.
"""
