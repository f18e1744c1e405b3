"""CPU float64 oracle for packed-sequence (varlen) block-diagonal causal attention.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
may import, call or run anything in this package.  The GPU library
(``packed_sequence_varlen_gb300``) never imports it, and this package never
imports the GPU library: the two share no code.  The only module both sides
use is ``seeded_inputs`` (random draws and workload sizes, no arithmetic of
the method).

What the oracle computes, and the passage each part follows:

* ``attention``  -- per-segment exact causal softmax attention and its analytic
  backward ("Packing与 FlashAttention Varlen", section 1 "Mental Model" and
  section 5 "FlashAttention Kernel：从 Boundary 到地址域"; the permission rule of
  "Pack sequences without joining their contexts", "Permission depends on the
  example"), plus a dense brute-force [T, T] permission-mask version.
* ``packing``    -- next-fit and best-fit-decreasing planners (blog section 2;
  course "Fill only the current row"), the boundary metadata (blog section 3),
  and the course's packed storage rows ("Fill only the current row").
* ``tiles``      -- the segment-aware tile maps (blog section 5 tile bounds;
  course "History" edge-traversal check).
* ``loss``       -- the token-weighted objective and the constructed-logit probe
  (course "Keep the same nine-target objective").

Pins (tests/test_oracle_*.py): brute force on tiny inputs, the pages' worked
layouts and printed loss values, closed forms, torch's float64 SDPA and
autograd, central finite differences, and segment invariants.  No function
here is "parity unpinned".
"""
