"""CPU oracle for shifted-window video attention.

This package is TEST INFRASTRUCTURE.  Only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never imports,
links or calls anything here, and this package imports nothing from the
product path.  The two share no code; only the seeded input generators in
``video_dit_shifted_gb300.synth`` (which hold none of the method's arithmetic)
feed both.

Everything is written for clarity, not speed: plain numpy in float64, one
window and one head at a time, following the definitions on the page
"Window-Aligned Sequence Parallelism (SeedVR2)" (vLLM-Omni design docs):

* ``oracle.plan``      -- §Window layouts: window size, regular and shifted
  intervals, window enumeration, canonical ids (obtained by windowing an
  arange cube, as the page says the reference does).
* ``oracle.permute``   -- §Motivation / §Plan A: at SP=1 a layout switch is a
  local row permutation.
* ``oracle.attention`` -- §SeedVR2 integration: one bidirectional attention
  per [video window ; replicated text] segment; §Text stream: the text output
  is the sum of per-window text outputs divided by the window count.

Parity pins (tests/test_oracle_*.py) tie each function to something other
than itself: closed forms, invariants the page states, library routines for
special cases (torch SDPA in float64) and brute force on tiny inputs.
One reading is NOT fixed by the pages: how half of an odd window length is
rounded when the shifted layout moves its cuts (floor is used).  Both roundings
partition the grid, so no invariant can tell them apart -- that choice is
"parity unpinned".
"""
