"""Float64 CPU oracle of the Hymba hybrid-head layer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the library or its binding.

* ``oracle.hymba_ref`` -- vectorised NumPy float64 definition (prefill, decode,
  residual stack).
* ``oracle.brute``     -- a loop-only second oracle for tiny shapes.

Parity status: the attention mask/count, the scan recurrence, the conv, the
norm/fusion, KV sharing and prefill/decode consistency are pinned by closed
forms, special cases, library routines and invariants in
``tests/test_oracle_pins.py``.  The absolute outputs at random weights have no
printed worked example on the pages; beyond the pins they are fixed only by
the agreement of the two oracles (parity unpinned in that narrow sense).
"""
