"""Float64 CPU oracle for the Mamba-2 SSD forward and the scalar selective scan.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links anything here; only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.
The oracle shares no code with the CUDA path: the only common module is the
seeded input generator, which holds none of the method's arithmetic.

Contents
  ssd.py      sequential recurrence (numpy, float64), the definition, and
              its single-token step (the decode step with a carried state)
  linscan.py  sequential scalar scan and the affine pair combine (numpy, float64)
  ssm_oracle.c + native.py
              the same two definitions in plain C (float64, OpenMP over
              independent units) for full-size workloads and CPU timing

Every function is pinned by tests that do not reuse its formula: the chunked
closed form, causal linear attention, the D*x special case, exact rational
folds of the pair combine in every bracketing, closed forms, and planted
mistakes that the pins must reject (see tests/test_oracle_*.py).
"""
