"""CPU oracle for sink-aware varlen attention (forward).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``, and by
nothing else.  The CUDA library never imports, links or calls anything here,
and nothing here calls the CUDA library.

Two independent forms of the same definition:

* :mod:`oracle.sa_oracle` -- the set-enumerating form in plain C (fp64,
  OpenMP over rows), fast enough for full-size sampled rows and timed as the
  CPU baseline;
* :mod:`oracle.brute` -- a dense NumPy form (a full logit matrix with a mask),
  for tiny inputs only.
"""
