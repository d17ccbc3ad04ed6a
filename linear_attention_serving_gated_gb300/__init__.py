"""KDA (Kimi Delta Attention) gated delta-rule serving path for one GB300.

The compute lives in ``libkda.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/kda.h``).  ``kda`` is the thin ctypes binding with the
same entry-point names; ``inputs`` draws the seeded synthetic workloads.
Importing the package loads nothing; the first call into ``kda`` loads the
library and raises if it is missing.
"""
