"""Complex SSD (complex-valued diagonal state space) forward and decode step on GB300.

The compute lives in ``libcssd.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/cssd.h``); ``complex_valued_state_gb300.cssd`` is
the thin ctypes binding.  ``workloads`` draws the seeded synthetic inputs.
Importing the package does not load the CUDA library.
"""

__all__ = ["workloads", "cssd"]
