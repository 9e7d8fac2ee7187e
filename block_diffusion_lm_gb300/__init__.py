"""GB300-native two-copy block-diffusion attention (CSBP per-rank math).

The compute path is the C-ABI library ``libcsbp.so`` built from ``csrc/``
(sm_103a kernels); ``csbp`` is its thin ctypes binding.  ``inputs`` draws the
seeded synthetic workloads.
"""
