"""GB300-native fused attention forward (sm_103a).

The compute path is the C-ABI library ``libfa_gb300.so`` built from ``csrc/``;
``fa.py`` is its thin ctypes binding.  Importing this package does not load
the library; the first call into ``fa`` does, and fails loudly if it is
missing.
"""
