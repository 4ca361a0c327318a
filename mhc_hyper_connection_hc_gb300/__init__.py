"""GB300-native (sm_103a) mHC site program: a C-ABI CUDA library plus a thin ctypes binding.

Importing the package loads nothing; `mhc_hyper_connection_hc_gb300.hc` opens the
CUDA library on first use and raises if it is missing.
"""
