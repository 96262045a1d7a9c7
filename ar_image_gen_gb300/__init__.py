"""Diagonal-aware sparse decode attention for GB300 (sm_103a).

The decode path lives in the CUDA library built from ``csrc/`` and is called
through ``ar_image_gen_gb300.dsa`` (a thin ctypes binding over its C ABI).
Importing this package does not load the library; ``dsa`` does, and fails
loudly if it is missing.
"""
