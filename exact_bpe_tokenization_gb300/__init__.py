"""Exact full-context BPE tokenization on GB300 (sm_103a).

The product is a C-ABI shared library (include/toktier.h) built from the CUDA
sources in csrc/; `binding` is a thin ctypes layer with the same names.
`synth` holds the seeded input generators used by the tests and the benchmark.
"""
