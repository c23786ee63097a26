"""GB300-native incremental (single-query decode) flash attention.

``kv_cache_incremental_split_gb300.ifa`` is the Python binding of the C-ABI
library ``libifa.so`` (built from ``csrc/``); ``inputs`` holds the seeded
synthetic input generators.  Importing the package loads nothing: the CUDA
library is opened on first use of the binding.
"""
