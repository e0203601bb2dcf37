"""Structured-sparse weight GEMM (2:4, tile-wise, tile-vector-wise) for GB300.

The compute lives in the C-ABI library ``libssdnn.so`` built from ``csrc/``;
``ssdnn`` is its thin ctypes binding. Importing the package does not load the
library: ``structured_sparse_dnn_gb300.ssdnn`` does, and raises if it is absent.
"""
