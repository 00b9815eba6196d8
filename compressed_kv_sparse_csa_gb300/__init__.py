"""GB300-native (sm_103a) compressed-KV sparse-attention (CSA) decode path.

The compute lives in libds4x.so (hand-written CUDA behind the C ABI in
include/ds4x.h); ``compressed_kv_sparse_csa_gb300.binding`` is a thin ctypes
layer over it.  Build with ``compressed_kv_sparse_csa_gb300.build.build()``.
Importing the package itself needs neither torch nor the built library.
"""

KV_ROW_BYTES = 583
IDX_ROW_BYTES = 68
