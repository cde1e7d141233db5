"""GB300 (sm_103a) library for the prefix-cached flow-matching action expert.

The compute lives in libvla.so (include/vla.h); this package is its thin
Python binding plus the in-tree build step.
"""
from .binding import (DTYPE_BF16, DTYPE_F32, EXPORTED, FLAG_ATTN_SPLIT, FLAG_ATTN_STREAM, FLAG_NO_GRAPH,  # noqa: F401
                      FLAG_LINEAR_SPLIT, FLAG_LINEAR_WIDE, FLAG_PERSIST, FLAG_SIMT_GEMM, LIB_PATH, Expert,
                      VlaError, gelu_forms, lib, noise_fill, quantize_rows, ternary_gemm, upload_weights)
