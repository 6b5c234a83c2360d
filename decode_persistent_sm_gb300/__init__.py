"""GB300 (sm_103a) batch-1 decode engine for the lane-structured decoder.

The engine is the C-ABI library ``liblaneformer.so`` (include/laneformer.h);
this package is a thin ctypes binding with the same call names.  Every step of
the decode runs in the library's CUDA kernels.  There is no fallback: if the
library has not been built, importing the binding raises.
"""
from .binding import (Engine, LfConfig, LaneformerError, STATUS, config_from_shape,
                      library_path, load_library, matmul_f16, matmul_add_f16, matmul_f16_async, gemv_f16,
                      sample_token, stream_read)

__all__ = ["Engine", "LfConfig", "LaneformerError", "STATUS", "config_from_shape",
           "library_path", "load_library", "matmul_f16", "matmul_add_f16", "matmul_f16_async", "gemv_f16",
           "sample_token", "stream_read"]
