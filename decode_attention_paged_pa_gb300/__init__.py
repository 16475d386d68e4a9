"""GB300-native paged decode attention (PagedAttention V2), single- and multi-query.

The computation lives in hand-written CUDA kernels for sm_103a behind a C ABI
(``include/pa_decode.h``, built into ``_build/libpa_decode.so``); this package
is its thin Python binding plus the seeded synthetic workloads used by the
tests and the bench.  The library is loaded lazily on the first call.
"""
from .binding import (  # noqa: F401
    PA_DTYPE_BF16, PA_DTYPE_FP16, PA_DTYPE_FP32, PA_ERR_CUDA, PA_ERR_DEVICE_BOUNDS, PA_ERR_INVALID_ARG,
    PA_ERR_TIMEOUT, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_OK, PA_VARIANT_AUTO, PA_VARIANT_MMA,
    PA_VARIANT_SIMT, PaError, device_status, host_io_workspace_bytes, pa_decode_v2,
    pa_decode_v2_fp8, pa_decode_v2_host_io, pa_decode_v2_mq, pa_decode_v2_mq_fp8, status_string,
    workspace_bytes, workspace_layout)
