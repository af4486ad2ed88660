"""dense_fp32_matrix_strict_gb300 — strict-FP32 SGEMM for GB300 (sm_103a).

C = alpha * A @ B + beta * C on row-major float32 matrices, computed by
hand-written FFMA kernels behind the C ABI in ``include/sgemm.h``. This
package is the thin Python binding over that library (``_binding``), its
build step (``build``) and the seeded synthetic inputs used to test and
measure it (``inputs``). PyTorch serves only for device memory and streams.
"""
from ._binding import (  # noqa: F401
    EXPORTED_SYMBOLS, SGEMM_ERR_CUDA, SGEMM_ERR_DEVICE_CHECK, SGEMM_ERR_DEVICE_TIMEOUT, SGEMM_ERR_INVALID_VALUE,
    SGEMM_ERR_LAUNCH, SGEMM_ERR_UNSUPPORTED_DEVICE, SGEMM_OK, SgemmError, check_status,
    fp32_peak, library_path, load, plan_tensors, sgemm, sgemm_check_status, sgemm_error_string,
    sgemm_config_names, sgemm_fp32_peak, sgemm_last_cuda_error, sgemm_noalloc, sgemm_plan, sgemm_selftest_wait_timeout,
    SGEMM_OP_N, SGEMM_OP_T, sgemm_ex, sgemm_plan_ex, sgemm_3xtf32_ex, sgemm_host,
    sgemm_host_tensors, sgemm_noalloc_check_status, sgemm_fp32_peak_ex, SGEMM_PEAK_FFMA,
    SGEMM_PEAK_FFMA2, SGEMM_PEAK_OUTER, sgemm_null_launch, sgemm_tf32_mma_peak, sgemm_selftest_occupy,
    sgemm_set_config, sgemm_set_shape_config, sgemm_clear_shape_configs, sgemm_set_wait_timeout_ns, sgemm_tensors, sgemm_3xtf32, sgemm_3xtf32_tensors,
)
