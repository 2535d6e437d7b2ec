"""GB300-native tiled FP32 matrix multiply C = A.B (sm_103a CUDA, C ABI).

``sgemm(A, B)`` multiplies CUDA float32 tensors through the C-ABI library
``libsgemm_f32.so`` (built by ``dense_fp32_tiled_gb300.build.build()``);
``sgemm_f32(...)`` is the raw C call on device addresses.  ``sgemm_host(A, B)``
takes CPU tensors (``sgemm_f32_host``: copies overlapped with the product).  ``transpose(x)`` /
``transpose_f32(...)`` run the FP32 transpose, the pages' second workload.
``copy_timeouts()``, ``tc_timeouts()`` and ``wait_selftest(case)`` expose the
bounded waits' failure reporting; ``bank_stride_probe(stride)`` measures the
bank page's stride law on the GPU.
"""
from ._binding import (SGEMM_OK, WAIT_SELFTESTS, SgemmError, bank_pattern_probe, bank_stride_probe, copy_timeouts, declared_functions, host_workspace_size,
                       load_library, sgemm, sgemm_f32, sgemm_f32_3xtf32, sgemm_f32_host, sgemm_host,
                       sgemm_f32_static_scratch, sgemm_f32_ws, sgemm_tc, smem_request, smem_shape, status_string,
                       tc_timeouts, tc_workspace_size, transpose, transpose_f32, transpose_smem_request,
                       transpose_status_string, wait_selftest, workspace_size, workspace_size_for,
                       ws_schedule)

__all__ = ["SGEMM_OK", "WAIT_SELFTESTS", "SgemmError", "bank_pattern_probe", "bank_stride_probe", "copy_timeouts", "declared_functions", "host_workspace_size",
           "load_library", "sgemm", "sgemm_f32", "sgemm_f32_3xtf32", "sgemm_f32_host", "sgemm_host",
           "sgemm_tc", "tc_timeouts", "tc_workspace_size",
           "sgemm_f32_static_scratch", "sgemm_f32_ws", "smem_request", "smem_shape", "status_string",
           "transpose", "transpose_f32", "transpose_smem_request", "transpose_status_string", "wait_selftest",
           "workspace_size", "workspace_size_for", "ws_schedule"]
