"""int8 paged-KV attention decode for NVIDIA GB300 (sm_103a).

The product is the C-ABI library ``libpa_q8.so`` (declared in
include/pa_q8.h, built by ``python -m int8_paged_kv_gb300.build``).  This
package holds its CUDA sources (``csrc/``), the build step, a ctypes binding
with the same function names (``pa_q8_*``) and the seeded synthetic
workloads (``workloads``).  Importing the package loads nothing; the first
binding call loads the library and fails loudly if it is missing.
"""
_BINDING_NAMES = {
    "pa_q8_reshape_and_cache", "pa_q8_decode", "pa_q8_decode_workspace_size", "pa_q8_decode_plan",
    "pa_q8_decode_rows", "pa_q8_decode_rows_workspace_size", "pa_q8_decode_append",
    "pa_f32_reshape_and_cache", "pa_f32_decode", "pa_f32_decode_workspace_size",
    "pa_q8c_cache_words", "pa_q8c_append", "pa_q8c_decode", "pa_q8c_decode_workspace_size",
    "pa_q8_device_status", "pa_q8_selftest_wait_timeout", "pa_q8_status_string", "pa_q8_version",
    "PaQ8Error", "lib", "LIB_PATH", "PA_Q8_KERNEL_AUTO", "PA_Q8_KERNEL_CUDA_CORE",
    "PA_Q8_KERNEL_TENSOR_CORE", "PA_Q8_KERNEL_TCGEN05", "PA_Q8_DEV_BAD_BLOCK", "PA_Q8_DEV_BAD_SLOT",
    "PA_Q8_DEV_WAIT_TIMEOUT", "header_functions",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
