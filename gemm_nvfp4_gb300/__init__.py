"""NVFP4 weights x bf16 activations on GB300 (sm_103a).

The compute path is the C-ABI library libnvfp4.so (include/nvfp4.h), built from
``gemm_nvfp4_gb300/csrc`` by ``gemm_nvfp4_gb300.build``.  This package only
marshals PyTorch tensors into that ABI (``binding``) and provides seeded
synthetic inputs (``inputs``).  There is no CPU fallback: if the library is
missing, every call raises.
"""
from .binding import (NVFP4_ERR_DEVICE_TIMEOUT, NVFP4_OK, NVFP4_STATUS_WORD_OFFSET,
                      NVFP4_OP_FP6_GATEUP_SWIGLU, NVFP4_OP_FP6_GEMM, NVFP4_OP_GATEUP_SWIGLU,
                      NVFP4_OP_GEMM_PREFILL, NVFP4_OP_GEMV_SKINNY, NVFP4_OP_QUANTIZE, NVFP4_OUT_BF16,
                      NVFP4_OUT_F32, FP6Weight, NVFP4Error, NVFP4Weight, nvfp4_fp6_gateup_swiglu,
                      nvfp4_device_status, nvfp4_fp6_gemm, nvfp4_fp6_quantize, nvfp4_fp6_quantize_bf16,
                      header_functions, library_path, load_library, nvfp4_gateup_swiglu,
                      nvfp4_blocked_scale_bytes, nvfp4_gemm_prefill, nvfp4_gemv_skinny,
                      nvfp4_gemv_skinny_noalloc, nvfp4_import_blocked_scales, nvfp4_noalloc_selftest_wait_timeout,
                      nvfp4_noalloc_status, SkinnyJob, StreamPlan, nvfp4_stream_plan, nvfp4_stream_plan_bytes,
                      nvfp4_stream_run, nvfp4_quantize,
                      nvfp4_quantize_bf16, nvfp4_selftest_wait_timeout, nvfp4_status_string, nvfp4_version,
                      nvfp4_workspace_bytes)

__all__ = [
    "NVFP4Error", "NVFP4Weight", "FP6Weight",
    "nvfp4_fp6_quantize", "nvfp4_fp6_quantize_bf16", "nvfp4_fp6_gemm", "nvfp4_fp6_gateup_swiglu",
    "NVFP4_OP_FP6_GEMM", "NVFP4_OP_FP6_GATEUP_SWIGLU", "header_functions", "library_path", "load_library",
    "nvfp4_gateup_swiglu", "nvfp4_gemm_prefill", "nvfp4_gemv_skinny", "nvfp4_gemv_skinny_noalloc",
    "nvfp4_quantize", "nvfp4_quantize_bf16", "nvfp4_blocked_scale_bytes", "nvfp4_import_blocked_scales",
    "nvfp4_status_string", "nvfp4_version", "nvfp4_workspace_bytes",
    "NVFP4_OP_QUANTIZE", "NVFP4_OP_GEMV_SKINNY", "NVFP4_OP_GATEUP_SWIGLU", "NVFP4_OP_GEMM_PREFILL",
    "NVFP4_OUT_F32", "NVFP4_OUT_BF16",
    "nvfp4_device_status", "nvfp4_selftest_wait_timeout", "NVFP4_OK", "NVFP4_ERR_DEVICE_TIMEOUT",
    "NVFP4_STATUS_WORD_OFFSET", "nvfp4_noalloc_status", "nvfp4_noalloc_selftest_wait_timeout",
    "SkinnyJob", "StreamPlan", "nvfp4_stream_plan", "nvfp4_stream_plan_bytes", "nvfp4_stream_run",
]
