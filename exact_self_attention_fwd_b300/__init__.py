"""Exact self-attention forward for B300 (sm_103a): a thin Python binding over the
C-ABI library libattn_fwd.so (include/attn_api.h). PyTorch supplies device memory
and streams; the attention itself runs only in the library's CUDA kernel.
"""
from ._lib import (ATTN_ERR_ALIGN, ATTN_ERR_BOUNDS, ATTN_ERR_CUDA, ATTN_ERR_NULLPTR, ATTN_ERR_SCRATCH_LIMIT,
                   ATTN_ERR_SHAPE, ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE,
                   ATTN_OK, DEBUG_LIB_PATH, AttnError,
                   attn_bwd, attn_fwd, attn_fwd_decode, attn_fwd_fp8, attn_fwd_host, bwd_row_sums,
                   bwd_workspace_size, decode_workspace_size,
                   device_error, header_functions, load, quantize_e4m3, quantize_e4m3_hadamard, selftest_wait_timeout,
                   sign_masks,
                   status_str, using, version)

__all__ = [
    "ATTN_OK", "ATTN_ERR_NULLPTR", "ATTN_ERR_ALIGN", "ATTN_ERR_SHAPE", "ATTN_ERR_UNSUPPORTED",
    "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_ERR_WORKSPACE", "ATTN_ERR_SCRATCH_LIMIT", "ATTN_ERR_BOUNDS",
    "DEBUG_LIB_PATH", "using",
    "AttnError", "attn_bwd", "attn_fwd", "bwd_row_sums", "bwd_workspace_size",
    "attn_fwd_decode", "attn_fwd_fp8", "attn_fwd_host", "decode_workspace_size", "device_error",
    "header_functions", "quantize_e4m3", "quantize_e4m3_hadamard", "sign_masks",
    "load", "selftest_wait_timeout", "status_str", "version",
]
