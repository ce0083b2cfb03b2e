"""GB300 (sm_103a) W8A8 / W4A8 quantized linear layer.

The compute lives in libw8a8.so (hand-written CUDA behind a C ABI declared in
include/w8a8.h); ``binding`` marshals torch tensors to it.  ``synth`` holds
the seeded input generators.
"""
from .binding import (W8A8Error, linear, linear_noalloc, load, pack_weight_int4, quantize_act_per_token,
                      quantize_act_per_token_h, quantize_weight_int8, w4a8_gemm,
                      w8a8_check_status, w8a8_gemm, w8a8_gemm_h, w8a8_gemm_i32,
                      w8a8_is_available, w8a8_linear_workspace_bytes, w8a8_mv,
                      w8a8_status_string, w8a8_test_set_fault, weight_only_gemm)

__all__ = ["W8A8Error", "linear", "linear_noalloc", "load", "pack_weight_int4", "quantize_act_per_token",
           "quantize_act_per_token_h", "w8a8_gemm_h", "quantize_weight_int8", "w4a8_gemm", "w8a8_check_status", "w8a8_gemm",
           "w8a8_gemm_i32", "w8a8_is_available", "w8a8_linear_workspace_bytes", "w8a8_mv",
           "w8a8_status_string", "w8a8_test_set_fault", "weight_only_gemm"]
