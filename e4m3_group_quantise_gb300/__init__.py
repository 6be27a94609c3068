"""jetfp8 for GB300: group-wise FP8-E4M3 quantisation and block-scaled FP8
GEMMs (Fprop, Dgrad, Wgrad) of a linear layer, one kernel set for rollout
and training.  See ``include/jetfp8.h`` for the C-ABI."""
from .jetfp8 import (  # noqa: F401
    Jetfp8Error,
    declared_functions,
    gemm_dgrad,
    gemm_fprop,
    gemm_wgrad,
    jetfp8_act_scale_count,
    jetfp8_e4m3_encode_range,
    jetfp8_gemm_dgrad,
    jetfp8_gemm_fprop,
    jetfp8_gemm_wgrad,
    jetfp8_poll_device_error,
    jetfp8_quantize_act,
    jetfp8_quantize_act_dual,
    jetfp8_quantize_act_transposed,
    jetfp8_quantize_weight,
    jetfp8_quantize_weight_group,
    jetfp8_rmsnorm_quantize_act,
    jetfp8_swiglu_quantize_act,
    jetfp8_status_string,
    jetfp8_watchdog_selftest,
    load_library,
    quantize_act,
    quantize_act_dual,
    quantize_act_transposed,
    quantize_weight,
    quantize_weights,
    rmsnorm_quantize_act,
    swiglu_quantize_act,
)
from .linear import FP8Linear, FP8LinearFunction, QuantizedWeight  # noqa: F401
