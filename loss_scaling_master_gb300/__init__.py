"""GB300-native mixed-precision optimizer step: loss-scale unscale/check,
dynamic scale state machine, FP32-master AdamW with bf16 emission, and
tensorwise dynamic FP8 quantization with transposed copies.

The compute lives in libampfp8.so (hand-written CUDA for sm_103a, C ABI in
include/ampfp8.h); this package is its thin ctypes binding.
"""
from ._lib import (AmpError, TensorList, amp_abi_version, amp_adamw_master_step,
                   amp_adamw_master_step_clip, amp_adamw_master_step_fp8_delayed,
                   amp_adamw_master_step_sr, amp_emit_bf16, amp_selftest_bounded_wait,
                   amp_adamw_master_step_clip_sr, amp_adamw_master_step_fp8_delayed_sr,
                   fp8_quant_tensorwise_list_sr, amp_tensor_list_check,
                   amp_noalloc_check, amp_tensor_list_copy_from_host,
                   amp_tensor_list_copy_to_host, amp_read_state, amp_scale_health, ScalerState,
                   fp8_quant_groupwise,
                   amp_adamw_master_step_noalloc, amp_last_error, amp_update_scale_fp8_history,
                   amp_unscale_check_norm, amp_tensor_list_create, amp_tensor_list_destroy,
                   amp_tensor_list_set_amax_slots, amp_unscale_check, amp_update_scale,
                   fp8_quant_rowwise, fp8_quant_tensorwise, fp8_quant_tensorwise_list, load)
from .step import AmpOptimizerStep

__all__ = ["AmpError", "TensorList", "AmpOptimizerStep", "load", "amp_abi_version",
           "amp_last_error", "amp_tensor_list_create", "amp_tensor_list_destroy",
           "amp_tensor_list_set_amax_slots", "amp_unscale_check", "amp_adamw_master_step",
           "amp_adamw_master_step_noalloc", "amp_adamw_master_step_clip", "amp_emit_bf16",
           "amp_unscale_check_norm", "amp_adamw_master_step_fp8_delayed",
           "amp_adamw_master_step_sr", "amp_tensor_list_check", "amp_selftest_bounded_wait", "amp_noalloc_check",
           "amp_tensor_list_copy_from_host", "amp_tensor_list_copy_to_host", "amp_read_state",
           "amp_scale_health", "ScalerState", "fp8_quant_groupwise",
           "amp_update_scale_fp8_history",
           "fp8_quant_tensorwise", "fp8_quant_tensorwise_list", "fp8_quant_rowwise",
           "amp_update_scale", "amp_adamw_master_step_clip_sr",
           "amp_adamw_master_step_fp8_delayed_sr", "fp8_quant_tensorwise_list_sr"]
