"""SiTU-GLU expert feed-forward on GB300 (sm_103a).

Hand-written CUDA kernels behind a C ABI (``include/situ.h``, ``libsitu.so``):
  * ``situ_glu_act``              standalone activation (memory bound)
  * ``situ_ffn_forward``          dense FFN: tcgen05 gate_up GEMM with the
                                  activation in its epilogue, tcgen05 down GEMM
  * ``situ_ffn_forward_train`` / ``situ_ffn_backward``   dense training step
  * ``situ_moe_build_index``      stable expert index of routed tokens
  * ``situ_moe_grouped_forward``  the FFN grouped over experts
  * ``situ_moe_grouped_forward_train`` / ``situ_moe_grouped_backward``
                                  grouped training step
  * ``situ_moe_combine``          router-weighted combine (deterministic)
  * ``situ_moe_grouped_forward_combined``  the layer output with the combine fused
                                  into the down projection (FP32 scatter-add)
  * ``mx_quantize_act`` / ``mx_quantize_weights``, ``situ_ffn_forward_mxfp8``,
    ``situ_moe_grouped_forward_mxfp8``   MX experts: MXFP8 activations, MXFP8 or
                                          MXFP4 weights (block-scaled tensor cores)
This package is the thin PyTorch binding over that ABI.
"""
from .api import (MX_DOWN, MX_E2M1, MX_E4M3, MX_GATE_UP, MxWeights, SituError,
                  moe_combined_workspace_bytes, situ_moe_grouped_forward_combined, ffn_mxfp8_workspace_bytes,
                  moe_mxfp8_workspace_bytes, mx_act_scales_bytes, mx_quantize_act,
                  mx_quantize_weights, mx_weight_scales_bytes, situ_ffn_forward_mxfp8,
                  situ_ffn_gate_up_mxfp8, situ_moe_grouped_forward_mxfp8, device_status, ffn_backward_workspace_bytes,
                  ffn_last_path, FFN_PATH_FUSED, FFN_PATH_TWO_LAUNCHES, ffn_set_single_launch,
                  moe_set_kgrouped_two_cta,
                  ffn_host_workspace_bytes, ffn_workspace_bytes, moe_backward_workspace_bytes,
                  moe_workspace_bytes, selftest_bounded_wait, selftest_group_maps, set_wait_limit_ns,
                  situ_ffn_backward, situ_ffn_down,
                  situ_ffn_forward, situ_ffn_forward_host, situ_ffn_forward_train,
                  situ_ffn_gate_up, situ_glu_act, situ_moe_build_index, situ_moe_combine,
                  situ_moe_grouped_backward, situ_moe_grouped_forward,
                  situ_moe_grouped_forward_train)

__all__ = [
    "SituError", "situ_glu_act", "situ_ffn_forward", "situ_ffn_forward_host", "situ_ffn_gate_up",
    "situ_ffn_down",
    "situ_moe_build_index",
    "situ_moe_grouped_forward", "ffn_workspace_bytes", "moe_workspace_bytes",
    "device_status", "selftest_bounded_wait", "selftest_group_maps", "set_wait_limit_ns", "ffn_host_workspace_bytes",
    "situ_moe_combine",
    "ffn_last_path", "FFN_PATH_FUSED", "FFN_PATH_TWO_LAUNCHES", "ffn_set_single_launch",
    "moe_set_kgrouped_two_cta",
    "situ_ffn_forward_train", "situ_ffn_backward", "ffn_backward_workspace_bytes",
    "situ_moe_grouped_forward_train", "situ_moe_grouped_backward", "moe_backward_workspace_bytes",
    "situ_moe_grouped_forward_combined", "moe_combined_workspace_bytes",
    "MX_GATE_UP", "MX_DOWN", "MX_E4M3", "MX_E2M1", "MxWeights", "mx_act_scales_bytes", "mx_weight_scales_bytes", "mx_quantize_act",
    "mx_quantize_weights", "situ_ffn_gate_up_mxfp8", "situ_ffn_forward_mxfp8",
    "ffn_mxfp8_workspace_bytes", "situ_moe_grouped_forward_mxfp8", "moe_mxfp8_workspace_bytes",
]
