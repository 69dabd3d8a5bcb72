"""GB300-native Float8 training linear with dynamic tensorwise scaling.

The compute path is libf8 (hand-written sm_103a CUDA behind the C ABI of
include/f8.h); ``binding`` marshals torch tensors into it.  ``workloads``
draws the seeded synthetic inputs.
"""
from .binding import (EXPORTS, F8_E4M3, F8_E5M2, F8Error, LinearSaved, f8_amax, f8_cast_transpose, f8_gemm,  # noqa: F401
                      f8_gemm_grouped, f8_last_device_status, f8_linear_bwd, f8_linear_fwd,
                      f8_linear_workspace_bytes, f8_quantize, f8_quantize_workspace_bytes,
                      f8_quantize_swiglu, f8_linear_fwd_swiglu, f8_linear_fwd_w13_swiglu,
                      f8_gemm_w13_swiglu, interleave_w13, split_ab, f8_linear_fwd_noalloc,
                      f8_linear_bwd_w13_swiglu, f8_quantize_swiglu_bwd, f8_kernel_launches,
                      f8_selftest_bounds, f8_quantize_multi, f8_quantize_multi_workspace_bytes,
                      f8_linear_fwd_group, f8_linear_bwd_group, f8_linear_group_workspace_bytes,
                      group_saved, group_workspace, f8_transpose_u8, f8_linear_fwd_qw,
                      f8_linear_fwd_qw_workspace_bytes,
                      f8_selftest_wait_timeout,
                      f8_set_wait_limit_ns, f8_status_string, lib, workspace)
