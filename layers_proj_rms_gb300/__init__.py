"""mHC residual-stream ops on GB300: Python binding of libmhc.

Every function here has the name of a libmhc C entry point and only
marshals arguments: it checks dtypes, shapes and contiguity of the torch
tensors it is given, passes their device pointers and the current CUDA
stream to the library, and raises MhcError on a nonzero status.  All
computation runs in the library's CUDA kernels; there is no other path.
The first use of any of them loads libmhc.so and raises ImportError if it
has not been built (``python -m layers_proj_rms_gb300.build``).

Tensor conventions (see include/mhc.h): x [T, n, C] bf16, W [n*C, O] fp32,
alpha3 [3] fp32, b [O] fp32, H_pre/H_post [T, n] fp32, H_res [T, n, n] fp32,
u_save [T, O] fp32, r_save [T] fp32, with O = n*n + 2*n.  Outputs are
passed in preallocated; the library writes every element.
"""
from __future__ import annotations

__all__ = [
    "MhcError", "lib", "lib_path", "workspace", "mhc_version", "mhc_workspace_bytes",
    "mhc_device_error", "mhc_sinkhorn_fwd", "mhc_sinkhorn_bwd", "mhc_proj_rms_compute_h_fwd",
    "mhc_proj_rms_compute_h_bwd", "mhc_h_aggregate_fwd", "mhc_h_aggregate_bwd",
    "mhc_h_post_bda_fwd", "mhc_h_post_bda_bwd", "rmsnorm_fwd", "rmsnorm_bwd", "mhc_layer_fwd",
    "mhc_layer_bwd", "OP_PROJ_RMS_COMPUTE_H_FWD", "OP_PROJ_RMS_COMPUTE_H_BWD",
    "OP_H_POST_BDA_BWD", "OP_LAYER_FWD", "OP_LAYER_BWD", "mhc_proj_rms_compute_h_fwd_noalloc",
    "mhc_h_aggregate_static_fwd", "mhc_h_aggregate_static_bwd", "rmsnorm_residual_fwd",
    "rmsnorm_residual_bwd", "mhc_h_aggregate_rmsnorm_fwd", "mhc_h_aggregate_rmsnorm_bwd",
    "mhc_proj_rms_partial_fwd", "mhc_compute_h_fwd", "mhc_compute_h_bwd",
    "mhc_proj_rms_partial_bwd", "OP_RMSNORM_RESIDUAL_BWD", "OP_H_AGGREGATE_RMSNORM_BWD",
    "OP_H_AGGREGATE_STATIC_BWD", "OP_PROJ_RMS_PARTIAL_FWD", "OP_COMPUTE_H_BWD",
    "OP_PROJ_RMS_PARTIAL_BWD", "mhc_set_batch_invariant", "mhc_batch_invariant",
    "mhc_set_pinned_reductions", "mhc_pinned_reductions",
    "mhc_h_post_bda_compute_h_fwd", "OP_H_POST_BDA_COMPUTE_H_FWD", "mhc_selftest_wait_timeout",
]


def __getattr__(name):
    if name in __all__:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
