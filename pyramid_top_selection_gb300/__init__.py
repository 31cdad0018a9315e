"""PISA pyramid Top-K block selection + causal block-sparse attention for GB300 (sm_103a).

The compute runs in libpisa.so (hand-written CUDA kernels behind a C ABI, see
include/pisa.h); this package is its thin Python binding.
"""
from ._pisa import (  # noqa: F401
    DecodeShape, PisaError, Shape, build_pyramid, decode_build_pyramid, decode_pyramid_layout,
    decode_step, default_scale, lib, make_decode_shape, make_shape, profile_read, profile_start,
    profile_stop, pyramid_layout, select, select_mean, select_meanvar, workspace,
    select_flat, shape_of, sparse_attn_bwd, sparse_attn_fwd, workspace_size,
    STATUS_POS_RANGE, STATUS_TIMEOUT, check_status, set_test_stall, set_wait_limit, workspace_status,
)
