"""GB300 (sm_103a) forward pass of chunkwise gated linear attention.

The compute lives in libgla.so (C ABI, include/gla.h); ``binding`` is the
ctypes layer over it with the same names. Importing this package does not
load the library; the first call does, and raises if it is not built.
"""
from .binding import (  # noqa: F401
    GLA_BF16, GLA_FP32, GLA_GATE_BILINEAR, GLA_GATE_HEAD_SCALAR, GLA_GATE_NONE, GLA_GATE_PER_KEY,
    GLA_GATE_TOKEN_SCALAR,
    GLA_PATH_AUTO, GLA_PATH_FUSED, GLA_PATH_SIMT, GLA_PATH_SPLIT, GLA_PATH_STAGED, GLA_PATH_TENSOR, GlaError,
    backward, forward, gla_bwd,
    gla_bwd_num_stages, gla_bwd_stage, gla_bwd_stage_name, gla_bwd_workspace_size, gla_device_status,
    gla_fwd, gla_fwd_ex, gla_fwd_host, gla_fwd_num_stages, gla_fwd_stage, gla_fwd_stage_name,
    gla_fwd_workspace_size, gla_host_release, gla_pair_combine, gla_pair_scan, gla_segment_pair,
    gla_segment_pair_workspace_size, gla_status_string, gla_version, make_params, pair_combine, pair_scan,
    segment_pair,
)
from .autograd import gla_attention  # noqa: F401,E402
