"""GB300-native AttnRes depth-wise aggregation (Full and Block AttnRes).

The compute lives in ``libattnres.so`` (hand-written CUDA for sm_103a, C ABI
declared in ``include/attnres.h``); ``binding`` exposes its entry points to
Python under the same names.
"""
from .binding import (  # noqa: F401
    AttnResError,
    attnres_abi_version,
    attnres_block_bwd,
    attnres_block_bwd_scratch_floats,
    attnres_block_merge,
    attnres_block_merge_prenorm,
    attnres_block_pass,
    attnres_block_stage1,
    attnres_block_summary_accumulate,
    attnres_device_status,
    attnres_full_bwd,
    attnres_full_fwd,
    attnres_full_fwd_dynq,
    attnres_full_fwd_prenorm,
    attnres_full_pass,
    attnres_full_pass_prenorm,
    attnres_kernel_path,
    attnres_query_projection,
    attnres_rmsnorm,
    attnres_stage1_dsplit_finish,
    attnres_stage1_dsplit_partials,
    attnres_status_string,
    lib,
)
