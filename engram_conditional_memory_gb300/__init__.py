"""Engram conditional memory, GB300-native (sm_103a): the hash-gather and context-aware-gate hot path.

The compute lives in the CUDA library ``_build/libengram_gb300.so`` (C ABI in
include/engram.h); this package is its thin binding.  Build it with
``build.build()`` (``__graft_entry__.build()`` at the repository root).
"""
from .binding import (  # noqa: F401
    BF16,
    DEVERR_COMPRESSED,
    DEVERR_SEQ_OFFSETS,
    DEVERR_TIMEOUT,
    DEVERR_TOKEN_ID,
    F32,
    EngramError,
    HashSpec,
    abi_version,
    check_wait_timeout,
    device_status,
    fuse_weight,
    gate_bwd,
    gate_bwd_reduce_noalloc,
    gate_bwd_num_partials,
    gate_fwd,
    gate_fwd_rms,
    gate_hc_bwd,
    gate_hc_fwd,
    grad_w_reduce,
    hash_gather,
    library_path,
    load_library,
    read_error_word,
    set_max_ctas,
    set_pdl,
    set_validation,
    short_conv_bwd,
    short_conv_fwd,
    short_conv_grad_reduce,
    short_conv_num_partials,
    sinkhorn_finalize,
    sinkhorn_momentum_update,
    sinkhorn_num_partials,
    sinkhorn_step,
    sinkhorn_step_reduce,
)
