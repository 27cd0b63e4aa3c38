"""Varlen block-diagonal causal attention for isolated sequence packing (GB300, sm_103a).

The compute path is the C-ABI library ``lib/libvlc.so`` (CUDA kernels for
sm_103a, declared in ``include/vlc.h``); ``binding`` marshals torch tensors to
it.  ``synth`` draws the seeded synthetic workloads used by tests and bench.
``shifted_cross_entropy`` is the next step after attention on the pages'
pipeline: loss sum and target count over the pre-shifted labels.
"""
from .binding import (  # noqa: F401
    VlcError,
    build_positions_labels,
    build_worklist,
    get_error,
    load_library,
    new_workspace,
    shifted_cross_entropy,
    varlen_attn_bwd,
    varlen_attn_fwd,
    workspace_bytes,
)
