"""Varlen block-diagonal causal attention for isolated sequence packing (GB300, sm_103a).

The compute path is the C-ABI library ``lib/libvlc.so`` (CUDA kernels for
sm_103a, declared in ``include/vlc.h``); ``binding`` marshals torch tensors to
it.  ``synth`` draws the seeded synthetic workloads used by tests and bench.
"""
from .binding import (  # noqa: F401
    VlcError,
    build_positions_labels,
    build_worklist,
    get_error,
    load_library,
    new_workspace,
    varlen_attn_bwd,
    varlen_attn_fwd,
    workspace_bytes,
)
