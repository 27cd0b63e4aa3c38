"""Varlen block-diagonal causal attention for isolated sequence packing (GB300, sm_103a).

The compute path is the C-ABI library ``lib/libvlc.so`` (CUDA kernels for
sm_103a, declared in ``include/vlc.h``); ``binding`` marshals torch tensors to
it.  ``synth`` draws the seeded synthetic workloads used by tests and bench.
``shifted_cross_entropy`` is the next step after attention on the pages'
pipeline: loss sum and target count over the pre-shifted labels; ``pack`` and
``shard_packs`` are the host step before it (windows by first-fit decreasing,
windows to ranks by sum of squared lengths); ``cp_partition``, ``cp_block_mode``,
``rope_pos`` and ``lse_merge`` split long segments over a context-parallel group.
``varlen_attn_fwd_rot`` is the forward with RoPE in the kernel that also returns the rotated
q', k' for a training step's backward.
"""
from .binding import (  # noqa: F401
    Packing,
    VlcError,
    build_positions_labels,
    build_worklist,
    cp_block_mode,
    cp_partition,
    get_error,
    load_library,
    lse_merge,
    new_workspace,
    pack,
    rope_pos,
    rope_qk,
    set_wait_limit_us,
    shard_packs,
    shifted_cross_entropy,
    sum_parts,
    varlen_attn_bwd,
    varlen_attn_fwd,
    varlen_attn_fwd_rot,
    workspace_bytes,
)
