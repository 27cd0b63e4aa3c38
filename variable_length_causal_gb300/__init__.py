"""Varlen block-diagonal causal attention for isolated sequence packing (GB300, sm_103a)."""
