"""Fused residual-add + normalization for GB300 (sm_103a)."""
