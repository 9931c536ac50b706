"""Deterministic selected-token log-probability over a tiled vocabulary (GB300, sm_103a)."""
