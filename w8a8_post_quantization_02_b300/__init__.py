"""SmoothQuant W8A8 linear-layer hot path for B300 (sm_103a)."""
