"""Exact IO-aware tiled attention for GB300 (sm_103a)."""
