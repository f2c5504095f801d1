"""Mamba2 recurrent-state update over a slot pool, for one GB300 (sm_103a)."""
