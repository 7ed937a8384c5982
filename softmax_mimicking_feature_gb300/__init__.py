"""Hedgehog / Taylor causal linear attention for GB300 (sm_103a)."""
