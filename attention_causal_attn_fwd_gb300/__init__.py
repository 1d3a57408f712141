"""PaTH causal attention forward and decode on GB300 (sm_103a)."""
