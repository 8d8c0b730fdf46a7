"""Paged grouped-query decode attention for GB300 (sm_103a)."""
