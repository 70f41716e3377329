"""Mamba-2 SSD chunked forward pass on GB300 (sm_103a)."""
