"""Packed gated-delta-rule (GDN) prefill for GB300 (sm_103a)."""
