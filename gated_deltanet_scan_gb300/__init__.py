"""Gated delta rule on GB300 (sm_103a)."""
