"""Seeded synthetic workloads (inputs only; no verification or scheduling arithmetic)."""
