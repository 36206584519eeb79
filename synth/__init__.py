"""Seeded synthetic inputs shared by the oracle and the CUDA path (no MoE arithmetic here)."""
