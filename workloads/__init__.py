"""Seeded synthetic inputs shared by the checker and the GPU path (no attention arithmetic)."""
