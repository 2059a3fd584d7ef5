"""Seeded synthetic inputs (random numbers and bf16 rounding only; no attention arithmetic)."""
from . import inputs, configs  # noqa: F401
