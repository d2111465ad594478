"""Seeded synthetic workloads (inputs only; no step of the method)."""
from .gen import *  # noqa: F401,F403
