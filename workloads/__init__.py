"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and by the oracle's tests."""

from .synthetic import *  # noqa: F401,F403
