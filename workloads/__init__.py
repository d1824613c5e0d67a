"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the
benchmark.  This package draws random numbers and lays them out; it holds
none of the indexer's arithmetic (no compression, scoring, selection or slot
translation)."""
from .synth import *  # noqa: F401,F403
