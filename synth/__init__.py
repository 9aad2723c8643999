"""Seeded synthetic inputs for the activation-sparse MoE workloads.

This package is shared by the CUDA path's tests/bench and by the CPU oracle.
It holds input synthesis only: random draws, the checkpoint-layout storage of
4-bit weights, and the calibration of per-neuron pre-activation offsets.  It
contains none of the method's arithmetic (no up-projection, no ReLU^2 of a
model activation, no down-projection, no routing).
"""
from .gen import *  # noqa: F401,F403
from .workloads import *  # noqa: F401,F403,E402
