"""Seeded synthetic inputs for the MoE layer (shared by the oracle tests and the GPU path).

This package holds no arithmetic of the MoE layer itself: only the counter-based
random stream that fills weight codes, row scales, router weights/biases and
hidden states, plus the layer shapes the workloads use.
"""
from .inputs import *  # noqa: F401,F403
