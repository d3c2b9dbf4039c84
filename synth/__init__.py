"""Seeded synthetic inputs for the routed expert FFN.

This package holds the input generators shared by the CUDA path and the CPU
oracle.  It draws numbers and lays them out in the boundary blob format; it
holds none of the layer's arithmetic (no routing, dequantisation or FFN).
"""
from .synth import *  # noqa: F401,F403
