"""Seeded synthetic inputs for the paged-expert MoE layer.

This package only draws random numbers and encodes them in the expert byte
layouts; it holds none of the layer's arithmetic (no routing, no expert math, no
residency logic). Both the oracle's tests and the CUDA path's tests and bench
draw their inputs from here, so the two sides see the same bytes.
"""

from .generators import *  # noqa: F401,F403
from .configs import CONFIGS, LayerShape  # noqa: F401
