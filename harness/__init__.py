"""Seeded synthetic input generators shared by the oracle and the CUDA library (no method arithmetic)."""
from .inputs import *  # noqa: F401,F403
# device-side generation needs torch + harness/libsynth.so; import it as harness.device
