"""CPU oracle of the blended prefill (test infrastructure only; see cacheblend.py)."""
from .cacheblend import *  # noqa: F401,F403
