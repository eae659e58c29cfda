"""Test infrastructure: the fp64 CPU oracle of the DFlash draft attention layer.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (CPU baseline and
reference arm) may import this package.  The product path never does.
"""
from .dflash_oracle import *  # noqa: F401,F403
