"""Plain CPU oracle of the DSA decode hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline and ``--impl reference`` legs) may import or
run anything in this package.  The CUDA path never calls it and shares no
code with it.
"""
from .dsa_oracle import *  # noqa: F401,F403
