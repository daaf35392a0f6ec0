"""CPU oracle of the MLA sublayer -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""
from .mla_oracle import *  # noqa: F401,F403
from .mla_oracle import Dims, KIMI_K2  # noqa: F401
