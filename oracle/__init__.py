"""fp64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The library's product path never does:
it has no CPU fallback.
"""

from .spec_oracle import *  # noqa: F401,F403
from .spec_oracle import NEAR_TIE  # noqa: F401
