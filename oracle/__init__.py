"""CPU oracle (test infrastructure only): see ``oracle/kvq_oracle.py``.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.
"""
from .kvq_oracle import *  # noqa: F401,F403
