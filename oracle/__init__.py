"""CPU oracle (fp64) for the Prism block-sparse attention path.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the library.
"""
from .prism_oracle import *  # noqa: F401,F403
