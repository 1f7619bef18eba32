"""CPU oracle for the ClusterKV decode path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never depends on it.
"""
from . import clusterkv  # noqa: F401
