"""CPU oracle for the layer-streamed decoder training step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  It shares no code with ``host_memory_streamed_gb300``.
"""
from .decoder import *  # noqa: F401,F403
from .decoder import __all__  # noqa: F401
