"""Oracle package: test infrastructure only (fp64 CPU statement of the layer and of QB).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import it.  The CUDA library never does.
"""
from .slmoe_oracle import *  # noqa: F401,F403
