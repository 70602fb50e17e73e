"""CPU fp64 oracle for exact attention — test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It never imports the CUDA library, and the
library never imports it.
"""
from .attention import (as_f64, backward, delta, forward, forward_rows, scores,  # noqa: F401
                        softmax_rows)
from .online_softmax import causal_blocks_visited, forward_blockwise  # noqa: F401
