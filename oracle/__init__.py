"""CPU fp64 oracle for exact attention — test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It never imports the CUDA library, and the
library never imports it.
"""
from .attention import (as_f64, backward, delta, forward, forward_rows, scores,  # noqa: F401
                        softmax_rows)
from .merge import forward_shards, merge_lse, split_bounds  # noqa: F401
from .grouped import backward_gqa, expand_kv, forward_gqa, group_size  # noqa: F401
from .online_softmax import causal_blocks_visited, forward_blockwise  # noqa: F401
from .varlen import backward_varlen, forward_varlen  # noqa: F401
