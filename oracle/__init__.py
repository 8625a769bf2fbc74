"""CPU oracle for the block-scaled FP8 linear layer (test infrastructure).

Plain, slow, float64 numpy restatement of what the layer computes, written
from the pages' statement of the method.  Only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it;
the GPU library never does, and this package imports nothing from the GPU
library.  Parity status of every function is listed in ``fp8blk_oracle``'s
header.
"""
from .fp8blk_oracle import *  # noqa: F401,F403
