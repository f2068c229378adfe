"""CPU oracle for the trellis-quantized MoE grouped GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may.  It shares no code with the CUDA library.

See ``oracle/trellis_moe.py`` for what it computes and which passage each
function follows.
"""
from .trellis_moe import *  # noqa: F401,F403
