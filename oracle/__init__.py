"""fp64 CPU oracles: GroupNorm forward/backward, and LayerNorm / RMSNorm over
rows (forward/backward).

Test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library in ``backward_normalization_gb300``.
"""
from .oracle import Oracle, get  # noqa: F401
from .row_oracle import RowOracle, get_row  # noqa: F401
