"""GroupNorm forward/backward for GB300 (sm_103a).

The compute path lives in the C-ABI library ``libgn.so`` built from ``csrc/``;
``backward_normalization_gb300.gn`` is the thin Python binding over it.  This
package imports nothing heavy on import, so ``synth`` (the seeded input
generator) can be used without the CUDA library.
"""

__all__ = ["gn", "synth"]
