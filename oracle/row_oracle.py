"""ctypes front end of the fp64 CPU LayerNorm / RMSNorm oracle (``row_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests and the reference leg of ``bench.py`` may
call it; the product path never does.

Arrays are row-major [M, N] (flat numpy buffers); inputs are converted to
float64 (fp16/bf16/fp32 values convert exactly) and every result is float64.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_P = ctypes.POINTER(ctypes.c_double)
_I = ctypes.c_int64
_D = ctypes.c_double


class RowOracle:
    """One loaded copy of the row oracle (the real one, or a mutant)."""

    def __init__(self, mutant: int = 0, outdir: str | None = None):
        path = _build.build(mutant, outdir, which="row")
        L = ctypes.CDLL(path)
        self.lib = L
        L.rno_ln_forward.argtypes = [_P, _I, _I, _P, _P, _D, _P, _P, _P]
        L.rno_rms_forward.argtypes = [_P, _I, _I, _P, _D, _P, _P]
        L.rno_ln_backward.argtypes = [_P, _P, _I, _I, _P, _D, _P, _P, _P]
        L.rno_rms_backward.argtypes = [_P, _P, _I, _I, _P, _D, _P, _P]
        for f in (L.rno_ln_forward, L.rno_rms_forward, L.rno_ln_backward, L.rno_rms_backward):
            f.restype = ctypes.c_int
        L.rno_mutant_id.restype = ctypes.c_int
        self.mutant = L.rno_mutant_id()

    @staticmethod
    def _d(a):
        if a is None:
            return None
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64).reshape(-1))

    @staticmethod
    def _p(a):
        return None if a is None else a.ctypes.data_as(_P)

    @staticmethod
    def _check(rc):
        if rc != 0:
            raise ValueError(f"row oracle rejected the arguments (code {rc})")

    def ln_forward(self, x, M, N, gamma, beta, eps):
        """(y, mean, rstd); gamma/beta may be None."""
        x = self._d(x)
        assert x.size == M * N
        y, mean, rstd = np.zeros(M * N), np.zeros(M), np.zeros(M)
        g, b = self._d(gamma), self._d(beta)
        self._check(self.lib.rno_ln_forward(self._p(x), M, N, self._p(g), self._p(b), eps,
                                            self._p(y), self._p(mean), self._p(rstd)))
        return y, mean, rstd

    def rms_forward(self, x, M, N, gamma, eps):
        """(y, rstd); gamma may be None."""
        x = self._d(x)
        assert x.size == M * N
        y, rstd = np.zeros(M * N), np.zeros(M)
        g = self._d(gamma)
        self._check(self.lib.rno_rms_forward(self._p(x), M, N, self._p(g), eps, self._p(y),
                                             self._p(rstd)))
        return y, rstd

    def ln_backward(self, dy, x, M, N, gamma, eps):
        """(dx, dgamma, dbeta); moments recomputed from x."""
        dy, x = self._d(dy), self._d(x)
        assert x.size == M * N and dy.size == x.size
        dx, dg, db = np.zeros(M * N), np.zeros(N), np.zeros(N)
        g = self._d(gamma)
        self._check(self.lib.rno_ln_backward(self._p(dy), self._p(x), M, N, self._p(g), eps,
                                             self._p(dx), self._p(dg), self._p(db)))
        return dx, dg, db

    def rms_backward(self, dy, x, M, N, gamma, eps):
        """(dx, dgamma); rstd recomputed from x."""
        dy, x = self._d(dy), self._d(x)
        assert x.size == M * N and dy.size == x.size
        dx, dg = np.zeros(M * N), np.zeros(N)
        g = self._d(gamma)
        self._check(self.lib.rno_rms_backward(self._p(dy), self._p(x), M, N, self._p(g), eps,
                                              self._p(dx), self._p(dg)))
        return dx, dg


_default = None


def get_row() -> RowOracle:
    """The real (unmutated) row oracle, loaded once per process."""
    global _default
    if _default is None:
        _default = RowOracle(0)
    return _default
