"""ctypes front end of the fp64 CPU GroupNorm oracle (``gn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may call it; the product path never does.

All arrays are flat numpy buffers holding the tensor in its memory layout:
``layout=0`` is NCHW (offset ``(n*C + c)*HW + hw``), ``layout=1`` is NHWC /
channels_last (offset ``(n*HW + hw)*C + c``).  Inputs are converted to float64
(fp16/bf16/fp32 values convert exactly); every result is float64.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_P = ctypes.POINTER(ctypes.c_double)
_PI = ctypes.POINTER(ctypes.c_int64)
_I = ctypes.c_int64


class Oracle:
    """One loaded copy of the oracle library (the real one, or a mutant)."""

    def __init__(self, mutant: int = 0, outdir: str | None = None):
        path = _build.build(mutant, outdir)
        self.lib = ctypes.CDLL(path)
        L = self.lib
        L.gno_stats.argtypes = [_P, _I, _I, _I, _I, ctypes.c_int, ctypes.c_double,
                                _P, _P, _P]
        L.gno_forward.argtypes = [_P, _I, _I, _I, _I, ctypes.c_int, _P, _P,
                                  ctypes.c_double, _P, _P, _P]
        L.gno_backward.argtypes = [_P, _P, _I, _I, _I, _I, ctypes.c_int, _P,
                                   ctypes.c_double, _P, _P, _P]
        L.gno_forward_at.argtypes = [_P, _I, _I, _I, _I, ctypes.c_int, _P, _P,
                                     ctypes.c_double, _PI, _I, _P, _P, _P]
        L.gno_backward_at.argtypes = [_P, _P, _I, _I, _I, _I, ctypes.c_int, _P,
                                      ctypes.c_double, _PI, _I, _P, _P, _P]
        for f in (L.gno_stats, L.gno_forward, L.gno_backward, L.gno_forward_at,
                  L.gno_backward_at):
            f.restype = ctypes.c_int
        L.gno_mutant_id.restype = ctypes.c_int
        self.mutant = L.gno_mutant_id()

    # ------------------------------------------------------------------ helpers
    @staticmethod
    def _d(a):
        if a is None:
            return None
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64).reshape(-1))

    @staticmethod
    def _p(a):
        if a is None:
            return None
        return a.ctypes.data_as(_P)

    @staticmethod
    def _check(rc):
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (code {rc})")

    # --------------------------------------------------------------- interface
    def stats(self, x, N, C, HW, G, layout, eps):
        """(mean, var, rstd), each of length N*G."""
        x = self._d(x)
        assert x.size == N * C * HW
        mean = np.zeros(N * G)
        var = np.zeros(N * G)
        rstd = np.zeros(N * G)
        self._check(self.lib.gno_stats(self._p(x), N, C, HW, G, layout, eps,
                                       self._p(mean), self._p(var), self._p(rstd)))
        return mean, var, rstd

    def forward(self, x, N, C, HW, G, layout, gamma, beta, eps):
        """(y, mean, rstd); gamma/beta may be None (no affine)."""
        x = self._d(x)
        assert x.size == N * C * HW
        g, b = self._d(gamma), self._d(beta)
        y = np.zeros(N * C * HW)
        mean = np.zeros(N * G)
        rstd = np.zeros(N * G)
        self._check(self.lib.gno_forward(self._p(x), N, C, HW, G, layout,
                                         self._p(g), self._p(b), eps, self._p(y),
                                         self._p(mean), self._p(rstd)))
        return y, mean, rstd

    def backward(self, dy, x, N, C, HW, G, layout, gamma, eps):
        """(dx, dgamma, dbeta); the oracle recomputes its own moments from x."""
        dy, x = self._d(dy), self._d(x)
        assert x.size == N * C * HW and dy.size == x.size
        g = self._d(gamma)
        dx = np.zeros(N * C * HW)
        dgamma = np.zeros(C)
        dbeta = np.zeros(C)
        self._check(self.lib.gno_backward(self._p(dy), self._p(x), N, C, HW, G,
                                          layout, self._p(g), eps, self._p(dx),
                                          self._p(dgamma), self._p(dbeta)))
        return dx, dgamma, dbeta

    def forward_at(self, x, N, C, HW, G, layout, gamma, beta, eps, idx):
        """(y at flat offsets idx, mean, rstd)."""
        x = self._d(x)
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
        g, b = self._d(gamma), self._d(beta)
        y = np.zeros(idx.size)
        mean = np.zeros(N * G)
        rstd = np.zeros(N * G)
        self._check(self.lib.gno_forward_at(
            self._p(x), N, C, HW, G, layout, self._p(g), self._p(b), eps,
            idx.ctypes.data_as(_PI), idx.size, self._p(y), self._p(mean),
            self._p(rstd)))
        return y, mean, rstd

    def backward_at(self, dy, x, N, C, HW, G, layout, gamma, eps, idx):
        """(dx at flat offsets idx, dgamma, dbeta)."""
        dy, x = self._d(dy), self._d(x)
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
        g = self._d(gamma)
        dx = np.zeros(idx.size)
        dgamma = np.zeros(C)
        dbeta = np.zeros(C)
        self._check(self.lib.gno_backward_at(
            self._p(dy), self._p(x), N, C, HW, G, layout, self._p(g), eps,
            idx.ctypes.data_as(_PI), idx.size, self._p(dx), self._p(dgamma),
            self._p(dbeta)))
        return dx, dgamma, dbeta


_default = None


def get() -> Oracle:
    """The real (unmutated) oracle, loaded once per process."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default
