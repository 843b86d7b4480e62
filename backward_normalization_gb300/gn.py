"""Thin Python binding of libgn.so (include/gn.h): argument marshalling only.

Every function here hands raw device pointers, sizes and a stream to the C
ABI; all GroupNorm arithmetic runs in the CUDA kernels of ``csrc/``.  Loading
fails loudly (ImportError / RuntimeError) when the library has not been built;
there is no fallback implementation.

Tensors are torch tensors holding the data flat in the chosen layout
(``"nchw"`` or ``"nhwc"``); torch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgn.so")

GN_OK, GN_ERR_INVALID, GN_ERR_UNSUPPORTED, GN_ERR_WORKSPACE, GN_ERR_CUDA, GN_ERR_TIMEOUT = range(6)
FAULT_NONE, FAULT_LAUNCH, FAULT_STALL = 0, 1, 2
OP_FWD, OP_BWD = 0, 1
LAYOUT = {"nchw": 0, "nhwc": 1}
DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.float64: 3}
DTYPE_NAME = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3}

_I64 = ctypes.c_int64
_VP = ctypes.c_void_p


class GnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class PlanDesc(ctypes.Structure):
    _fields_ = [("regime", ctypes.c_int), ("launches", ctypes.c_int),
                ("vector_width", ctypes.c_int), ("threads", ctypes.c_int),
                ("ctas", ctypes.c_int64), ("partials", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("cluster_ctas", ctypes.c_int),
                ("max_clusters", ctypes.c_int), ("smem_bytes", ctypes.c_size_t),
                ("err_offset", ctypes.c_size_t), ("finalise_second", ctypes.c_int),
                ("level1_items", ctypes.c_int), ("clear_bytes", ctypes.c_size_t),
                ("piece_elems", ctypes.c_int64), ("pieces_per_unit", ctypes.c_int64),
                ("slots", ctypes.c_int), ("hold_buffers", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        L.gn_workspace_size.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int]
        L.gn_workspace_size.restype = ctypes.c_size_t
        L.gn_fwd.argtypes = [_VP, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _VP, _VP,
                             ctypes.c_float, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]
        L.gn_fwd.restype = ctypes.c_int
        L.gn_bwd.argtypes = [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, ctypes.c_int,
                             ctypes.c_int, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]
        L.gn_bwd.restype = ctypes.c_int
        L.gn_status_string.argtypes = [ctypes.c_int]
        L.gn_status_string.restype = ctypes.c_char_p
        L.gn_last_cuda_error.argtypes = []
        L.gn_last_cuda_error.restype = ctypes.c_int
        L.gn_plan_info.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.POINTER(PlanDesc)]
        L.gn_plan_info.restype = ctypes.c_int
        L.gn_fwd_static_ws.argtypes = [_VP, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _VP,
                                       _VP, ctypes.c_float, _VP, _VP, _VP, _VP]
        L.gn_fwd_static_ws.restype = ctypes.c_int
        L.gn_fwd_ex.argtypes = [_VP, _I64, _I64, _I64, _I64, _I64, _I64, ctypes.c_int,
                                ctypes.c_int, _VP, _VP, ctypes.c_float, _VP, _I64, _I64, _VP, _VP,
                                _VP, ctypes.c_size_t, _VP]
        L.gn_fwd_ex.restype = ctypes.c_int
        L.gn_bwd_ex.argtypes = [_VP, _I64, _I64, _VP, _I64, _I64, _VP, _VP, _VP, _I64, _I64, _I64,
                                _I64, ctypes.c_int, ctypes.c_int, _VP, _I64, _I64, _VP, _VP, _VP,
                                ctypes.c_size_t, _VP]
        L.gn_bwd_ex.restype = ctypes.c_int
        L.gn_workspace_status.argtypes = [_VP, _VP]
        L.gn_workspace_status.restype = ctypes.c_int
        L.gn_set_fault_injection.argtypes = [ctypes.c_int]
        L.gn_set_fault_injection.restype = ctypes.c_int
        L.gn_set_regime.argtypes = [ctypes.c_int]
        L.gn_set_regime.restype = ctypes.c_int
        L.gn_set_timing_events.argtypes = [_VP, _VP, _VP]
        L.gn_set_timing_events.restype = ctypes.c_int
        # LayerNorm / RMSNorm over rows (include/ln.h)
        L.ln_workspace_size.argtypes = [_I64, _I64, ctypes.c_int]
        L.ln_workspace_size.restype = ctypes.c_size_t
        L.ln_fwd.argtypes = [_VP, _I64, _I64, ctypes.c_int, _VP, _VP, ctypes.c_float, _VP, _VP,
                             _VP, _VP]
        L.ln_bwd.argtypes = [_VP, _VP, _VP, _VP, _VP, _I64, _I64, ctypes.c_int, _VP, _VP, _VP,
                             _VP, ctypes.c_size_t, _VP]
        L.rms_fwd.argtypes = [_VP, _I64, _I64, ctypes.c_int, _VP, ctypes.c_float, _VP, _VP, _VP]
        L.rms_bwd.argtypes = [_VP, _VP, _VP, _VP, _I64, _I64, ctypes.c_int, _VP, _VP, _VP,
                              ctypes.c_size_t, _VP]
        L.ln_fwd_ex.argtypes = [_VP, _I64, _I64, _I64, ctypes.c_int, _VP, _VP, ctypes.c_float,
                                _VP, _I64, _VP, _VP, _VP]
        L.ln_bwd_ex.argtypes = [_VP, _I64, _VP, _I64, _VP, _VP, _VP, _I64, _I64, ctypes.c_int,
                                _VP, _I64, _VP, _VP, _VP, ctypes.c_size_t, _VP]
        L.rms_fwd_ex.argtypes = [_VP, _I64, _I64, _I64, ctypes.c_int, _VP, ctypes.c_float, _VP,
                                 _I64, _VP, _VP]
        L.rms_bwd_ex.argtypes = [_VP, _I64, _VP, _I64, _VP, _VP, _I64, _I64, ctypes.c_int, _VP,
                                 _I64, _VP, _VP, ctypes.c_size_t, _VP]
        for f in (L.ln_fwd, L.ln_bwd, L.rms_fwd, L.rms_bwd, L.ln_fwd_ex, L.ln_bwd_ex,
                  L.rms_fwd_ex, L.rms_bwd_ex):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gn_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_size(op, N, C, HW, G, layout, dtype) -> int:
    lay = LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = DTYPE[dtype] if isinstance(dtype, torch.dtype) else (
        DTYPE_NAME[dtype] if isinstance(dtype, str) else int(dtype))
    return int(lib().gn_workspace_size(op, N, C, HW, G, lay, dt))


def plan_info(op, N, C, HW, G, layout, dtype, aligned=True) -> PlanDesc:
    lay = LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = DTYPE[dtype] if isinstance(dtype, torch.dtype) else (
        DTYPE_NAME[dtype] if isinstance(dtype, str) else int(dtype))
    d = PlanDesc()
    rc = lib().gn_plan_info(op, N, C, HW, G, lay, dt, int(bool(aligned)), ctypes.byref(d))
    if rc != GN_OK:
        raise GnError(rc, "gn_plan_info")
    return d


def fwd_raw(x, N, C, HW, G, layout, gamma, beta, eps, y, mean, rstd, workspace,
            stream=None) -> int:
    """gn_fwd on torch tensors; returns the gn_status."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().gn_fwd(_ptr(x), N, C, HW, G, LAYOUT[layout], DTYPE[x.dtype], _ptr(gamma),
                        _ptr(beta), float(eps), _ptr(y), _ptr(mean), _ptr(rstd),
                        _ptr(workspace), ws_bytes, _stream(stream))


def fwd_static_ws_raw(x, N, C, HW, G, layout, gamma, beta, eps, y, mean, rstd,
                      stream=None) -> int:
    """gn_fwd_static_ws on torch tensors (no workspace argument); returns the
    gn_status."""
    return lib().gn_fwd_static_ws(_ptr(x), N, C, HW, G, LAYOUT[layout], DTYPE[x.dtype],
                                  _ptr(gamma), _ptr(beta), float(eps), _ptr(y), _ptr(mean),
                                  _ptr(rstd), _stream(stream))


def bwd_raw(dy, x, mean, rstd, gamma, N, C, HW, G, layout, dx, dgamma, dbeta, workspace,
            stream=None) -> int:
    """gn_bwd on torch tensors; returns the gn_status."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().gn_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(gamma), N, C, HW, G,
                        LAYOUT[layout], DTYPE[x.dtype], _ptr(dx), _ptr(dgamma), _ptr(dbeta),
                        _ptr(workspace), ws_bytes, _stream(stream))


def fwd_ex_raw(x, x_s, N, C, HW, G, layout, gamma, beta, eps, y, y_s, mean, rstd, workspace,
               stream=None) -> int:
    """gn_fwd_ex: x and y are tensors whose data_ptr() is element (0, 0, 0) of
    the view; x_s and y_s are (sample stride, plane or row stride) in
    elements.  Returns the gn_status."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().gn_fwd_ex(_ptr(x), x_s[0], x_s[1], N, C, HW, G, LAYOUT[layout], DTYPE[x.dtype],
                           _ptr(gamma), _ptr(beta), float(eps), _ptr(y), y_s[0], y_s[1],
                           _ptr(mean), _ptr(rstd), _ptr(workspace), ws_bytes, _stream(stream))


def bwd_ex_raw(dy, dy_s, x, x_s, mean, rstd, gamma, N, C, HW, G, layout, dx, dx_s, dgamma,
               dbeta, workspace, stream=None) -> int:
    """gn_bwd_ex on strided views (see fwd_ex_raw); returns the gn_status."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().gn_bwd_ex(_ptr(dy), dy_s[0], dy_s[1], _ptr(x), x_s[0], x_s[1], _ptr(mean),
                           _ptr(rstd), _ptr(gamma), N, C, HW, G, LAYOUT[layout], DTYPE[x.dtype],
                           _ptr(dx), dx_s[0], dx_s[1], _ptr(dgamma), _ptr(dbeta),
                           _ptr(workspace), ws_bytes, _stream(stream))


REGIME_AUTO, REGIME_TWO_KERNEL, REGIME_RESIDENT, REGIME_PIPELINED, REGIME_WAVE, REGIME_FLAT = \
    -1, 0, 1, 2, 3, 4


def set_regime(regime: int) -> None:
    """Test hook: force the kernel family (REGIME_AUTO restores the default)."""
    rc = lib().gn_set_regime(int(regime))
    if rc != GN_OK:
        raise GnError(rc, "gn_set_regime")


def set_timing_events(ev_begin=None, ev_mid=None, ev_end=None) -> None:
    """Make the following calls of this thread record torch.cuda.Event objects
    before, between and after their two kernels (None: no record)."""
    def h(e):
        if e is None:
            return None
        if not e.cuda_event:  # torch creates the CUDA event on first record
            e.record()
        return e.cuda_event
    lib().gn_set_timing_events(h(ev_begin), h(ev_mid), h(ev_end))


def alloc_workspace(op, N, C, HW, G, layout, dtype, device="cuda"):
    """A workspace for gn_fwd / gn_bwd of this problem.  Its contents do not
    matter: every call clears the counters it uses before its kernels run."""
    n = workspace_size(op, N, C, HW, G, layout, dtype)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def workspace_status(workspace, stream=None) -> int:
    """gn_workspace_status: waits for `stream` and returns GN_OK, or
    GN_ERR_TIMEOUT when a bounded wait of the last call on `workspace` ran out."""
    return lib().gn_workspace_status(_ptr(workspace), _stream(stream))


def set_fault_injection(mode: int) -> None:
    """Test hook: FAULT_NONE, FAULT_LAUNCH (calls fail before enqueuing
    anything) or FAULT_STALL (the next wave-regime call withholds one arrival)."""
    rc = lib().gn_set_fault_injection(int(mode))
    if rc != GN_OK:
        raise GnError(rc, "gn_set_fault_injection")


def forward(x, N, C, HW, G, layout, gamma=None, beta=None, eps=1e-5, workspace=None,
            stream=None):
    """Allocates y/mean/rstd (and a workspace if none is given), calls gn_fwd.
    Returns (y, mean, rstd)."""
    y = torch.empty_like(x)
    mean = torch.empty(N * G, dtype=torch.float32, device=x.device)
    rstd = torch.empty(N * G, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(OP_FWD, N, C, HW, G, layout, x.dtype, x.device)
    rc = fwd_raw(x, N, C, HW, G, layout, gamma, beta, eps, y, mean, rstd, workspace, stream)
    if rc != GN_OK:
        raise GnError(rc, "gn_fwd")
    return y, mean, rstd


def backward(dy, x, mean, rstd, N, C, HW, G, layout, gamma=None, workspace=None,
             need_params=True, stream=None):
    """Allocates dx (and dgamma/dbeta, a workspace), calls gn_bwd.
    Returns (dx, dgamma, dbeta)."""
    dx = torch.empty_like(x)
    dgamma = dbeta = None
    if need_params:
        dgamma = torch.empty(C, dtype=torch.float32, device=x.device)
        dbeta = torch.empty(C, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(OP_BWD, N, C, HW, G, layout, x.dtype, x.device)
    rc = bwd_raw(dy, x, mean, rstd, gamma, N, C, HW, G, layout, dx, dgamma, dbeta, workspace,
                 stream)
    if rc != GN_OK:
        raise GnError(rc, "gn_bwd")
    return dx, dgamma, dbeta


# ------------------------------------------------ LayerNorm / RMSNorm over rows
def ln_workspace_size(M, N, dtype) -> int:
    dt = DTYPE[dtype] if isinstance(dtype, torch.dtype) else (
        DTYPE_NAME[dtype] if isinstance(dtype, str) else int(dtype))
    return int(lib().ln_workspace_size(M, N, dt))


def ln_fwd_raw(x, M, N, gamma, beta, eps, y, mean, rstd, stream=None) -> int:
    return lib().ln_fwd(_ptr(x), M, N, DTYPE[x.dtype], _ptr(gamma), _ptr(beta), float(eps),
                        _ptr(y), _ptr(mean), _ptr(rstd), _stream(stream))


def ln_bwd_raw(dy, x, mean, rstd, gamma, M, N, dx, dgamma, dbeta, workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().ln_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(gamma), M, N,
                        DTYPE[x.dtype], _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(workspace),
                        ws_bytes, _stream(stream))


def rms_fwd_raw(x, M, N, gamma, eps, y, rstd, stream=None) -> int:
    return lib().rms_fwd(_ptr(x), M, N, DTYPE[x.dtype], _ptr(gamma), float(eps), _ptr(y),
                         _ptr(rstd), _stream(stream))


def rms_bwd_raw(dy, x, rstd, gamma, M, N, dx, dgamma, workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().rms_bwd(_ptr(dy), _ptr(x), _ptr(rstd), _ptr(gamma), M, N, DTYPE[x.dtype],
                         _ptr(dx), _ptr(dgamma), _ptr(workspace), ws_bytes, _stream(stream))


def _row_ws(M, N, dtype, device):
    n = ln_workspace_size(M, N, dtype)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def ln_forward(x, M, N, gamma=None, beta=None, eps=1e-5, stream=None):
    """LayerNorm over rows of x [M, N] (flat); returns (y, mean, rstd)."""
    y = torch.empty_like(x)
    mean = torch.empty(M, dtype=torch.float32, device=x.device)
    rstd = torch.empty(M, dtype=torch.float32, device=x.device)
    rc = ln_fwd_raw(x, M, N, gamma, beta, eps, y, mean, rstd, stream)
    if rc != GN_OK:
        raise GnError(rc, "ln_fwd")
    return y, mean, rstd


def ln_backward(dy, x, mean, rstd, M, N, gamma=None, want=(True, True), workspace=None,
                stream=None):
    """LayerNorm backward; returns (dx, dgamma or None, dbeta or None)."""
    dx = torch.empty_like(x)
    dg = torch.empty(N, dtype=torch.float32, device=x.device) if want[0] else None
    db = torch.empty(N, dtype=torch.float32, device=x.device) if want[1] else None
    if workspace is None:
        workspace = _row_ws(M, N, x.dtype, x.device)
    rc = ln_bwd_raw(dy, x, mean, rstd, gamma, M, N, dx, dg, db, workspace, stream)
    if rc != GN_OK:
        raise GnError(rc, "ln_bwd")
    return dx, dg, db


def rms_forward(x, M, N, gamma=None, eps=1e-5, stream=None):
    """RMSNorm over rows of x [M, N] (flat); returns (y, rstd)."""
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=x.device)
    rc = rms_fwd_raw(x, M, N, gamma, eps, y, rstd, stream)
    if rc != GN_OK:
        raise GnError(rc, "rms_fwd")
    return y, rstd


def rms_backward(dy, x, rstd, M, N, gamma=None, want_dgamma=True, workspace=None, stream=None):
    """RMSNorm backward; returns (dx, dgamma or None)."""
    dx = torch.empty_like(x)
    dg = torch.empty(N, dtype=torch.float32, device=x.device) if want_dgamma else None
    if workspace is None:
        workspace = _row_ws(M, N, x.dtype, x.device)
    rc = rms_bwd_raw(dy, x, rstd, gamma, M, N, dx, dg, workspace, stream)
    if rc != GN_OK:
        raise GnError(rc, "rms_bwd")
    return dx, dg


def ln_fwd_ex_raw(x, ldx, M, N, gamma, beta, eps, y, ldy, mean, rstd, stream=None) -> int:
    """ln_fwd_ex: rows ldx / ldy elements apart (x and y may be views into wider buffers)."""
    return lib().ln_fwd_ex(_ptr(x), ldx, M, N, DTYPE[x.dtype], _ptr(gamma), _ptr(beta),
                           float(eps), _ptr(y), ldy, _ptr(mean), _ptr(rstd), _stream(stream))


def ln_bwd_ex_raw(dy, lddy, x, ldx, mean, rstd, gamma, M, N, dx, lddx, dgamma, dbeta,
                  workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().ln_bwd_ex(_ptr(dy), lddy, _ptr(x), ldx, _ptr(mean), _ptr(rstd), _ptr(gamma),
                           M, N, DTYPE[x.dtype], _ptr(dx), lddx, _ptr(dgamma), _ptr(dbeta),
                           _ptr(workspace), ws_bytes, _stream(stream))


def rms_fwd_ex_raw(x, ldx, M, N, gamma, eps, y, ldy, rstd, stream=None) -> int:
    return lib().rms_fwd_ex(_ptr(x), ldx, M, N, DTYPE[x.dtype], _ptr(gamma), float(eps),
                            _ptr(y), ldy, _ptr(rstd), _stream(stream))


def rms_bwd_ex_raw(dy, lddy, x, ldx, rstd, gamma, M, N, dx, lddx, dgamma, workspace,
                   stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib().rms_bwd_ex(_ptr(dy), lddy, _ptr(x), ldx, _ptr(rstd), _ptr(gamma), M, N,
                            DTYPE[x.dtype], _ptr(dx), lddx, _ptr(dgamma), _ptr(workspace),
                            ws_bytes, _stream(stream))
