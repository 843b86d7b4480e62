"""Seeded synthetic inputs for GroupNorm forward/backward.

This module only draws random numbers and lays them out in memory; it holds
none of the normalisation arithmetic, so both the CUDA path and the fp64 oracle
can be fed from it.  Shapes and distributions are the five workloads the
library is measured on (activations [N, C, H, W]; N(mu, sigma) means mean mu
and standard deviation sigma).

Every tensor is returned FLAT, in its memory layout: ``"nchw"`` is
``[(n*C + c)*HW + hw]`` and ``"nhwc"`` (channels_last) is
``[(n*HW + hw)*C + c]``.  gamma and beta are fp32 ``[C]``.
"""
from __future__ import annotations

import dataclasses

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "f64": torch.float64}
LAYOUTS = {"nchw": 0, "nhwc": 1}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" | "f16" | "bf16" | "f64"  (x, y, dy, dx)
    layout: str         # "nchw" | "nhwc"
    N: int
    C: int
    G: int
    H: int
    W: int
    eps: float
    x: tuple            # ("normal", mu, sigma)
    dy: tuple
    gamma: tuple        # ("normal", mu, sigma) or ("const", v)
    beta: tuple
    channel_offset: tuple | None = None   # ("uniform", lo, hi): one draw per channel

    @property
    def HW(self) -> int:
        return self.H * self.W

    @property
    def E(self) -> int:
        return self.N * self.C * self.H * self.W

    def scaled(self, **kw) -> "Workload":
        """The same distributions on another shape (for small parity cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = [
    Workload("fp32_nchw_2x32x16x16_g8", "f32", "nchw", 2, 32, 8, 16, 16, 1e-5,
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
             ("normal", 1.0, 0.1), ("normal", 0.0, 0.1)),
    Workload("fp16_nhwc_1x128x1024x2048_g16", "f16", "nhwc", 1, 128, 16, 1024, 2048,
             1e-5, ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0)),
    Workload("bf16_nhwc_8x320x64x64_g32", "bf16", "nhwc", 8, 320, 32, 64, 64, 1e-6,
             ("normal", 0.5, 2.0), ("normal", 0.0, 1e-2),
             ("normal", 1.0, 0.1), ("normal", 0.0, 0.1)),
    Workload("fp32_nchw_112x64x512x512_g8", "f32", "nchw", 112, 64, 8, 512, 512, 1e-5,
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
             ("const", 1.0), ("const", 0.0)),
    Workload("bf16_nhwc_32x512x32x32_g32", "bf16", "nhwc", 32, 512, 32, 32, 32, 1e-5,
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
             ("normal", 1.0, 0.1), ("normal", 0.0, 0.1),
             channel_offset=("uniform", -4.0, 4.0)),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _draw(spec, n, gen, device, dtype=torch.float32):
    kind = spec[0]
    if kind == "normal":
        t = torch.randn(n, generator=gen, device=device, dtype=dtype)
        return t.mul_(spec[2]).add_(spec[1])
    if kind == "uniform":
        t = torch.rand(n, generator=gen, device=device, dtype=dtype)
        return t.mul_(spec[2] - spec[1]).add_(spec[1])
    if kind == "const":
        return torch.full((n,), float(spec[1]), device=device, dtype=dtype)
    raise ValueError(spec)


def _activation(w: Workload, spec, gen, device, offset):
    # f64 activations are drawn in f64 (most values then lie between fp32 values)
    t = _draw(spec, w.E, gen, device, torch.float64 if w.dtype == "f64" else torch.float32)
    if offset is not None:
        # one value per channel, shared by every n and every spatial position
        if w.layout == "nchw":
            t.view(w.N, w.C, w.HW).add_(offset.view(1, w.C, 1))
        else:
            t.view(w.N, w.HW, w.C).add_(offset.view(1, 1, w.C))
    return t.to(DTYPES[w.dtype])


def make_inputs(w: Workload, device="cpu", seed: int = 0, need_dy: bool = True):
    """dict(x, dy, gamma, beta): x/dy flat in w.layout and w.dtype.

    Draw order: channel offsets (if any), x, dy, gamma, beta."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    offset = None
    if w.channel_offset is not None:
        offset = _draw(w.channel_offset, w.C, gen, device)
    x = _activation(w, w.x, gen, device, offset)
    dy = _activation(w, w.dy, gen, device, None) if need_dy else None
    gamma = _draw(w.gamma, w.C, gen, device)
    beta = _draw(w.beta, w.C, gen, device)
    return {"x": x, "dy": dy, "gamma": gamma, "beta": beta}


def to_nchw_view(flat: torch.Tensor, w: Workload) -> torch.Tensor:
    """A [N, C, HW] view of a flat tensor stored in w.layout (data movement only)."""
    if w.layout == "nchw":
        return flat.view(w.N, w.C, w.HW)
    return flat.view(w.N, w.HW, w.C).permute(0, 2, 1)


# ------------------------------------------------ rows: LayerNorm / RMSNorm
@dataclasses.dataclass(frozen=True)
class RowWorkload:
    """A row-normalization problem over the last dimension of [M, N].  The
    shapes are those of the ROCm normalization-backward benchmark table
    (M = product of the leading dimensions); the page gives no value
    distributions, so x, dy ~ N(0, 1), gamma ~ N(1, 0.1), beta ~ N(0, 0.1)."""
    name: str
    op: str       # "ln" | "rms"
    dtype: str    # "f32" | "f16" | "bf16"
    M: int
    N: int
    eps: float = 1e-5

    @property
    def E(self) -> int:
        return self.M * self.N


ROW_WORKLOADS = [
    RowWorkload("ln_f16_4096x1024", "ln", "f16", 4096, 1024),
    RowWorkload("ln_bf16_4096x1024", "ln", "bf16", 4096, 1024),
    RowWorkload("ln_f32_4096x1024", "ln", "f32", 4096, 1024),
    RowWorkload("ln_f16_1024x768", "ln", "f16", 1024, 768),
    RowWorkload("ln_f16_131072x64", "ln", "f16", 131072, 64),
    RowWorkload("ln_bf16_131072x4096", "ln", "bf16", 32 * 4096, 4096),
    RowWorkload("ln_f16_8192x768", "ln", "f16", 8 * 1024, 768),
    RowWorkload("rms_f16_4096x1024", "rms", "f16", 4096, 1024),
    RowWorkload("rms_bf16_131072x4096", "rms", "bf16", 32 * 4096, 4096),
    RowWorkload("rms_f16_131072x64", "rms", "f16", 131072, 64),
]
ROW_BY_NAME = {w.name: w for w in ROW_WORKLOADS}


def make_row_inputs(w: RowWorkload, device="cpu", seed: int = 0):
    """dict(x, dy, gamma, beta): x/dy flat [M*N] in w.dtype; gamma/beta fp32 [N].
    Draw order: x, dy, gamma, beta."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = _draw(("normal", 0.0, 1.0), w.E, gen, device).to(DTYPES[w.dtype])
    dy = _draw(("normal", 0.0, 1.0), w.E, gen, device).to(DTYPES[w.dtype])
    gamma = _draw(("normal", 1.0, 0.1), w.N, gen, device)
    beta = _draw(("normal", 0.0, 0.1), w.N, gen, device)
    return {"x": x, "dy": dy, "gamma": gamma, "beta": beta}
