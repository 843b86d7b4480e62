"""Shared GPU parity inputs that the CPU tests also inspect.

Only seeded input construction lives here (no normalisation arithmetic): the
cases whose 16-byte vectors hold channels of more than one group, and the
strongly correlated dy they are run with.
"""
from __future__ import annotations

import torch

from backward_normalization_gb300 import synth


# 16-byte vectors that hold channels of more than one group (4 fp32 or 8
# fp16/bf16 channels per vector against Cg = 10, 3, 1), with a dy that makes
# every term of dx large (see strong_dy) and per-channel offsets that give
# neighbouring groups different statistics.
def _spanning_cases():
    c0, c1, c2 = synth.WORKLOADS[0], synth.WORKLOADS[1], synth.WORKLOADS[2]
    off = ("uniform", -4.0, 4.0)
    xs = ("normal", 0.5, 2.0)
    return [
        ("fp32_nhwc_2x40x9x11_g4_cg10", c0.scaled(name="v10", layout="nhwc", C=40, G=4, H=9, W=11,
                                                  x=xs, channel_offset=off)),
        ("fp32_nhwc_2x48x7x13_g16_cg3", c0.scaled(name="v3", layout="nhwc", C=48, G=16, H=7, W=13,
                                                  x=xs, channel_offset=off)),
        ("fp32_nhwc_3x32x6x10_g32_cg1", c0.scaled(name="v1", layout="nhwc", N=3, C=32, G=32, H=6,
                                                  W=10, x=xs, channel_offset=off)),
        ("bf16_nhwc_3x320x17x17_g32_cg10", c2.scaled(name="b10", N=3, H=17, W=17, channel_offset=off)),
        ("fp16_nhwc_2x80x13x11_g8_cg10", c2.scaled(name="h10", dtype="f16", N=2, C=80, G=8, H=13,
                                                   W=11, channel_offset=off)),
        ("bf16_nhwc_2x64x9x14_g64_cg1", c2.scaled(name="b1", N=2, C=64, G=64, H=9, W=14,
                                                  channel_offset=off)),
        ("fp16_nhwc_2x48x10x10_g48_cg1", c1.scaled(name="h1", N=2, C=48, G=48, H=10, W=10, x=xs,
                                                   channel_offset=off)),
    ]


SPANNING = _spanning_cases()
SPANNING_NAMES = {c[1].name for c in SPANNING}


def strong_dy(inp, w, seed=0):
    """dy = 0.5 + 0.5*x + N(0, 1): mean(gamma*dy) and mean(gamma*dy*xhat) are
    then far from zero in every group, so a dx that dropped either mean term,
    flipped a sign or used another group's coefficients misses the tolerance
    by a wide margin (test_parity_inputs_cpu.py checks this with the oracle's
    planted-mistake copies)."""
    gen = torch.Generator().manual_seed(1000 + seed)
    noise = torch.randn(w.E, generator=gen, dtype=torch.float64)
    dy = 0.5 + 0.5 * inp["x"].double() + noise
    out = dict(inp)
    out["dy"] = dy.to(synth.DTYPES[w.dtype])
    return out
