"""Shared helpers of the GPU parity tests: the tolerance and the comparison.

Tolerance for fp16 q/K/V with fp32 accumulation and fp16 output, element by
element over every compared output:
    max |gpu - oracle|                        <= 2e-3
    max |gpu - oracle| / max(|oracle|, 1e-3)  <= 1e-2
Rounding the exact result to fp16 alone costs a relative 2^-11 (4.9e-4).
The 1e-3 floor keeps near-zero outputs from making the ratio meaningless.

For bf16 q/K/V/out, rounding the output alone costs up to half an ulp, a
relative 2^-8 (3.9e-3): the absolute bound is 8e-3 (twice that at |out| = 1),
and the relative bound and its floor are the fp16 ones.

Every path, decode and multi-token alike, is held to these bounds.
"""

from __future__ import annotations

import numpy as np

MAX_ABS = 2e-3
MAX_REL = 1e-2
REL_FLOOR = 1e-3
BF16_MAX_ABS = 8e-3


def errors(got, want, rel_floor=REL_FLOOR):
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    d = np.abs(g - w)
    return float(d.max(initial=0.0)), float((d / np.maximum(np.abs(w), rel_floor)).max(initial=0.0))


def assert_close(got, want, what="", dtype="fp16", rel_floor=REL_FLOOR):
    assert np.all(np.isfinite(np.asarray(got, np.float64))), f"{what}: non-finite output"
    ea, er = errors(got, want, rel_floor)
    max_abs = BF16_MAX_ABS if dtype == "bf16" else MAX_ABS
    assert ea <= max_abs and er <= MAX_REL, f"{what}: max_abs={ea:.3g} max_rel={er:.3g}"
    return ea, er
