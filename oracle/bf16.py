"""Rounding to bfloat16, for the oracle's "bf16 storage" reading.

TEST INFRASTRUCTURE (imported only through the oracle).

The workloads are stated as "bf16 in, fp32 acc": every tensor-core GEMM takes bf16
operands and accumulates in fp32.  Inside the block that means the activations a
GEMM consumes (the LayerNorm output, the saved pre-activations, A, and dZ) are
stored in bf16.  ``round_bf16`` gives the oracle that storage step: the value of x
rounded to the nearest number with 8 significant bits (bf16's precision, same
exponent range as fp32), ties to even.
"""
from __future__ import annotations

import numpy as np

_BF16_MIN_NORMAL_EXP = -125   # frexp exponent of 2**-126
_BF16_SUBNORMAL_QUANTUM = -133


def round_bf16(x):
    """Nearest bf16 value of float64 x (round half to even), returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e with 0.5 <= |m| < 1
    normal = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    sub = np.ldexp(np.rint(np.ldexp(x, -_BF16_SUBNORMAL_QUANTUM)), _BF16_SUBNORMAL_QUANTUM)
    return np.where(e >= _BF16_MIN_NORMAL_EXP, normal, sub)


def identity(x):
    return np.asarray(x, dtype=np.float64)
