"""fp64 CPU oracle of the block with FP8 (E4M3) GEMMs: per-tensor current scaling.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.

Sources (page title, section):
  [Onegen]  "Megatron-LM: advanced language model training" (onegen.ai), sections "Why
            Megatron-LM Matters" and "Key Features": mixed precision down to FP8.
  [Concept] "Megatron-LM / Megatron-Core" concept note, section "Key math / How it
            works": FP8 through Transformer Engine.

The pages name FP8 training and nothing of its arithmetic.  The plainest reading,
taken here (and listed with its reasons in the design notes):

  * every operand of every one of the six GEMMs is stored in E4M3 (4 exponent bits,
    3 mantissa bits, bias 7, no infinities, largest finite 448, subnormal quantum
    2^-9), with one scale per tensor ("per-tensor current scaling": the scale comes
    from the tensor's own absolute maximum, taken over the whole tensor, i.e. over
    all tensor-parallel shards at once -- the amax reduction across the TP group);
  * the scale is a power of two, s = 2^k with k the largest integer such that
    amax * 2^k <= 448 (k = 0 for an all-zero tensor), so that x * s is exact and the
    only rounding is the one to E4M3: q = e4m3(x * 2^k), round to nearest, ties to
    even;  the GEMM multiplies the codes and rescales by 2^-(k_a + k_b);
  * what is not a GEMM operand keeps the bf16 block's precision: Z (G, U), A and dZ
    are stored in bf16 before they are quantized or used, biases and bias gradients
    and the LayerNorm are unchanged, Y, dX and the weight gradients are exact here
    (fp32 on the GPU).

A GEMM operand and its transpose have one scale (per-tensor), so fc1, dX and dW1
see the same quantized X / W1 / dZ values in either orientation.
"""
from __future__ import annotations

import numpy as np

from . import mlp as _mlp
from .bf16 import round_bf16

E4M3_MAX = 448.0
_E4M3_MIN_NORMAL_EXP = -5        # frexp exponent of 2**-6, the smallest normal
_E4M3_SUBNORMAL_QUANTUM = -9     # 2**-9


def round_e4m3(x):
    """Nearest E4M3 value of float64 x (ties to even), saturating at +-448; float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                                   # x = m 2^e, 0.5 <= |m| < 1
    normal = np.ldexp(np.rint(np.ldexp(m, 4)), e - 4)   # 4 significant bits
    sub = np.ldexp(np.rint(np.ldexp(x, -_E4M3_SUBNORMAL_QUANTUM)), _E4M3_SUBNORMAL_QUANTUM)
    r = np.where(e >= _E4M3_MIN_NORMAL_EXP, normal, sub)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def scale_exponent(amax):
    """The largest integer k with amax * 2^k <= 448 (0 when amax is 0)."""
    amax = float(amax)
    if amax == 0.0:
        return 0
    m, e = np.frexp(amax)                # amax = m 2^e;  448 = 0.875 * 2^9
    return int(9 - e) if m <= 0.875 else int(8 - e)


def quantize(x):
    """(dequantized values q * 2^-k, codes q = e4m3(x 2^k), k) of one tensor."""
    x = np.asarray(x, dtype=np.float64)
    k = scale_exponent(np.abs(x).max() if x.size else 0.0)
    q = round_e4m3(np.ldexp(x, k))
    return np.ldexp(q, -k), q, k


def deq(x):
    """The values a GEMM sees for operand x: its E4M3 quantization, rescaled."""
    return quantize(x)[0]


# ---------------------------------------------------------------- the block
def mlp_forward_fp8(X, W1, b1, W2, b2, act="gelu"):
    """Forward with E4M3 GEMMs.  Returns Y and the saved bf16 activations (Z or G, U; A)."""
    X, b1, b2 = np.asarray(X, np.float64), _mlp._f64(b1), _mlp._f64(b2)
    Xd = deq(X)
    W1d = deq(W1)                       # one scale over all shards (and gate and up)
    W2d = _mlp.full_w2(deq(W2))
    out = {}
    if act == "swiglu":
        Wg, Wu = _mlp.full_w1(W1d, act)
        G, U = Xd @ Wg.T, Xd @ Wu.T
        A = round_bf16(_mlp.silu(G) * U)
        out.update(G=round_bf16(G), U=round_bf16(U))
    else:
        fn, _ = _mlp._POINTWISE[act]
        Z = Xd @ _mlp.full_w1(W1d, act).T
        if b1 is not None:
            Z = Z + b1
        A = round_bf16(fn(Z))
        out["Z"] = round_bf16(Z)
    Y = deq(A) @ W2d.T
    if b2 is not None:
        Y = Y + b2
    out.update(A=A, Y=Y)
    return out


def mlp_backward_fp8(X, W1, b1, W2, dY, act="gelu"):
    """Backward with E4M3 GEMMs: dgrad and wgrad operands quantized per tensor."""
    X, dY = np.asarray(X, np.float64), np.asarray(dY, np.float64)
    t = np.asarray(W2).shape[0]
    fwd = mlp_forward_fp8(X, W1, b1, W2, None, act)
    Xd, dYd, Ad = deq(X), deq(dY), deq(fwd["A"])
    W1d = deq(W1)
    W2f = _mlp.full_w2(deq(W2))
    db2 = dY.sum(axis=0)
    dA = dYd @ W2f
    dW2f = dYd.T @ Ad
    if act == "swiglu":
        G, U = fwd["G"], fwd["U"]
        dG = round_bf16(dA * U * _mlp.silu_grad(G))
        dU = round_bf16(dA * _mlp.silu(G))
        dZd = deq(np.concatenate([dG, dU], axis=1))        # one scale over [dG | dU]
        F = G.shape[1]
        dGd, dUd = dZd[:, :F], dZd[:, F:]
        Wg, Wu = _mlp.full_w1(W1d, act)
        dX = dGd @ Wg + dUd @ Wu
        dW1 = _mlp.shard_w1_grad((dGd.T @ Xd, dUd.T @ Xd), t, act)
        db1 = None
    else:
        _, dfn = _mlp._POINTWISE[act]
        dZ = round_bf16(dA * dfn(fwd["Z"]))
        dZd = deq(dZ)
        dX = dZd @ _mlp.full_w1(W1d, act)
        dW1 = _mlp.shard_w1_grad(dZd.T @ Xd, t, act)
        db1 = dZ.sum(axis=0) if b1 is not None else None
    out = {"dX": dX, "dW1": dW1, "dW2": _mlp.shard_w2_grad(dW2f, t), "db1": db1, "db2": db2}
    if act == "swiglu":
        out.update(dG_bf16=dG, dU_bf16=dU)
    else:
        out["dZ_bf16"] = dZ
    return out


def block_fp8(X, gamma, beta, eps, W1, b1, W2, b2, dY, act):
    """The pre-LN block with E4M3 GEMMs: LN (unchanged, Xn stored in bf16), the FP8 MLP on
    Xn, and the LN backward of its input gradient."""
    from . import layernorm as _ln
    X = np.asarray(X, np.float64)
    Xn, mu, rstd = _ln.layernorm_fwd(X, gamma, beta, eps)
    Xn = round_bf16(Xn)
    out = mlp_forward_fp8(Xn, W1, b1, W2, b2, act)
    g = mlp_backward_fp8(Xn, W1, b1, W2, dY, act)
    dX, dgamma, dbeta = _ln.layernorm_bwd(X, gamma, mu, rstd, g["dX"])
    out.update(g)
    out.update(Xn=Xn, dXn=g["dX"], dX=dX, dgamma=dgamma, dbeta=dbeta)
    return out
