"""fp64 CPU oracle of the sequence-parallel LayerNorm, the pre-LN block and the
pre-norm MLP branch with its residual connection.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.

Sources (page title, section):
  [Tour]    "Megatron-LM" source tour (pyshine.com/megatron-lm),
            section "The Tensor-Parallel Primitives": with sequence
            parallelism on, layer norms run on sequence-sharded activations;
            gather_from_sequence_parallel_region all-gathers along the
            sequence in the forward and reduce-scatters gradients back.
  [Concept] "Megatron-LM / Megatron-Core" concept note, section
            "Key math / How it works": LN/dropout/residual split along the
            sequence, interleaved with tensor parallelism.

LayerNorm itself is not defined on the pages; the textbook form is used, per
row r over the hidden dimension h:
  mu = mean_h x,  var = mean_h (x - mu)^2 (biased),  rstd = 1 / sqrt(var + eps)
  xhat = (x - mu) rstd,  y = xhat * gamma + beta
and its exact gradient
  g = dy * gamma,  dx = rstd (g - mean_h g - xhat mean_h(g xhat)),
  dgamma = sum_r dy xhat,  dbeta = sum_r dy.
Under sequence parallelism each shard s holds rows [s T/t, (s+1) T/t) and
computes partial dgamma_s, dbeta_s; summing them over shards (an all-reduce
the pages leave implicit) gives the full gradients.
"""
from __future__ import annotations

import numpy as np

from . import mlp as _mlp


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def layernorm_fwd(X, gamma, beta, eps):
    """Returns (Xn, mean, rstd)."""
    X, gamma, beta = _f64(X), _f64(gamma), _f64(beta)
    mu = X.mean(axis=1)
    xc = X - mu[:, None]
    var = (xc * xc).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = xc * rstd[:, None]
    return xhat * gamma + beta, mu, rstd


def layernorm_bwd(X, gamma, mean, rstd, dXn):
    """Returns (dX, dgamma, dbeta) for the given saved statistics."""
    X, gamma, mean, rstd, dXn = map(_f64, (X, gamma, mean, rstd, dXn))
    xhat = (X - mean[:, None]) * rstd[:, None]
    g = dXn * gamma
    dX = rstd[:, None] * (g - g.mean(axis=1, keepdims=True)
                          - xhat * (g * xhat).mean(axis=1, keepdims=True))
    return dX, (dXn * xhat).sum(axis=0), dXn.sum(axis=0)


def layernorm_sp_fwd(X, gamma, beta, eps, t):
    """LN on t sequence shards, then the emulated all-gather (concatenation)."""
    X = _f64(X)
    T = X.shape[0]
    assert T % t == 0
    ts = T // t
    shards = [layernorm_fwd(X[s * ts:(s + 1) * ts], gamma, beta, eps) for s in range(t)]
    Xn = np.concatenate([sh[0] for sh in shards], axis=0)        # all-gather
    mu = np.concatenate([sh[1] for sh in shards])
    rstd = np.concatenate([sh[2] for sh in shards])
    return Xn, mu, rstd


def layernorm_sp_bwd(X, gamma, mean, rstd, dXn, t):
    """Per-shard LN backward; dgamma/dbeta partials summed over the t shards."""
    X, dXn = _f64(X), _f64(dXn)
    T, H = X.shape
    ts = T // t
    dX = np.empty_like(X)
    dgamma = np.zeros(H)
    dbeta = np.zeros(H)
    for s in range(t):
        r = slice(s * ts, (s + 1) * ts)
        dXs, dg_s, db_s = layernorm_bwd(X[r], gamma, mean[r], rstd[r], dXn[r])
        dX[r] = dXs
        dgamma = dgamma + dg_s                                   # all-reduce of partials
        dbeta = dbeta + db_s
    return dX, dgamma, dbeta


# ---------------------------------------------------------------- pre-LN block, Y = MLP(LN(X))
# ``store`` (default exact) is applied to the LN output, which the block keeps as
# fc1's and dW1's GEMM input, and passed on to the MLP (see ``mlp.mlp_forward``).
def block_forward(X, gamma, beta, eps, W1, b1, W2, b2, act, t, store=None):
    S = store or _mlp._identity
    Xn, mu, rstd = layernorm_fwd(X, gamma, beta, eps)
    Xn = S(Xn)
    out = _mlp.mlp_forward(Xn, W1, b1, W2, b2, act, store)
    out.update(Xn=Xn, mean=mu, rstd=rstd)
    return out


def block_backward(X, gamma, beta, eps, W1, b1, W2, dY, act, t, store=None):
    S = store or _mlp._identity
    Xn, mu, rstd = layernorm_fwd(X, gamma, beta, eps)
    g = _mlp.mlp_backward(S(Xn), W1, b1, W2, dY, act, store)
    dX, dgamma, dbeta = layernorm_bwd(X, gamma, mu, rstd, g["dX"])
    g.update(dXn=g["dX"], dX=dX, dgamma=dgamma, dbeta=dbeta)
    return g


def block_sp_forward_backward(X, gamma, beta, eps, W1, b1, W2, b2, dY, act, t):
    """The pre-LN block as t ranks with sequence + tensor parallelism run it.

    Forward: LN on seq shard s -> all-gather along the sequence -> each TP rank
    i computes its partial P_i [T, H] -> reduce-scatter: seq shard s of Y is
    rows s of sum_i P_i (+ b2).  Backward: all-gather the seq shards of dY ->
    each rank's partial dXn_i -> reduce-scatter to dXn_s -> LN backward per
    shard, dgamma/dbeta partials all-reduced.
    """
    X, dY = _f64(X), _f64(dY)
    W1, W2, b1, b2 = _f64(W1), _f64(W2), _f64(b1), _f64(b2)
    T, H = X.shape
    ts = T // t
    Fs = W2.shape[2]
    rows = [slice(s * ts, (s + 1) * ts) for s in range(t)]
    # forward: per-shard LN, then gather
    ln = [layernorm_fwd(X[r], gamma, beta, eps) for r in rows]
    Xn = np.concatenate([l[0] for l in ln], axis=0)
    partials, dXn_parts = [], []
    dYfull = np.concatenate([dY[r] for r in rows], axis=0)         # all-gather of dY
    dW1 = np.zeros_like(W1)
    dW2 = np.zeros_like(W2)
    for i in range(t):
        if act == "swiglu":
            Gi, Ui = Xn @ W1[i, 0].T, Xn @ W1[i, 1].T
            Ai = _mlp.silu(Gi) * Ui
            dAi = dYfull @ W2[i]
            dGi = dAi * Ui * _mlp.silu_grad(Gi)
            dUi = dAi * _mlp.silu(Gi)
            dW1[i, 0], dW1[i, 1] = dGi.T @ Xn, dUi.T @ Xn
            dXn_parts.append(dGi @ W1[i, 0] + dUi @ W1[i, 1])
        else:
            Zi = Xn @ W1[i].T
            if b1 is not None:
                Zi = Zi + b1[i * Fs:(i + 1) * Fs]
            Ai = _mlp.gelu_tanh(Zi)
            dZi = (dYfull @ W2[i]) * _mlp.gelu_tanh_grad(Zi)
            dW1[i] = dZi.T @ Xn
            dXn_parts.append(dZi @ W1[i])
        partials.append(Ai @ W2[i].T)
        dW2[i] = dYfull.T @ Ai
    Y = np.empty((T, H))
    dXn = np.empty((T, H))
    for r in rows:                                                  # reduce-scatters
        acc = np.zeros((ts, H))
        for P in partials:
            acc = acc + P[r]
        Y[r] = acc if b2 is None else acc + b2
        accd = np.zeros((ts, H))
        for P in dXn_parts:
            accd = accd + P[r]
        dXn[r] = accd
    dX = np.empty((T, H))
    dgamma = np.zeros(H)
    dbeta = np.zeros(H)
    for s, r in enumerate(rows):
        dXs, dg, db = layernorm_bwd(X[r], gamma, ln[s][1], ln[s][2], dXn[r])
        dX[r] = dXs
        dgamma, dbeta = dgamma + dg, dbeta + db
    return {"Y": Y, "Xn": Xn, "dXn": dXn, "dX": dX, "dW1": dW1, "dW2": dW2,
            "dgamma": dgamma, "dbeta": dbeta}


# ---------------------------------------------------------------- pre-norm MLP branch
# [Tour] §The Transformer Stack: the layer runs its MLP branch on the layer-normalised
# input and adds the branch input back through a residual connection.  Dropout is left
# out (it is stochastic), so with the branch input X:
#   out = X + MLP(LN(X)),   dX = dout + LN'(dXn)   (dXn: the MLP's input gradient)
def branch_forward(X, gamma, beta, eps, W1, b1, W2, b2, act, t, store=None):
    out = block_forward(X, gamma, beta, eps, W1, b1, W2, b2, act, t, store)
    out["Y"] = _f64(X) + out["Y"]
    return out


def branch_backward(X, gamma, beta, eps, W1, b1, W2, dY, act, t, store=None):
    g = block_backward(X, gamma, beta, eps, W1, b1, W2, dY, act, t, store)
    g["dX"] = _f64(dY) + g["dX"]  # the residual path carries dout unchanged
    return g


def branch_rows(X, gamma, beta, eps, W1, b1, W2, b2, dY, rows, act, store=None):
    """Y[rows] and dX[rows] of the pre-norm branch."""
    rows = np.asarray(rows)
    r = block_rows(X, gamma, beta, eps, W1, b1, W2, b2, dY, rows, act, store)
    r["Y"] = _f64(X)[rows] + r["Y"]
    r["dX"] = _f64(dY)[rows] + r["dX"]
    return r


def block_rows(X, gamma, beta, eps, W1, b1, W2, b2, dY, rows, act, store=None):
    """Y[rows] and dX[rows] of the pre-LN block (row-separable end to end)."""
    S = store or _mlp._identity
    rows = np.asarray(rows)
    Xr = _f64(X)[rows]
    Xn, mu, rstd = layernorm_fwd(Xr, gamma, beta, eps)
    r = _mlp.mlp_rows(S(Xn), W1, b1, W2, b2, _f64(dY)[rows], np.arange(len(rows)), act, store)
    dX, _, _ = layernorm_bwd(Xr, gamma, mu, rstd, r["dX"])
    return {"Y": r["Y"], "dXn": r["dX"], "dX": dX}


def block_ffn_cols(X, gamma, beta, eps, W1, b1, W2, dY, cols, act, store=None):
    """Sampled ffn-feature gradients of the pre-LN block (fc1 sees LN(X))."""
    S = store or _mlp._identity
    Xn, _, _ = layernorm_fwd(X, gamma, beta, eps)
    return _mlp.mlp_ffn_cols(S(Xn), W1, b1, W2, dY, cols, act, store)
