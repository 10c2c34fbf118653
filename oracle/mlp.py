"""fp64 CPU oracle of the tensor-parallel transformer MLP block.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.  The
library never calls it, and it shares no code with the CUDA path.

Sources (page title, section):
  [Tour]    "Megatron-LM" source tour (pyshine.com/megatron-lm),
            section "The Tensor-Parallel Primitives" and "The Transformer Stack".
  [Concept] "Megatron-LM / Megatron-Core" concept note (research hub),
            section "Key math / How it works".

What is computed.  [Tour] §Tensor-Parallel Primitives: fc1 is a
ColumnParallelLinear (weight split along its output dimension, every rank
sees the full input), fc2 a RowParallelLinear (weight split along its input
dimension, partial sums all-reduced at the end); chaining the two needs one
all-reduce per block.  [Concept] §Key math names the conjugate operators:
f = identity forward / all-reduce backward (in front of fc1), g = all-reduce
forward / identity backward (after fc2).  [Tour] §Transformer Stack: a fused
bias-GELU sits between fc1 and fc2; gated variants (SwiGLU) swap the
activation for a gate/up pair multiplied together.  Tensor parallelism only
re-associates sums, so the unsharded definition is the exact result:

  GELU:    Z = X W1^T + b1,  A = gelu_tanh(Z),          Y = A W2^T + b2
  SwiGLU:  G = X Wg^T, U = X Wu^T, A = silu(G) * U,     Y = A W2^T
  backward, dY given:
    db2 = sum_t dY,  dA = dY W2,  dW2 = dY^T A
    GELU:   dZ = dA * gelu'(Z)
    SwiGLU: dG = dA * U * silu'(G),  dU = dA * silu(G)
    db1 = sum_t dZ,  dW1 = dZ^T X,  dX = dZ W1

Readings where the pages are silent (each is listed with its reason in the
design notes): GELU is the tanh form and its derivative the exact derivative
of that form; SwiGLU is silu(x Wg^T) * (x Wu^T) with each shard holding
[gate_i; up_i]; b1 is split with W1's output rows; b2 is added once, after the
sum over shards; LayerNorm uses the biased variance with eps inside the root.

Each public function works on float64 numpy arrays whose values are the bf16
inputs converted exactly.  A matmul (``@``) and ``sum``/``mean`` are the only
library primitives used as steps.
"""
from __future__ import annotations

import math

import numpy as np

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_GELU_CUBIC = 0.044715


# ---------------------------------------------------------------- activations
def gelu_tanh(z):
    """Tanh-form GELU: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(_SQRT_2_OVER_PI * (z + _GELU_CUBIC * z ** 3)))


def gelu_tanh_grad(z):
    """d/dz of :func:`gelu_tanh` (the derivative of the tanh form itself)."""
    z = np.asarray(z, dtype=np.float64)
    th = np.tanh(_SQRT_2_OVER_PI * (z + _GELU_CUBIC * z ** 3))
    du = _SQRT_2_OVER_PI * (1.0 + 3.0 * _GELU_CUBIC * z ** 2)
    return 0.5 * (1.0 + th) + 0.5 * z * (1.0 - th * th) * du


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    """x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def silu_grad(x):
    """sigmoid(x) (1 + x (1 - sigmoid(x)))."""
    s = sigmoid(x)
    return s * (1.0 + np.asarray(x, dtype=np.float64) * (1.0 - s))


def _identity(z):
    return np.asarray(z, dtype=np.float64)


def _identity_grad(z):
    return np.ones_like(np.asarray(z, dtype=np.float64))


# "identity" exists only so that a test can pin the two GEMMs against the
# closed form Y = X (W2 W1)^T + W2 b1 + b2; the block never uses it.
_POINTWISE = {"gelu": (gelu_tanh, gelu_tanh_grad), "identity": (_identity, _identity_grad)}


# ---------------------------------------------------------------- layouts
def full_w1(W1, act):
    """Shard-major fc1 weight -> unsharded matrices in ``nn.Linear`` (out x in) form.

    GELU: [t, Fs, H] -> W1f [F, H] with row i*Fs + j = shard i, row j
    (the column split of [Tour] §Tensor-Parallel Primitives).
    SwiGLU: [t, 2, Fs, H] -> (Wg [F, H], Wu [F, H]).
    """
    W1 = np.asarray(W1, dtype=np.float64)
    if act == "swiglu":
        t, two, Fs, H = W1.shape
        assert two == 2
        return W1[:, 0].reshape(t * Fs, H), W1[:, 1].reshape(t * Fs, H)
    t, Fs, H = W1.shape
    return W1.reshape(t * Fs, H)


def full_w2(W2):
    """Shard-major fc2 weight [t, H, Fs] -> unsharded W2f [H, F].

    Row-parallel split along the input dimension: W2f[:, i*Fs + j] = W2[i, :, j].
    """
    W2 = np.asarray(W2, dtype=np.float64)
    return np.concatenate([W2[i] for i in range(W2.shape[0])], axis=1)


def shard_w1_grad(dW1f, t, act):
    """Inverse of :func:`full_w1` for gradients (fp64)."""
    if act == "swiglu":
        dWg, dWu = dW1f
        F, H = dWg.shape
        Fs = F // t
        return np.stack([dWg.reshape(t, Fs, H), dWu.reshape(t, Fs, H)], axis=1)
    F, H = dW1f.shape
    return dW1f.reshape(t, F // t, H)


def shard_w2_grad(dW2f, t):
    """Inverse of :func:`full_w2` for gradients: [H, F] -> [t, H, Fs]."""
    H, F = dW2f.shape
    Fs = F // t
    return np.stack([dW2f[:, i * Fs:(i + 1) * Fs] for i in range(t)], axis=0)


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- plain (unsharded) path
def mlp_forward(X, W1, b1, W2, b2, act="gelu", store=None):
    """Unsharded forward.  Returns Y and the saved activations.

    GELU -> {"Y", "Z", "A"};  SwiGLU -> {"Y", "G", "U", "A"} (b1, b2 unused/None).
    ``store`` (default: exact) is applied to every activation the block keeps as a
    GEMM input -- A, and the saved Z or G, U -- e.g. ``bf16.round_bf16``.
    """
    S = store or _identity
    X, b1, b2 = _f64(X), _f64(b1), _f64(b2)
    W2f = full_w2(W2)
    out = {}
    if act == "swiglu":
        Wg, Wu = full_w1(W1, act)
        G = X @ Wg.T
        U = X @ Wu.T
        A = S(silu(G) * U)
        out.update(G=S(G), U=S(U))
    else:
        fn, _ = _POINTWISE[act]
        W1f = full_w1(W1, act)
        Z = X @ W1f.T
        if b1 is not None:
            Z = Z + b1
        A = S(fn(Z))
        out["Z"] = S(Z)
    Y = A @ W2f.T
    if b2 is not None:
        Y = Y + b2
    out.update(A=A, Y=Y)
    return out


def mlp_backward(X, W1, b1, W2, dY, act="gelu", store=None, recompute=False):
    """Unsharded backward (recomputes the forward activations itself).

    Returns dX [T, H], dW1 (shard-major like W1), dW2 [t, H, Fs], db1 [F] (or
    None without bias), db2 [H].  With ``store``, the derivative uses the stored
    Z (or G, U), dW2 the stored A, and dZ is stored before its three uses.

    ``recompute`` (selective activation recomputation, [Concept] §Key math): dW2 uses
    A recomputed from the stored Z (or G, U) instead of the A the forward kept, i.e.
    store(act(store(Z))).  Without ``store`` the two are the same number.
    """
    S = store or _identity
    X, b1, dY = _f64(X), _f64(b1), _f64(dY)
    t = np.asarray(W2).shape[0]
    fwd = mlp_forward(X, W1, b1, W2, None, act, store)
    A = fwd["A"]
    if recompute:
        if act == "swiglu":
            A = S(silu(fwd["G"]) * fwd["U"])
        else:
            A = S(_POINTWISE[act][0](fwd["Z"]))
    W2f = full_w2(W2)
    db2 = dY.sum(axis=0)
    dA = dY @ W2f
    dW2f = dY.T @ A
    if act == "swiglu":
        Wg, Wu = full_w1(W1, act)
        G, U = fwd["G"], fwd["U"]
        dG = S(dA * U * silu_grad(G))
        dU = S(dA * silu(G))
        dX = dG @ Wg + dU @ Wu
        dW1 = shard_w1_grad((dG.T @ X, dU.T @ X), t, act)
        db1 = None
    else:
        _, dfn = _POINTWISE[act]
        W1f = full_w1(W1, act)
        dZ = S(dA * dfn(fwd["Z"]))
        dX = dZ @ W1f
        dW1 = shard_w1_grad(dZ.T @ X, t, act)
        db1 = dZ.sum(axis=0) if b1 is not None else None
    return {"dX": dX, "dW1": dW1, "dW2": shard_w2_grad(dW2f, t), "db1": db1, "db2": db2}


# ---------------------------------------------------------------- gradient accumulation
PARAM_GRADS = ("dW1", "dW2", "db1", "db2", "dgamma", "dbeta")


def accumulate_param_grads(main, grads):
    """One micro-batch of gradient accumulation ([Tour] §Tensor-Parallel Primitives:
    the linear layers' autograd function accumulates the weight gradients).

    ``main`` holds the main-grad buffers carried across micro-batches; the result is
    main[k] + grads[k] for every parameter gradient (``PARAM_GRADS``) present in both.
    Activation gradients (dX, dXn) are per micro-batch and are not accumulated.
    Reading: the step's loss is the sum of the micro-batches' losses, so its parameter
    gradient is the plain sum of theirs (no averaging by the micro-batch count).
    """
    out = {}
    for k in PARAM_GRADS:
        if main.get(k) is not None and grads.get(k) is not None:
            out[k] = _f64(main[k]) + _f64(grads[k])
    return out


# ---------------------------------------------------------------- explicitly sharded path
def mlp_forward_sharded(X, W1, b1, W2, b2, act="gelu"):
    """Forward as t tensor-parallel ranks would run it, each with its own buffers.

    Rank i: f (identity) hands it the full X; its column shard of fc1 gives
    Z_i, A_i; its row shard of fc2 gives a partial P_i [T, H].  g then sums
    the t partials (the all-reduce) and b2 is added once.
    """
    X, b1, b2 = _f64(X), _f64(b1), _f64(b2)
    W1, W2 = _f64(W1), _f64(W2)
    t = W2.shape[0]
    Fs = W2.shape[2]
    partials = []
    for i in range(t):
        Xi = X.copy()                                   # f forward: identity
        if act == "swiglu":
            Gi = Xi @ W1[i, 0].T
            Ui = Xi @ W1[i, 1].T
            Ai = silu(Gi) * Ui
        else:
            fn, _ = _POINTWISE[act]
            Zi = Xi @ W1[i].T
            if b1 is not None:
                Zi = Zi + b1[i * Fs:(i + 1) * Fs]
            Ai = fn(Zi)
        partials.append(Ai @ W2[i].T)                   # row-parallel partial
    Y = np.zeros_like(partials[0])
    for P in partials:                                  # g forward: all-reduce
        Y = Y + P
    if b2 is not None:
        Y = Y + b2
    return Y


def mlp_backward_sharded(X, W1, b1, W2, dY, act="gelu"):
    """Backward as t ranks would run it: g backward hands every rank the same
    dY; each rank forms its own weight gradients and a partial dX_i; f
    backward all-reduces the partials."""
    X, b1, dY = _f64(X), _f64(b1), _f64(dY)
    W1, W2 = _f64(W1), _f64(W2)
    t = W2.shape[0]
    Fs = W2.shape[2]
    dW1 = np.zeros_like(W1)
    dW2 = np.zeros_like(W2)
    db1 = np.zeros(t * Fs) if (b1 is not None and act != "swiglu") else None
    dX_parts = []
    for i in range(t):
        dYi = dY.copy()                                 # g backward: identity
        if act == "swiglu":
            Gi = X @ W1[i, 0].T
            Ui = X @ W1[i, 1].T
            Ai = silu(Gi) * Ui
            dAi = dYi @ W2[i]
            dGi = dAi * Ui * silu_grad(Gi)
            dUi = dAi * silu(Gi)
            dW1[i, 0] = dGi.T @ X
            dW1[i, 1] = dUi.T @ X
            dX_parts.append(dGi @ W1[i, 0] + dUi @ W1[i, 1])
        else:
            fn, dfn = _POINTWISE[act]
            Zi = X @ W1[i].T
            if b1 is not None:
                Zi = Zi + b1[i * Fs:(i + 1) * Fs]
            Ai = fn(Zi)
            dAi = dYi @ W2[i]
            dZi = dAi * dfn(Zi)
            dW1[i] = dZi.T @ X
            if db1 is not None:
                db1[i * Fs:(i + 1) * Fs] = dZi.sum(axis=0)
            dX_parts.append(dZi @ W1[i])
        dW2[i] = dYi.T @ Ai
    dX = np.zeros_like(dX_parts[0])
    for P in dX_parts:                                  # f backward: all-reduce
        dX = dX + P
    return {"dX": dX, "dW1": dW1, "dW2": dW2, "db1": db1, "db2": dY.sum(axis=0)}


# ---------------------------------------------------------------- sampled outputs
def mlp_rows(X, W1, b1, W2, b2, dY, rows, act="gelu", store=None):
    """Y[rows] and dX[rows]: every output row depends only on its own input row."""
    rows = np.asarray(rows)
    Xr = _f64(X)[rows]
    dYr = _f64(dY)[rows]
    fwd = mlp_forward(Xr, W1, b1, W2, b2, act, store)
    bwd = mlp_backward(Xr, W1, b1, W2, dYr, act, store)
    return {"Y": fwd["Y"], "dX": bwd["dX"]}


def mlp_ffn_cols(X, W1, b1, W2, dY, cols, act="gelu", store=None):
    """Gradients of the sampled ffn features f (over all T tokens).

    Returns dW1_rows (GELU: [n, H]; SwiGLU: [n, 2, H] gate then up),
    dW2_cols [n, H] (column f of the unsharded dW2, i.e. W2-shard i, [:, j]),
    db1 [n] or None.  Feature f depends only on row f of W1 (gate and up),
    column f of W2 and entry f of b1.
    """
    S = store or _identity
    cols = np.asarray(cols)
    X, dY, b1 = _f64(X), _f64(dY), _f64(b1)
    W2f = full_w2(W2)[:, cols]                          # [H, n]
    dA = dY @ W2f                                       # [T, n]
    if act == "swiglu":
        Wg, Wu = full_w1(W1, act)
        G = X @ Wg[cols].T
        U = X @ Wu[cols].T
        A = S(silu(G) * U)
        G, U = S(G), S(U)
        dG = S(dA * U * silu_grad(G))
        dU = S(dA * silu(G))
        dW1 = np.stack([dG.T @ X, dU.T @ X], axis=1)
        db1 = None
    else:
        fn, dfn = _POINTWISE[act]
        W1f = full_w1(W1, act)
        Z = X @ W1f[cols].T
        if b1 is not None:
            Z = Z + b1[cols]
        A = S(fn(Z))
        dZ = S(dA * dfn(S(Z)))
        dW1 = dZ.T @ X
        db1 = dZ.sum(axis=0) if b1 is not None else None
    dW2 = (dY.T @ A).T                                  # [n, H]
    return {"dW1": dW1, "dW2": dW2, "db1": db1}
