"""Pins of the fp64 oracle to facts outside itself.

Every check here is something the pages or the mathematics fix without
re-typing the oracle's own formula:
  * tensor parallelism only re-associates sums ([Tour] "The Tensor-Parallel
    Primitives"; [Concept] "Key math": column->row pairing, conjugate f/g), so
    the explicitly sharded loop nest must equal the unsharded definition;
  * sequence-parallel LayerNorm with gather / reduce-scatter equals plain
    LayerNorm ([Tour] same section; [Concept] "Key math");
  * the tanh GELU is the textbook approximation of x*Phi(x) (max gap < 5e-4),
    is odd-symmetric in the sense gelu(x) - gelu(-x) = x, and tends to x / 0;
  * silu(x) - silu(-x) = x and silu(x) = x/2 (1 + tanh(x/2));
  * every gradient equals central finite differences of L = sum dY*Y;
  * with an identity activation the block collapses to a single affine map;
  * brute-force scalar loops over the shard-major arrays on tiny inputs.
A final group plants plausible mistakes into a copy of the oracle and checks
that at least one pin catches each.
"""
import math

import numpy as np
import pytest

from oracle import layernorm as ln
from oracle import mlp
from oracle.bf16 import round_bf16

RNG = np.random.default_rng(1234)


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


def _mlp_inputs(T, H, F, t, act, bias, scale=0.3, seed=0):
    r = np.random.default_rng(seed)
    Fs = F // t
    w1 = (t, 2, Fs, H) if act == "swiglu" else (t, Fs, H)
    return dict(
        X=r.standard_normal((T, H)),
        W1=r.standard_normal(w1) * scale,
        b1=r.standard_normal(F) * 0.1 if bias else None,
        W2=r.standard_normal((t, H, Fs)) * scale,
        b2=r.standard_normal(H) * 0.1 if bias else None,
        dY=r.standard_normal((T, H)),
    )


# ------------------------------------------------------------------ activations
def test_gelu_zero_and_odd_identity():
    x = np.linspace(-8, 8, 4001)
    assert mlp.gelu_tanh(0.0) == 0.0
    # tanh is odd => gelu(x) - gelu(-x) = x exactly (up to rounding)
    assert np.abs(mlp.gelu_tanh(x) - mlp.gelu_tanh(-x) - x).max() < 1e-14


def test_gelu_limits():
    assert abs(mlp.gelu_tanh(40.0) - 40.0) < 1e-12
    assert abs(mlp.gelu_tanh(-40.0)) < 1e-12


def test_gelu_tanh_approximates_erf_gelu():
    """Textbook: the tanh form approximates x*Phi(x) to within ~4.7e-4."""
    x = np.linspace(-10, 10, 20001)
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    gap = np.abs(mlp.gelu_tanh(x) - exact).max()
    assert 1e-4 < gap < 5e-4


def test_gelu_grad_matches_finite_difference():
    x = np.linspace(-6, 6, 1201)
    h = 1e-6
    fd = (mlp.gelu_tanh(x + h) - mlp.gelu_tanh(x - h)) / (2 * h)
    assert np.abs(mlp.gelu_tanh_grad(x) - fd).max() < 1e-8
    assert abs(mlp.gelu_tanh_grad(0.0) - 0.5) < 1e-15


def test_silu_identities_and_grad():
    x = np.linspace(-12, 12, 2401)
    assert np.abs(mlp.silu(x) - mlp.silu(-x) - x).max() < 1e-13
    assert np.abs(mlp.silu(x) - 0.5 * x * (1.0 + np.tanh(0.5 * x))).max() < 1e-13
    h = 1e-6
    fd = (mlp.silu(x + h) - mlp.silu(x - h)) / (2 * h)
    assert np.abs(mlp.silu_grad(x) - fd).max() < 1e-8
    assert mlp.silu(0.0) == 0.0 and mlp.silu_grad(0.0) == 0.5


# ------------------------------------------------------------------ sharding
@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("act,bias", [("gelu", True), ("gelu", False), ("swiglu", False)])
def test_sharded_equals_unsharded(t, act, bias):
    d = _mlp_inputs(16, 24, 64, t, act, bias, seed=t)
    y = mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)["Y"]
    ys = mlp.mlp_forward_sharded(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)
    assert _rel(ys, y) < 1e-12
    g = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    gs = mlp.mlp_backward_sharded(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    for k in ("dX", "dW1", "dW2", "db2") + (("db1",) if (bias and act == "gelu") else ()):
        assert _rel(gs[k], g[k]) < 1e-12, k


def test_b2_added_once_not_per_shard():
    d = _mlp_inputs(4, 8, 16, 4, "gelu", True, seed=3)
    zero_w2 = np.zeros_like(d["W2"])
    y = mlp.mlp_forward_sharded(d["X"], d["W1"], d["b1"], zero_w2, d["b2"], "gelu")
    assert np.allclose(y, np.broadcast_to(d["b2"], y.shape), rtol=0, atol=1e-15)


# ------------------------------------------------------------------ brute force
def _brute_forward(X, W1, b1, W2, b2, act):
    """Scalar loops straight over the shard-major arrays (tiny shapes only)."""
    T, H = X.shape
    t, _, Fs = W2.shape
    Y = np.zeros((T, H))
    for r in range(T):
        for h in range(H):
            s = 0.0 if b2 is None else float(b2[h])
            for i in range(t):
                for j in range(Fs):
                    if act == "swiglu":
                        g = sum(X[r, k] * W1[i, 0, j, k] for k in range(H))
                        u = sum(X[r, k] * W1[i, 1, j, k] for k in range(H))
                        a = g / (1.0 + math.exp(-g)) * u
                    else:
                        z = sum(X[r, k] * W1[i, j, k] for k in range(H))
                        if b1 is not None:
                            z += b1[i * Fs + j]
                        a = 0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0)))
                    s += a * W2[i, h, j]
            Y[r, h] = s
    return Y


@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_forward_against_brute_force_loops(act, bias):
    d = _mlp_inputs(3, 4, 6, 2, act, bias, scale=0.5, seed=7)
    ref = _brute_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)
    y = mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)["Y"]
    # the brute force uses the exact erf GELU: allow the tanh-approximation gap
    tol = 5e-4 * 6 * 0.5 * 2 if act == "gelu" else 1e-13
    assert np.abs(y - ref).max() < tol


def test_identity_activation_closed_form():
    """With act = identity: Y = X (W2 W1)^T + W2 b1 + b2 (a different association)."""
    d = _mlp_inputs(8, 12, 16, 4, "gelu", True, seed=11)
    W1f = mlp.full_w1(d["W1"], "gelu")
    W2f = mlp.full_w2(d["W2"])
    closed = d["X"] @ (W2f @ W1f).T + W2f @ d["b1"] + d["b2"]
    y = mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], "identity")["Y"]
    assert _rel(y, closed) < 1e-12
    ys = mlp.mlp_forward_sharded(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], "identity")
    assert _rel(ys, closed) < 1e-12


def test_layout_helpers_roundtrip():
    d = _mlp_inputs(2, 8, 12, 3, "swiglu", False, seed=2)
    t = 3
    g, u = mlp.full_w1(d["W1"], "swiglu")
    assert np.array_equal(mlp.shard_w1_grad((g, u), t, "swiglu"), d["W1"])
    assert np.array_equal(mlp.shard_w2_grad(mlp.full_w2(d["W2"]), t), d["W2"])
    # column f = i*Fs + j of the unsharded W2 is shard i, column j
    W2f = mlp.full_w2(d["W2"])
    assert np.array_equal(W2f[:, 1 * 4 + 2], d["W2"][1, :, 2])


# ------------------------------------------------------------------ finite differences
def _loss(d, act):
    y = mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)["Y"]
    return float((d["dY"] * y).sum())


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("act,bias", [("gelu", True), ("gelu", False), ("swiglu", False)])
def test_backward_matches_finite_differences(t, act, bias):
    d = _mlp_inputs(8, 16, 32, t, act, bias, seed=100 + t)
    g = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    names = {"X": "dX", "W1": "dW1", "W2": "dW2", "b1": "db1", "b2": "db2"}
    h = 1e-6
    r = np.random.default_rng(t)
    for p, gname in names.items():
        if d[p] is None:
            continue
        flat = d[p].reshape(-1)
        idx = r.choice(flat.size, size=min(12, flat.size), replace=False)
        for k in idx:
            old = flat[k]
            flat[k] = old + h
            lp = _loss(d, act)
            flat[k] = old - h
            lm = _loss(d, act)
            flat[k] = old
            fd = (lp - lm) / (2 * h)
            an = g[gname].reshape(-1)[k]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (p, k, fd, an)


def test_backward_is_linear_in_dY():
    d = _mlp_inputs(8, 16, 32, 2, "gelu", True, seed=5)
    dY2 = np.random.default_rng(9).standard_normal(d["dY"].shape)
    a = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], "gelu")
    b = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], dY2, "gelu")
    c = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"] + dY2, "gelu")
    for k in ("dX", "dW1", "dW2", "db1", "db2"):
        assert _rel(c[k], a[k] + b[k]) < 1e-12


# ------------------------------------------------------------------ gradient accumulation
def _split_tokens(a, parts):
    return np.split(np.asarray(a), parts, axis=0)


@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_accumulated_micro_batches_equal_concatenated_batch(act, bias):
    """The gradient of a loss summed over tokens is the sum over any split of the tokens:
    accumulating three micro-batches from zeroed buffers gives the whole batch's
    parameter gradients (the batch backward is a separate computation, not a sum)."""
    d = _mlp_inputs(12, 16, 32, 2, act, bias, seed=21)
    full = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    main = {k: np.zeros_like(full[k]) for k in mlp.PARAM_GRADS if full.get(k) is not None}
    for Xk, dYk in zip(_split_tokens(d["X"], 3), _split_tokens(d["dY"], 3)):
        g = mlp.mlp_backward(Xk, d["W1"], d["b1"], d["W2"], dYk, act)
        main = mlp.accumulate_param_grads(main, g)
    assert set(main) == ({"dW1", "dW2", "db1", "db2"} if bias else {"dW1", "dW2", "db2"})
    for k, v in main.items():
        assert _rel(v, full[k]) < 1e-12, k


def test_accumulation_adds_to_existing_main_grads_and_skips_dX():
    d = _mlp_inputs(8, 16, 32, 2, "gelu", True, seed=22)
    g = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], "gelu")
    r = np.random.default_rng(23)
    main0 = {k: r.standard_normal(np.shape(g[k])) for k in ("dW1", "dW2", "db1", "db2")}
    main0["dX"] = r.standard_normal(g["dX"].shape)
    out = mlp.accumulate_param_grads(main0, g)
    assert "dX" not in out
    for k in ("dW1", "dW2", "db1", "db2"):
        assert np.array_equal(out[k], main0[k] + g[k]), k
    # an all-zero micro-batch (T = 0 has no tokens) leaves the buffers as they are
    z = mlp.accumulate_param_grads(main0, {k: np.zeros_like(main0[k]) for k in main0})
    for k in ("dW1", "dW2", "db1", "db2"):
        assert np.array_equal(z[k], main0[k]), k


def test_accumulated_layernorm_params_equal_concatenated_batch():
    X, gamma, beta, _ = _ln_inputs(8, 16, 24)
    d = _mlp_inputs(8, 16, 32, 2, "swiglu", False, seed=25)
    full = ln.block_backward(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], d["dY"], "swiglu", 2)
    main = {"dgamma": np.zeros(16), "dbeta": np.zeros(16), "dW1": np.zeros_like(full["dW1"])}
    for Xk, dYk in zip(_split_tokens(X, 2), _split_tokens(d["dY"], 2)):
        g = ln.block_backward(Xk, gamma, beta, 1e-5, d["W1"], None, d["W2"], dYk, "swiglu", 2)
        main = mlp.accumulate_param_grads(main, g)
    for k in ("dgamma", "dbeta", "dW1"):
        assert _rel(main[k], full[k]) < 1e-12, k


# ------------------------------------------------------------------ LayerNorm
def _ln_inputs(T, H, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((T, H)) * 2.0 + 0.5, 1.0 + 0.1 * r.standard_normal(H),
            0.02 * r.standard_normal(H), r.standard_normal((T, H)))


def test_layernorm_unit_gamma_invariants():
    X, _, _, _ = _ln_inputs(16, 64, 1)
    eps = 1e-5
    Xn, mu, rstd = ln.layernorm_fwd(X, np.ones(64), np.zeros(64), eps)
    var = X.var(axis=1)  # numpy's biased variance, independent of the oracle's
    assert np.abs(Xn.mean(axis=1)).max() < 1e-14
    assert np.abs((Xn * Xn).mean(axis=1) - var / (var + eps)).max() < 1e-13
    assert np.abs(mu - X.mean(axis=1)).max() < 1e-14


def test_layernorm_shift_scale_invariance():
    X, gamma, beta, _ = _ln_inputs(8, 32, 2)
    a, _, _ = ln.layernorm_fwd(X, gamma, beta, 0.0)
    b, _, _ = ln.layernorm_fwd(3.0 * X - 7.0, gamma, beta, 0.0)
    assert np.abs(a - b).max() < 1e-12


def test_layernorm_backward_rowsum_zero_and_fd():
    X, gamma, beta, dXn = _ln_inputs(6, 24, 3)
    eps = 1e-5
    Xn, mu, rstd = ln.layernorm_fwd(X, gamma, beta, eps)
    dX, dgamma, dbeta = ln.layernorm_bwd(X, gamma, mu, rstd, dXn)
    assert np.abs(dX.sum(axis=1)).max() < 1e-12

    def loss(X_, g_, b_):
        return float((dXn * ln.layernorm_fwd(X_, g_, b_, eps)[0]).sum())

    h = 1e-6
    for arr, grad in ((X, dX), (gamma, dgamma), (beta, dbeta)):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for k in range(0, flat.size, max(1, flat.size // 10)):
            old = flat[k]
            flat[k] = old + h
            lp = loss(X, gamma, beta)
            flat[k] = old - h
            lm = loss(X, gamma, beta)
            flat[k] = old
            assert abs((lp - lm) / (2 * h) - gflat[k]) < 1e-6 * max(1.0, abs(gflat[k]))


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sp_layernorm_equals_layernorm(t):
    X, gamma, beta, dXn = _ln_inputs(32, 40, 4 + t)
    a = ln.layernorm_fwd(X, gamma, beta, 1e-5)
    b = ln.layernorm_sp_fwd(X, gamma, beta, 1e-5, t)
    for u, v in zip(a, b):
        assert _rel(v, u) < 1e-14
    ga = ln.layernorm_bwd(X, gamma, a[1], a[2], dXn)
    gb = ln.layernorm_sp_bwd(X, gamma, b[1], b[2], dXn, t)
    for u, v in zip(ga, gb):
        assert _rel(v, u) < 1e-12


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_sp_block_equals_plain_composition(act):
    t = 4
    d = _mlp_inputs(16, 24, 32, t, act, act == "gelu", seed=21)
    X, gamma, beta, _ = _ln_inputs(16, 24, 22)
    ref_f = ln.block_forward(X, gamma, beta, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], act, t)
    ref_b = ln.block_backward(X, gamma, beta, 1e-5, d["W1"], d["b1"], d["W2"], d["dY"], act, t)
    sp = ln.block_sp_forward_backward(X, gamma, beta, 1e-5, d["W1"], d["b1"], d["W2"],
                                      d["b2"], d["dY"], act, t)
    assert _rel(sp["Y"], ref_f["Y"]) < 1e-12
    for k in ("dX", "dW1", "dW2", "dgamma", "dbeta", "dXn"):
        assert _rel(sp[k], ref_b[k]) < 1e-12, k


def test_block_backward_matches_finite_differences():
    t = 2
    d = _mlp_inputs(6, 16, 16, t, "swiglu", False, seed=31)
    X, gamma, beta, _ = _ln_inputs(6, 16, 32)
    eps = 1e-5
    g = ln.block_backward(X, gamma, beta, eps, d["W1"], None, d["W2"], d["dY"], "swiglu", t)

    def loss():
        y = ln.block_forward(X, gamma, beta, eps, d["W1"], None, d["W2"], None, "swiglu", t)["Y"]
        return float((d["dY"] * y).sum())

    h = 1e-6
    for arr, grad in ((X, g["dX"]), (gamma, g["dgamma"]), (beta, g["dbeta"])):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for k in range(0, flat.size, max(1, flat.size // 8)):
            old = flat[k]
            flat[k] = old + h
            lp = loss()
            flat[k] = old - h
            lm = loss()
            flat[k] = old
            assert abs((lp - lm) / (2 * h) - gflat[k]) < 1e-6 * max(1.0, abs(gflat[k]))


# ------------------------------------------------------------------ selective recomputation
@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_recompute_changes_only_dW2_and_only_by_rounding(act, bias):
    """Recomputing A from the stored Z moves dW2 by bf16 rounding alone and touches no
    other gradient; in exact arithmetic it changes nothing."""
    d = _mlp_inputs(16, 32, 64, 2, act, bias, seed=71)
    a = (d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    for store in (None, round_bf16):
        keep = mlp.mlp_backward(*a, store=store)
        re = mlp.mlp_backward(*a, store=store, recompute=True)
        for k in ("dX", "dW1", "db1", "db2"):
            if keep[k] is not None:
                assert np.array_equal(keep[k], re[k]), (k, store)
        diff = re["dW2"] - keep["dW2"]
        rel = np.sqrt(np.mean(diff ** 2) / np.mean(keep["dW2"] ** 2))
        if store is None:
            assert rel == 0.0
        else:
            # a few bf16 units of A per term (RMS); a wrong activation is O(1) away
            assert 0.0 < rel < 1e-2, rel


def test_recompute_with_identity_activation_is_exact_under_rounding():
    """act = identity: A = store(Z) either way (rounding is idempotent), so the
    recomputed dW2 equals the kept one exactly."""
    d = _mlp_inputs(8, 16, 32, 2, "identity", True, seed=72)
    a = (d["X"], d["W1"], d["b1"], d["W2"], d["dY"], "identity")
    keep = mlp.mlp_backward(*a, store=round_bf16)
    re = mlp.mlp_backward(*a, store=round_bf16, recompute=True)
    assert np.array_equal(keep["dW2"], re["dW2"])


# ------------------------------------------------------------------ pre-norm MLP branch
@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_branch_backward_matches_finite_differences(act, bias):
    """dX of out = X + MLP(LN(X)) against central differences of sum(dY * out); the
    residual path makes dX differ from the block's by exactly the upstream gradient."""
    t = 2
    d = _mlp_inputs(6, 16, 16, t, act, bias, seed=61)
    X, gamma, beta, _ = _ln_inputs(6, 16, 62)
    eps = 1e-5
    g = ln.branch_backward(X, gamma, beta, eps, d["W1"], d["b1"], d["W2"], d["dY"], act, t)

    def loss():
        y = ln.branch_forward(X, gamma, beta, eps, d["W1"], d["b1"], d["W2"], d["b2"], act,
                              t)["Y"]
        return float((d["dY"] * y).sum())

    h = 1e-6
    for arr, grad in ((X, g["dX"]), (gamma, g["dgamma"]), (beta, g["dbeta"]),
                      (d["W2"], g["dW2"])):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for k in range(0, flat.size, max(1, flat.size // 8)):
            old = flat[k]
            flat[k] = old + h
            lp = loss()
            flat[k] = old - h
            lm = loss()
            flat[k] = old
            assert abs((lp - lm) / (2 * h) - gflat[k]) < 1e-6 * max(1.0, abs(gflat[k]))


def test_branch_with_zero_fc2_is_the_residual_alone():
    """W2 = 0: the MLP adds only b2, so out = X + b2 exactly and dX = dY exactly (the
    LayerNorm sees a zero gradient: dgamma = dbeta = 0)."""
    d = _mlp_inputs(8, 16, 32, 2, "gelu", True, seed=63)
    X, gamma, beta, _ = _ln_inputs(8, 16, 64)
    W2 = np.zeros_like(d["W2"])
    f = ln.branch_forward(X, gamma, beta, 1e-5, d["W1"], d["b1"], W2, d["b2"], "gelu", 2)
    g = ln.branch_backward(X, gamma, beta, 1e-5, d["W1"], d["b1"], W2, d["dY"], "gelu", 2)
    assert np.array_equal(f["Y"], X + d["b2"])
    assert np.array_equal(g["dX"], d["dY"])
    assert not g["dgamma"].any() and not g["dbeta"].any()


def test_branch_rows_match_full():
    d = _mlp_inputs(12, 16, 32, 2, "swiglu", False, seed=65)
    X, gamma, beta, _ = _ln_inputs(12, 16, 66)
    f = ln.branch_forward(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], None, "swiglu", 2)
    g = ln.branch_backward(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], d["dY"], "swiglu", 2)
    rows = [0, 5, 11]
    r = ln.branch_rows(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], None, d["dY"], rows,
                       "swiglu")
    assert _rel(r["Y"], f["Y"][rows]) < 1e-13
    assert _rel(r["dX"], g["dX"][rows]) < 1e-13


# ------------------------------------------------------------------ sampled modes
@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_sampled_rows_and_cols_match_full(act, bias):
    t = 4
    d = _mlp_inputs(20, 16, 32, t, act, bias, seed=41)
    fwd = mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)
    bwd = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    rows = np.array([0, 3, 19])
    r = mlp.mlp_rows(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], d["dY"], rows, act)
    assert _rel(r["Y"], fwd["Y"][rows]) < 1e-13
    assert _rel(r["dX"], bwd["dX"][rows]) < 1e-13
    cols = np.array([0, 7, 8, 31])
    c = mlp.mlp_ffn_cols(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], cols, act)
    Fs = 32 // t
    for n, f in enumerate(cols):
        i, j = divmod(int(f), Fs)
        assert _rel(c["dW2"][n], bwd["dW2"][i, :, j]) < 1e-13
        if act == "swiglu":
            assert _rel(c["dW1"][n, 0], bwd["dW1"][i, 0, j]) < 1e-13
            assert _rel(c["dW1"][n, 1], bwd["dW1"][i, 1, j]) < 1e-13
        else:
            assert _rel(c["dW1"][n], bwd["dW1"][i, j]) < 1e-13
            assert abs(c["db1"][n] - bwd["db1"][f]) < 1e-12


def test_block_sampled_matches_full():
    t = 2
    d = _mlp_inputs(8, 16, 16, t, "swiglu", False, seed=51)
    X, gamma, beta, _ = _ln_inputs(8, 16, 52)
    fwd = ln.block_forward(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], None, "swiglu", t)
    bwd = ln.block_backward(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], d["dY"], "swiglu", t)
    rows = np.array([1, 7])
    r = ln.block_rows(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], None, d["dY"], rows, "swiglu")
    assert _rel(r["Y"], fwd["Y"][rows]) < 1e-13
    assert _rel(r["dX"], bwd["dX"][rows]) < 1e-12
    c = ln.block_ffn_cols(X, gamma, beta, 1e-5, d["W1"], None, d["W2"], d["dY"], [0, 15], "swiglu")
    assert _rel(c["dW2"][1], bwd["dW2"][1, :, 7]) < 1e-13


# ------------------------------------------------------------------ planted mistakes
def _all_pins_pass():
    """A compact subset of the pins above, re-run against a mutated oracle."""
    try:
        test_gelu_zero_and_odd_identity()
        test_gelu_tanh_approximates_erf_gelu()
        test_gelu_grad_matches_finite_difference()
        test_silu_identities_and_grad()
        for act, bias in (("gelu", True), ("swiglu", False)):
            test_sharded_equals_unsharded(4, act, bias)
            test_backward_matches_finite_differences(2, act, bias)
            test_forward_against_brute_force_loops(act, bias)
        test_identity_activation_closed_form()
        test_layout_helpers_roundtrip()
        test_layernorm_backward_rowsum_zero_and_fd()
        test_sp_block_equals_plain_composition("swiglu")
        test_layernorm_unit_gamma_invariants()
        test_accumulated_micro_batches_equal_concatenated_batch("gelu", True)
        test_accumulation_adds_to_existing_main_grads_and_skips_dX()
        test_branch_backward_matches_finite_differences("gelu", True)
        test_branch_with_zero_fc2_is_the_residual_alone()
    except AssertionError:
        return False
    return True


def _mut_dropped_cubic(z):
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * z))


def _mut_silu_grad(x):
    s = mlp.sigmoid(x)
    return s * (1.0 - np.asarray(x) * (1.0 - s))


def _mut_full_w2(W2):
    W2 = np.asarray(W2, dtype=np.float64)
    return np.concatenate([W2[i] for i in range(W2.shape[0])], axis=1)[:, ::-1]


def _mut_layernorm_bwd(X, gamma, mean, rstd, dXn):
    xhat = (X - mean[:, None]) * rstd[:, None]
    g = dXn * gamma
    dX = rstd[:, None] * (g - g.mean(axis=1, keepdims=True))  # dropped xhat term
    return dX, (dXn * xhat).sum(axis=0), dXn.sum(axis=0)


def _mut_accumulate_overwrites(main, grads):
    return {k: np.asarray(grads[k], dtype=np.float64) for k in mlp.PARAM_GRADS
            if main.get(k) is not None and grads.get(k) is not None}


def _mut_accumulate_averages(main, grads):
    return {k: 0.5 * (np.asarray(main[k]) + np.asarray(grads[k])) for k in mlp.PARAM_GRADS
            if main.get(k) is not None and grads.get(k) is not None}


def _mut_branch_backward_drops_residual(X, gamma, beta, eps, W1, b1, W2, dY, act, t,
                                        store=None):
    return ln.block_backward(X, gamma, beta, eps, W1, b1, W2, dY, act, t, store)


def _mut_branch_forward_residual_sign(X, gamma, beta, eps, W1, b1, W2, b2, act, t, store=None):
    out = ln.block_forward(X, gamma, beta, eps, W1, b1, W2, b2, act, t, store)
    out["Y"] = out["Y"] - np.asarray(X, dtype=np.float64)
    return out


@pytest.mark.parametrize("target,attr,mutant", [
    (ln, "branch_backward", _mut_branch_backward_drops_residual),
    (ln, "branch_forward", _mut_branch_forward_residual_sign),
    (mlp, "accumulate_param_grads", _mut_accumulate_overwrites),
    (mlp, "accumulate_param_grads", _mut_accumulate_averages),
    (mlp, "gelu_tanh", _mut_dropped_cubic),
    (mlp, "silu_grad", _mut_silu_grad),
    (mlp, "full_w2", _mut_full_w2),
    (ln, "layernorm_bwd", _mut_layernorm_bwd),
])
def test_planted_mistake_is_caught(monkeypatch, target, attr, mutant):
    assert _all_pins_pass()
    monkeypatch.setattr(target, attr, mutant)
    if attr == "gelu_tanh":
        monkeypatch.setitem(mlp._POINTWISE, "gelu", (mutant, mlp.gelu_tanh_grad))
    assert not _all_pins_pass()


# ------------------------------------------------------------------ bf16 storage reading
def test_round_bf16_matches_torch_conversion():
    """Pinned to torch's own float32 -> bfloat16 conversion (round to nearest even)."""
    import torch
    from oracle.bf16 import round_bf16
    r = np.random.default_rng(5)
    x32 = np.concatenate([
        r.standard_normal(200000).astype(np.float32) * np.float32(10.0) ** r.integers(-30, 30, 200000).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, 1e-39, -2.5e-40], dtype=np.float32),
    ])
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_bf16(x32.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_bf16_ties_to_even_and_idempotent():
    from oracle.bf16 import round_bf16
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even significand (1)
    assert round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    x = np.random.default_rng(6).standard_normal(10000)
    once = round_bf16(x)
    assert np.array_equal(round_bf16(once), once)
    assert np.all(np.abs(once - x) <= np.abs(x) * 2.0 ** -8)


@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_store_hook_and_sampled_modes_agree(act, bias):
    from oracle.bf16 import identity, round_bf16
    t = 2
    d = _mlp_inputs(16, 16, 32, t, act, bias, seed=61)
    a = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act)
    b = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act, identity)
    for k in ("dX", "dW1", "dW2"):
        assert np.array_equal(a[k], b[k])
    full_b = mlp.mlp_backward(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], act, round_bf16)
    full_f = mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act, round_bf16)
    rows = np.array([0, 9, 15])
    r = mlp.mlp_rows(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], d["dY"], rows, act, round_bf16)
    assert _rel(r["Y"], full_f["Y"][rows]) < 1e-13 and _rel(r["dX"], full_b["dX"][rows]) < 1e-13
    cols = np.array([0, 15, 16, 31])
    c = mlp.mlp_ffn_cols(d["X"], d["W1"], d["b1"], d["W2"], d["dY"], cols, act, round_bf16)
    for n, f in enumerate(cols):
        i, j = divmod(int(f), 16)
        assert _rel(c["dW2"][n], full_b["dW2"][i, :, j]) < 1e-13
        want = full_b["dW1"][i, :, j] if act == "swiglu" else full_b["dW1"][i, j]
        assert _rel(c["dW1"][n], want) < 1e-13
    # the stored activations really are bf16 values
    assert np.array_equal(round_bf16(full_f["A"]), full_f["A"])
    # and the rounded result stays within a few bf16 units of the exact one
    assert _rel(full_f["Y"], mlp.mlp_forward(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], act)["Y"]) < 2e-2
