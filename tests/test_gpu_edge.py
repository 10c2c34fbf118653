"""GPU parity on the method's edge cases, element by element against the fp64 oracle.

* Saturated activations: fc1's weights scaled so that |Z| (GELU) and |G|, |U| (SwiGLU)
  reach ~110, far past the point (|x| ~ 88 for SiLU, |z| ~ 10 for the tanh-form GELU,
  whose exponent is 2 sqrt(2/pi) (z + 0.044715 z^3)) where exp overflows fp32: the
  activations, their derivatives and everything downstream must stay finite and on the
  oracle.
* Exact-zero blocks of X and dY rows and columns, crossing tile boundaries.
* LayerNorm rows that are constant (variance 0), carry a common offset of 1000 times
  their spread, or start with a 50-sigma outlier, through the LayerNorm alone and through
  the whole sequence-parallel block.
Every case at H = 64 (one 64-wide k-block, ragged N tiles) and H = 8192.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import (LN_EDGE_KINDS, MLPShape, make_inputs, make_ln_edge_rows, make_ln_grad,
                    make_saturating_inputs, make_zero_block_inputs)
from oracle import layernorm as oln

from _harness import check_full, fmt_rel, oracle_refs, run_gpu, to_f64

pytestmark = pytest.mark.gpu

SHAPES = [
    pytest.param(MLPShape(256, 64, 1024, 4, "gelu", True), id="gelu-bias-H64"),
    pytest.param(MLPShape(256, 8192, 1024, 4, "gelu", True), id="gelu-bias-H8192"),
    pytest.param(MLPShape(256, 64, 512, 2, "swiglu", False), id="swiglu-H64"),
    pytest.param(MLPShape(256, 8192, 512, 4, "swiglu", False), id="swiglu-H8192"),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_saturated_activations(shape):
    d = make_saturating_inputs(shape, 71)
    refs = oracle_refs(shape, d)
    exact = refs[0]
    # the case reaches the saturated tails (overflowing exp in fp32) on both sides
    if shape.act == "gelu":
        assert exact["Z"].min() < -60 and exact["Z"].max() > 60
    else:
        assert exact["G"].min() < -88 and exact["G"].max() > 88
    gpu = run_gpu(shape, d)
    rel = check_full(shape, gpu, refs)
    print(shape, fmt_rel(rel))


@pytest.mark.parametrize("shape", SHAPES)
def test_zero_blocks(shape):
    d = make_zero_block_inputs(shape, 72)
    gpu = run_gpu(shape, d)
    rel = check_full(shape, gpu, oracle_refs(shape, d))
    # zero rows of dY give exactly zero rows of dZ, hence of dX
    assert torch.count_nonzero(gpu["dX"][100:228]).item() == 0
    print(shape, fmt_rel(rel))


def _by_kind(T):
    kind = np.arange(T) % len(LN_EDGE_KINDS)
    return {name: kind == i for i, name in enumerate(LN_EDGE_KINDS)}


@pytest.mark.parametrize("H", [64, 8192])
def test_layernorm_edge_rows(H):
    """The LayerNorm forward and backward alone on the edge rows, each row kind checked
    on its own scale: mean within 1e-6 of the row's RMS, rstd within 1e-5 relative per
    row, Xn within one bf16 rounding plus 1e-3 of its RMS, dX within 1e-4 of its RMS."""
    T, t = 256, 4
    shape = MLPShape(T, H, 8 * t, t, "swiglu", False, sp_ln=True)
    d = make_inputs(shape, 73)
    X = make_ln_edge_rows(T, H, 73)
    dXn = make_ln_grad(shape, 73)
    dev = torch.device("cuda:0")
    h = mlpb.mlpb_create(mlpb.make_config(T, H, 8 * t, t, "swiglu", False, True, 1e-5))
    Xd, gm, bt = X.to(dev), d["gamma"].to(dev), d["beta"].to(dev)
    Xn = torch.empty_like(Xd)
    mean = torch.empty(T, device=dev)
    rstd = torch.empty(T, device=dev)
    mlpb.mlpb_layernorm_sp_fwd(h, Xd, gm, bt, Xn, mean, rstd)
    ws = torch.empty(mlpb.mlpb_workspace_size(h), dtype=torch.uint8, device=dev)
    dX = torch.empty((T, H), device=dev)
    dg = torch.empty(H, device=dev)
    db = torch.empty(H, device=dev)
    mlpb.mlpb_layernorm_sp_bwd(h, Xd, gm, mean, rstd, dXn.to(dev), dX, dg, db, ws)
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(h) == 0
    mlpb.mlpb_destroy(h)
    x64, g64, b64 = to_f64(X), to_f64(d["gamma"]), to_f64(d["beta"])
    rXn, rmu, rrs = oln.layernorm_sp_fwd(x64, g64, b64, 1e-5, t)
    rdX, rdg, rdb = oln.layernorm_sp_bwd(x64, g64, rmu, rrs, to_f64(dXn), t)
    got = {k: to_f64(v) for k, v in dict(Xn=Xn, mean=mean, rstd=rstd, dX=dX).items()}
    for name, rows in _by_kind(T).items():
        row_rms = np.sqrt(np.mean(x64[rows] ** 2, axis=1))
        assert np.all(np.abs(got["mean"][rows] - rmu[rows]) <= 1e-6 * row_rms), name
        assert np.all(np.abs(got["rstd"][rows] - rrs[rows]) <= 1e-5 * rrs[rows]), name
        ref = rXn[rows]
        bound = np.abs(ref) * 2.0 ** -8 + 1e-3 * np.sqrt(np.mean(ref ** 2))
        ok = np.abs(got["Xn"][rows] - ref) <= bound
        assert ok.all(), f"{name}: {int((~ok).sum())} Xn entries beyond one bf16 rounding"
        ref = rdX[rows]
        err = np.abs(got["dX"][rows] - ref).max()
        assert err <= 1e-4 * np.sqrt(np.mean(ref ** 2)), f"{name}: dX {err:.3e}"
    # constant rows normalise to exactly beta (xhat = 0)
    const = _by_kind(T)["constant"]
    assert np.array_equal(got["Xn"][const], np.broadcast_to(b64, got["Xn"][const].shape))
    for name, g, r in (("dgamma", to_f64(dg), rdg), ("dbeta", to_f64(db), rdb)):
        err = np.abs(g - r).max()
        assert err <= 1e-4 * np.sqrt(np.mean(r ** 2)), f"{name}: {err:.3e}"


@pytest.mark.parametrize("H", [64, 8192])
def test_sp_block_edge_rows(H):
    """The whole sequence-parallel pre-LN SwiGLU block with the LayerNorm edge rows as X."""
    shape = MLPShape(256, H, 512, 4, "swiglu", False, sp_ln=True)
    d = make_inputs(shape, 74)
    d["X"] = make_ln_edge_rows(shape.tokens, H, 74)
    gpu = run_gpu(shape, d)
    rel = check_full(shape, gpu, oracle_refs(shape, d))
    print(H, fmt_rel(rel))
