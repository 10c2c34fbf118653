"""The allocation-free bias-gradient entry point against fp64 column sums and against the
existing entry point.

mlpb_bias_grad_noalloc serves callers that cannot allocate device memory where they need
a bias gradient (code under a memory manager that owns all of the GPU's memory, or inside
that manager's callbacks).  Its column sums must match the exact (fp64) column sums of the
same bf16 input, and the db2 that mlpb_backward computes with workspace scratch, on two
calls in a row (the fixed scratch array keeps the previous call's contents).  This file
sorts last so that a run stopping at its first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_bf16, make_inputs

from _harness import TOL, compare, to_f64

pytestmark = pytest.mark.gpu


def _colsum64(x):
    """The column sums of a bf16 tensor in fp64 (the definition of the bias gradient)."""
    return to_f64(x).sum(axis=0)


def test_noalloc_matches_exact_sums_and_backward_twice():
    shape = MLPShape(1024, 1024, 4096, 4, "gelu", True)
    d = make_inputs(shape, 61)
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in d.items() if v is not None}
    blk = mlpb.MLPBlock(shape.tokens, shape.hidden, shape.ffn, shape.tp, "gelu", True)
    blk.forward(g["X"], g["W1"], g["b1"], g["W2"], g["b2"])
    grads = blk.backward(g["X"], g["W1"], g["W2"], g["dY"])
    # a [T][F] bf16 matrix this test owns, standing in for dZ
    dZ = make_bf16((shape.tokens, shape.ffn), 61, std=0.05).to(dev)
    ref_db2, ref_db1 = _colsum64(d["dY"]), _colsum64(dZ)
    for _ in range(2):
        db2 = torch.full((shape.hidden,), float("nan"), device=dev)
        db1 = torch.full((shape.ffn,), float("nan"), device=dev)
        mlpb.mlpb_bias_grad_noalloc(g["dY"], db2)
        mlpb.mlpb_bias_grad_noalloc(dZ, db1)
        torch.cuda.synchronize()
        compare("db2 vs fp64", to_f64(db2), ref_db2, tol=TOL)
        compare("db1 vs fp64", to_f64(db1), ref_db1, tol=TOL)
        # the existing entry point on the same dY
        compare("db2 vs mlpb_backward", to_f64(db2), to_f64(grads["db2"]), tol=TOL)
    assert mlpb.mlpb_last_device_error(blk.handle) == 0
    blk.close()


def test_noalloc_ragged_splits_and_leftover_partials():
    """A row count whose last split is short and a width that ends inside a 512-column
    chunk, called after a wider input (whose partials stay in the array) and then again:
    each call's result depends on its own input only."""
    dev = torch.device("cuda:0")
    wide = make_bf16((160, 262144), 62).to(dev)
    ragged = make_bf16((1001, 4104), 63, log2_spread=4).to(dev)
    out_w = torch.empty(262144, device=dev)
    out_r = [torch.full((4104,), float("nan"), device=dev) for _ in range(2)]
    mlpb.mlpb_bias_grad_noalloc(wide, out_w)
    mlpb.mlpb_bias_grad_noalloc(ragged, out_r[0])
    mlpb.mlpb_bias_grad_noalloc(wide, out_w)
    mlpb.mlpb_bias_grad_noalloc(ragged, out_r[1])
    torch.cuda.synchronize()
    compare("wide", to_f64(out_w), _colsum64(wide), tol=TOL)
    ref = _colsum64(ragged)
    for o in out_r:
        compare("ragged", to_f64(o), ref, tol=TOL)
    assert torch.equal(out_r[0], out_r[1])


def test_noalloc_rejects_oversize_and_handles_empty():
    dev = torch.device("cuda:0")
    wide = torch.zeros((1, (1 << 20) + 8), dtype=torch.bfloat16, device=dev)
    out = torch.zeros(((1 << 20) + 8,), dtype=torch.float32, device=dev)
    with pytest.raises(mlpb.MLPBError) as e:
        mlpb.mlpb_bias_grad_noalloc(wide, out)
    assert e.value.status == mlpb.MLPB_EUNSUPPORTED
    empty = torch.zeros((0, 64), dtype=torch.bfloat16, device=dev)
    out = torch.full((64,), 3.0, device=dev)
    mlpb.mlpb_bias_grad_noalloc(empty, out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    assert np.isfinite(to_f64(out)).all()
