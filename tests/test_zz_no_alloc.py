"""The allocation-free bias-gradient entry point against the existing one.

mlpb_bias_grad_noalloc serves callers that cannot allocate device memory where they need
a bias gradient (code under a memory manager that owns all of the GPU's memory, or inside
that manager's callbacks).  Its column sums must match the db2 and db1 that
mlpb_backward computes with workspace scratch, on two calls in a row (the fixed scratch
array keeps the previous call's contents).  This file sorts last so that a run stopping
at its first failure has run every other test already.
"""
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_inputs

from _harness import TOL, compare, to_f64

pytestmark = pytest.mark.gpu


def test_noalloc_matches_backward_bias_grads_twice():
    shape = MLPShape(1024, 1024, 4096, 4, "gelu", True)
    d = make_inputs(shape, 61)
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in d.items() if v is not None}
    blk = mlpb.MLPBlock(shape.tokens, shape.hidden, shape.ffn, shape.tp, "gelu", True)
    blk.forward(g["X"], g["W1"], g["b1"], g["W2"], g["b2"])
    grads = blk.backward(g["X"], g["W1"], g["W2"], g["dY"])
    # mlpb_backward leaves dZ [T][F] bf16 at the start of its workspace
    dZ = blk.workspace[: shape.tokens * shape.ffn * 2].view(torch.bfloat16).view(
        shape.tokens, shape.ffn)
    for _ in range(2):
        db2 = torch.full((shape.hidden,), float("nan"), device=dev)
        db1 = torch.full((shape.ffn,), float("nan"), device=dev)
        mlpb.mlpb_bias_grad_noalloc(g["dY"], db2)
        mlpb.mlpb_bias_grad_noalloc(dZ, db1)
        torch.cuda.synchronize()
        compare("db2", to_f64(db2), to_f64(grads["db2"]), tol=TOL)
        compare("db1", to_f64(db1), to_f64(grads["db1"]), tol=TOL)
    assert mlpb.mlpb_last_device_error(blk.handle) == 0
    blk.close()


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
