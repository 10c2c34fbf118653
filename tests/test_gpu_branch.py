"""GPU parity of the pre-norm MLP branch Y = X + MLP(LN(X)) (mlpb_branch_forward /
mlpb_branch_backward): the residual added in fc2's epilogue, the residual gradient added
in the LayerNorm backward, and dX formed in place.

  * small shapes: every element of Y, dX and every parameter gradient against the fp64
    oracle's branch, within the parity gate;
  * bit for bit, the branch equals the separate calls it fuses plus the residual added
    on the host in fp32: Y = Y_block + X and dX = dX_block + dY (one fp32 add each);
  * the SP pre-LN SwiGLU workload at full size (T8192 H8192 F28672 t8): the same
    bitwise identity, and 128 seeded rows of Y and dX against the oracle;
  * T = 0, and argument errors that launch nothing.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, WORKLOADS, make_inputs, sample_rows
from oracle import layernorm as oln
from oracle.bf16 import round_bf16

from _harness import gate, run_gpu, to_f64

pytestmark = pytest.mark.gpu

SMALL = [
    pytest.param(MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True), 71,
                 id="swiglu-t4"),
    pytest.param(MLPShape(384, 320, 1408, 4, "gelu", True, sp_ln=True), 72,
                 id="gelu-t4-bias-raggedH-Fs352"),
    pytest.param(MLPShape(128, 128, 512, 2, "gelu", True, sp_ln=True), 73, id="gelu-t2-tiny"),
    # the LayerNorm backward's residual variant at 2 and 8 vectors a thread
    pytest.param(MLPShape(256, 3072, 512, 2, "gelu", True, sp_ln=True), 76, id="gelu-H3072"),
    pytest.param(MLPShape(128, 16384, 256, 2, "swiglu", False, sp_ln=True), 77,
                 id="swiglu-H16384"),
]


def run_branch(shape, d):
    dev = torch.device("cuda:0")
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    br = mlpb.MLPBranch(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act, shape.bias,
                        shape.ln_eps)
    Y = br.forward(g["X"], g["gamma"], g["beta"], g["W1"], g["b1"], g["W2"], g["b2"])
    grads = br.backward(g["X"], g["gamma"], g["W1"], g["W2"], g["dY"])
    torch.cuda.synchronize()
    out = {"Y": Y, **grads, "status": mlpb.mlpb_last_device_error(br.handle)}
    br.close()
    return out


def oracle_branch(shape, d, store=None):
    f = {k: to_f64(v) for k, v in d.items()}
    a = (f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"], f["W2"])
    fw = oln.branch_forward(*a, f["b2"], shape.act, shape.tp, store)
    bw = oln.branch_backward(*a, f["dY"], shape.act, shape.tp, store)
    return {**fw, **bw}


def _names(shape):
    return ["Y", "dX", "dW1", "dW2", "dgamma", "dbeta"] + (["db1", "db2"] if shape.bias else [])


def _check_against_block(shape, d, br):
    """The branch equals the unfused calls plus the residual, bit for bit."""
    blk = run_gpu(shape, d)
    assert blk["status"] == 0
    X = d["X"].to("cuda:0").float()
    dY = d["dY"].to("cuda:0").float()
    assert torch.equal(br["Y"], blk["Y"] + X), "Y != Y_block + X"
    assert torch.equal(br["dX"], blk["dX"] + dY), "dX != dX_block + dY"
    for k in _names(shape)[2:]:
        assert torch.equal(br[k], blk[k]), k


@pytest.mark.parametrize("shape,wid", SMALL)
def test_branch_every_element(shape, wid):
    d = make_inputs(shape, wid)
    br = run_branch(shape, d)
    assert br["status"] == 0
    exact, stored = oracle_branch(shape, d), oracle_branch(shape, d, round_bf16)
    for k in _names(shape):
        gate(k, to_f64(br[k]), exact[k], stored[k])
    _check_against_block(shape, d, br)


def test_branch_full_size_sp_swiglu():
    shape = WORKLOADS[5]
    wid = 5
    d = make_inputs(shape, wid)
    br = run_branch(shape, d)
    assert br["status"] == 0
    _check_against_block(shape, d, br)
    rows = sample_rows(shape, wid).numpy()
    idx = torch.from_numpy(rows).cuda()
    got = {"Y": to_f64(br["Y"][idx]), "dX": to_f64(br["dX"][idx])}
    del br
    torch.cuda.empty_cache()
    f = {k: to_f64(v) for k, v in d.items()}
    a = (f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"], f["W2"], f["b2"],
         f["dY"], rows, shape.act)
    ex, st = oln.branch_rows(*a), oln.branch_rows(*a, round_bf16)
    for k in ("Y", "dX"):
        gate(k, got[k], ex[k], st[k])


def test_branch_empty_batch_and_argument_errors():
    dev = torch.device("cuda:0")
    d = make_inputs(MLPShape(128, 256, 1024, 2, "gelu", True, sp_ln=True), 74)
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    br = mlpb.MLPBranch(0, 256, 1024, 2, "gelu", True)
    X = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    Y = br.forward(X, g["gamma"], g["beta"], g["W1"], g["b1"], g["W2"], g["b2"])
    grads = br.alloc_grads(g["W1"], g["W2"])
    for k in ("dW1", "dW2", "db1", "db2", "dgamma", "dbeta"):
        grads[k].fill_(7.0)
    br.backward(X, g["gamma"], g["W1"], g["W2"], torch.empty_like(X), grads)
    torch.cuda.synchronize()
    assert Y.shape == (0, 256) and mlpb.mlpb_last_device_error(br.handle) == 0
    for k in ("dW1", "dW2", "db1", "db2", "dgamma", "dbeta"):
        assert torch.count_nonzero(grads[k]).item() == 0, k
    br.close()

    # a handle without the LayerNorm cannot run the branch; a missing bias is an error
    blk = mlpb.MLPBlock(128, 256, 1024, 2, "gelu", True)
    Xs = g["X"]
    scratch = [torch.empty((128, 256), dtype=torch.bfloat16, device=dev),
               torch.empty(128, device=dev), torch.empty(128, device=dev)]
    with pytest.raises(mlpb.MLPBError) as e:
        mlpb.mlpb_branch_forward(blk.handle, Xs, g["gamma"], g["beta"], g["W1"], g["b1"],
                                 g["W2"], g["b2"], torch.empty((128, 256), device=dev),
                                 *scratch, blk.Z, blk.A)
    assert e.value.status == mlpb.MLPB_EUNSUPPORTED
    blk.close()
    br = mlpb.MLPBranch(128, 256, 1024, 2, "gelu", True)
    Yb = torch.full((128, 256), 5.0, device=dev)
    with pytest.raises(mlpb.MLPBError) as e:
        br.forward(Xs, g["gamma"], g["beta"], g["W1"], None, g["W2"], g["b2"], Yb)
    assert e.value.status == mlpb.MLPB_EINVAL
    torch.cuda.synchronize()
    assert bool((Yb == 5.0).all())  # nothing ran
    assert mlpb.mlpb_last_device_error(br.handle) == 0
    br.close()


def test_branch_with_recompute_and_accumulation_is_block_plus_residual_and_start():
    """The residual branch with selective recomputation and gradient accumulation at once:
    bit for bit the unfused block run with recomputation, plus the residual (Y + X,
    dX + dY), with the parameter gradients added to seeded starting values."""
    from inputs import make_main_grads
    shape = MLPShape(384, 320, 1408, 4, "gelu", True, sp_ln=True)
    d = make_inputs(shape, 75)
    blk = run_gpu(shape, d, flags=mlpb.MLPB_FLAG_RECOMPUTE_ACT)
    assert blk["status"] == 0
    dev = torch.device("cuda:0")
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    br = mlpb.MLPBranch(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act, shape.bias,
                        shape.ln_eps,
                        flags=mlpb.MLPB_FLAG_RECOMPUTE_ACT | mlpb.MLPB_FLAG_ACCUMULATE_GRADS)
    grads = br.alloc_grads(g["W1"], g["W2"])
    names = ("dW1", "dW2", "db1", "db2", "dgamma", "dbeta")
    main0 = make_main_grads({k: tuple(grads[k].shape) for k in names}, 75)
    for k in names:
        grads[k].copy_(main0[k])
    Y = br.forward(g["X"], g["gamma"], g["beta"], g["W1"], g["b1"], g["W2"], g["b2"])
    br.A.fill_(float("nan"))  # recomputation must not read the forward's A
    br.backward(g["X"], g["gamma"], g["W1"], g["W2"], g["dY"], grads)
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(br.handle) == 0
    br.close()
    assert torch.equal(Y, blk["Y"] + g["X"].float())
    assert torch.equal(grads["dX"], blk["dX"] + g["dY"].float())
    for k in names:
        assert torch.equal(grads[k], main0[k].to(dev) + blk[k]), k
