"""The emulated sequence-parallel exchange as device copies (MLPB_FLAG_EMULATE_COPIES).

The gathers (X in front of fc1, and again with dY in the backward) and the scatters (of
Y after fc2 and of dX after the dX GEMM) move bytes but change no value: every output,
saved activation and parameter gradient must equal the view mode's bit for bit -- plain,
with bf16 outputs, with E4M3 GEMMs, and through the residual branch.  With timing on,
each copy has its own record whose bytes are the copy's read plus write.
"""
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_inputs

from _harness import run_gpu

pytestmark = pytest.mark.gpu

EMU = mlpb.MLPB_FLAG_EMULATE_COPIES

CASES = [
    pytest.param(MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True), 101, 0,
                 id="swiglu-t4"),
    pytest.param(MLPShape(384, 320, 1408, 4, "gelu", True, sp_ln=True), 102, 0,
                 id="gelu-t4-bias-raggedH"),
    pytest.param(MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True), 103,
                 mlpb.MLPB_FLAG_BF16_OUT, id="swiglu-t4-bf16-out"),
    pytest.param(MLPShape(256, 512, 2048, 4, "gelu", True, sp_ln=True), 104,
                 mlpb.MLPB_FLAG_FP8, id="gelu-t4-fp8"),
]

KEYS = ("Y", "Xn", "mean", "rstd", "Z", "A", "dXn", "dX", "dW1", "dW2", "dgamma", "dbeta")


@pytest.mark.parametrize("shape,wid,flags", CASES)
def test_emulated_copies_change_no_bit(shape, wid, flags):
    d = make_inputs(shape, wid)
    view = run_gpu(shape, d, flags=flags)
    copy = run_gpu(shape, d, flags=flags | EMU, timing=True)
    assert view["status"] == 0 and copy["status"] == 0
    for k in KEYS + (("db1", "db2") if shape.bias else ()):
        assert torch.equal(view[k], copy[k]), k
    recs = {r["name"]: r for r in copy["timings"]}
    T, H = shape.tokens, shape.hidden
    ob = 2 if flags & mlpb.MLPB_FLAG_BF16_OUT else 4
    assert recs["sp_gather_x"]["bytes"] == 2 * 2 * T * H
    assert recs["sp_gather_dy"]["bytes"] == 2 * 2 * T * H
    assert recs["sp_scatter_y"]["bytes"] == 2 * ob * T * H
    assert recs["sp_scatter_dx"]["bytes"] == 2 * ob * T * H
    assert all(recs[n]["flops"] == 0.0 for n in recs if n.startswith("sp_"))


def test_emulated_copies_branch():
    shape = MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True)
    d = make_inputs(shape, 105)
    dev = torch.device("cuda:0")
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    outs = []
    for flags in (0, EMU):
        br = mlpb.MLPBranch(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act,
                            shape.bias, shape.ln_eps, flags)
        Y = br.forward(g["X"], g["gamma"], g["beta"], g["W1"], g["b1"], g["W2"], g["b2"])
        gr = br.backward(g["X"], g["gamma"], g["W1"], g["W2"], g["dY"])
        torch.cuda.synchronize()
        assert mlpb.mlpb_last_device_error(br.handle) == 0
        outs.append(dict(Y=Y, **gr))
        br.close()
    for k in ("Y", "dX", "dW1", "dW2", "dgamma", "dbeta"):
        assert torch.equal(outs[0][k], outs[1][k]), k


def test_emulated_copies_need_the_sequence_parallel_layout_and_a_workspace():
    with pytest.raises(mlpb.MLPBError) as e:
        mlpb.MLPBlock(128, 256, 1024, 2, "gelu", True, False, 1e-5, EMU)
    assert e.value.status == mlpb.MLPB_EUNSUPPORTED
    blk = mlpb.MLPBlock(128, 256, 1024, 2, "gelu", True, True, 1e-5, EMU)
    dev = torch.device("cuda:0")
    X = torch.zeros((128, 256), dtype=torch.bfloat16, device=dev)
    W1 = torch.zeros((2, 512, 256), dtype=torch.bfloat16, device=dev)
    W2 = torch.zeros((2, 256, 512), dtype=torch.bfloat16, device=dev)
    b1 = torch.zeros(1024, dtype=torch.bfloat16, device=dev)
    b2 = torch.zeros(256, dtype=torch.bfloat16, device=dev)
    Y = torch.empty((128, 256), device=dev)
    with pytest.raises(mlpb.MLPBError) as e:
        mlpb.mlpb_forward(blk.handle, X, W1, b1, W2, b2, Y, blk.Z, blk.A, None)
    assert e.value.status == mlpb.MLPB_EINVAL
    blk.close()
