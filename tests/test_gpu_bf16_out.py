"""The bf16-output mode (MLPB_FLAG_BF16_OUT): Y, dX and the LayerNorm backward's dXn / dX
stored as bf16.

The mode changes no sum, only where it is rounded: every bf16 output must equal, bit for
bit, the fp32 mode's output rounded once to bf16 (nearest, ties to even) -- through the
plain epilogues, the tail split's fixup, the FP8 GEMMs' epilogue, and the residual
branch.  The LayerNorm backward then reads the bf16 dXn: its bf16 dX (and dgamma, dbeta)
must equal the fp32 LayerNorm backward applied to that same bf16 dXn, rounded once.  The
parameter gradients do not change at all.  Distances to the fp64 oracle are printed (the
mode's parity is reported, not gated: the final rounding alone can move a value by
2^-9 of itself).
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_inputs

from _harness import max_rel, oracle_pair, run_gpu, to_f64

pytestmark = pytest.mark.gpu

BF16 = mlpb.MLPB_FLAG_BF16_OUT

SHAPES = [
    # 80 pair tiles on 76 pairs: fc2's and dX's tail tiles go through the split fixup
    pytest.param(MLPShape(1024, 5120, 2048, 2, "gelu", True), 91, 0, id="gelu-tail-split"),
    pytest.param(MLPShape(256, 192, 704, 8, "swiglu", False), 92, 0, id="swiglu-t8-raggedH"),
    pytest.param(MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True), 93, 0,
                 id="sp-ln-swiglu-t4"),
    pytest.param(MLPShape(256, 512, 2048, 4, "gelu", True), 94, mlpb.MLPB_FLAG_FP8,
                 id="gelu-fp8"),
]


def _bits_equal(name, got, want):
    assert got.dtype == torch.bfloat16, name
    diff = int((got.view(torch.int16) != want.view(torch.int16)).sum().item())
    assert diff == 0, f"{name}: {diff} entries differ from the fp32 result rounded once"


def _ln_bwd_fp32(shape, d, gpu, dXn):
    """The fp32-mode LayerNorm backward of `dXn` (fp32 values) with the saved statistics."""
    T, H, t = shape.tokens, shape.hidden, shape.tp
    dev = torch.device("cuda:0")
    h = mlpb.mlpb_create(mlpb.make_config(T, H, shape.ffn, t, shape.act, shape.bias, True,
                                          shape.ln_eps))
    ws = torch.empty(mlpb.mlpb_workspace_size(h), dtype=torch.uint8, device=dev)
    dX = torch.empty((T, H), device=dev)
    dg = torch.empty(H, device=dev)
    db = torch.empty(H, device=dev)
    mlpb.mlpb_layernorm_sp_bwd(h, d["X"].to(dev), d["gamma"].to(dev), gpu["mean"], gpu["rstd"],
                               dXn.contiguous(), dX, dg, db, ws)
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(h) == 0
    mlpb.mlpb_destroy(h)
    return dX, dg, db


@pytest.mark.parametrize("shape,wid,flags", SHAPES)
def test_bf16_outputs_are_the_fp32_outputs_rounded_once(shape, wid, flags):
    d = make_inputs(shape, wid)
    f32 = run_gpu(shape, d, flags=flags)
    b16 = run_gpu(shape, d, flags=flags | BF16)
    assert f32["status"] == 0 and b16["status"] == 0
    _bits_equal("Y", b16["Y"], f32["Y"].to(torch.bfloat16))
    for k in ("dW1", "dW2") + (("db1", "db2") if shape.bias else ()):
        assert torch.equal(b16[k], f32[k]), k
    if shape.sp_ln:
        _bits_equal("dXn", b16["dXn"], f32["dXn"].to(torch.bfloat16))
        dX, dg, db = _ln_bwd_fp32(shape, d, b16, b16["dXn"].float())
        _bits_equal("dX", b16["dX"], dX.to(torch.bfloat16))
        assert torch.equal(b16["dgamma"], dg) and torch.equal(b16["dbeta"], db)
    else:
        _bits_equal("dX", b16["dX"], f32["dX"].to(torch.bfloat16))
    if flags == 0:  # the mode's distance to the oracle, reported
        exact, stored = oracle_pair(shape, d)
        rep = {k: (round(max_rel(to_f64(b16[k]), exact[k]), 5),
                   round(max_rel(to_f64(b16[k]), stored[k]), 5)) for k in ("Y", "dX")}
        print(shape, "bf16 outputs: max/RMS vs exact, vs bf16-storage", rep)


def test_bf16_output_branch():
    """The residual branch: Y = X + MLP(LN(X)) rounded once, and dX = dY + LN'(dXn) with the
    bf16 dXn formed in the dX buffer and rewritten in place."""
    shape = MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True)
    d = make_inputs(shape, 95)
    dev = torch.device("cuda:0")
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    outs = {}
    for flags in (0, BF16):
        br = mlpb.MLPBranch(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act,
                            shape.bias, shape.ln_eps, flags)
        Y = br.forward(g["X"], g["gamma"], g["beta"], g["W1"], g["b1"], g["W2"], g["b2"])
        gr = br.backward(g["X"], g["gamma"], g["W1"], g["W2"], g["dY"])
        torch.cuda.synchronize()
        assert mlpb.mlpb_last_device_error(br.handle) == 0
        outs[flags] = dict(Y=Y, Xn=br.Xn.clone(), mean=br.mean.clone(), rstd=br.rstd.clone(),
                           **gr)
        br.close()
    b16 = outs[BF16]
    _bits_equal("Y", b16["Y"], outs[0]["Y"].to(torch.bfloat16))
    # the bf16 dXn of the MLP backward on the branch's Xn, then the fp32 LayerNorm backward
    blk = mlpb.MLPBlock(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act, shape.bias,
                        True, shape.ln_eps, BF16)
    blk.forward(b16["Xn"], g["W1"], g["b1"], g["W2"], g["b2"])
    dXn = blk.backward(b16["Xn"], g["W1"], g["W2"], g["dY"])["dX"]
    torch.cuda.synchronize()
    blk.close()
    dX, dg, db = _ln_bwd_fp32(shape, d, b16, dXn.float())
    _bits_equal("dX", b16["dX"], (dX + g["dY"].float()).to(torch.bfloat16))
    assert torch.equal(b16["dgamma"], dg) and torch.equal(b16["dbeta"], db)
    assert np.isfinite(to_f64(b16["dX"])).all()
