"""GPU parity of gradient-accumulation fusion (MLPB_FLAG_ACCUMULATE_GRADS).

Two micro-batches run forward + backward through one accumulating handle into main-grad
buffers that start from seeded non-zero contents.  Checked:
  * bit for bit, each accumulated buffer equals (start + g1) + g2 in fp32, where g1, g2 are
    the same library's overwrite-mode gradients of the two micro-batches (every fused
    epilogue performs exactly one fp32 add per element and micro-batch);
  * against the fp64 oracle, (final - start) is the parameter gradient of the
    concatenated batch, within the parity gate;
  * dX (an activation gradient) is overwritten, not accumulated;
  * an empty micro-batch (T = 0) leaves the buffers untouched.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_inputs, make_main_grads
from oracle import mlp as omlp

from _harness import gate, oracle_pair, to_f64

pytestmark = pytest.mark.gpu

ACC = mlpb.MLPB_FLAG_ACCUMULATE_GRADS

SHAPES = [
    # ragged H (320 = 64 mod 128) and Fs = 352 (a shard seam inside a K block), bias
    pytest.param(MLPShape(512, 320, 1408, 4, "gelu", True), 51, id="gelu-t4-bias-ragged"),
    # SwiGLU behind the sequence-parallel LayerNorm: dgamma / dbeta accumulate too
    pytest.param(MLPShape(512, 384, 1024, 4, "swiglu", False, sp_ln=True), 52,
                 id="sp-ln-swiglu-t4"),
    # micro-batches of 1024 tokens: dW1's 160 pair tiles end in a tail-split wave whose
    # fixup adds into the buffers
    pytest.param(MLPShape(2048, 5120, 2048, 2, "gelu", True), 54, id="gelu-tail-split"),
]


def _param_names(shape):
    names = ["dW1", "dW2"] + (["db1", "db2"] if shape.bias else [])
    return names + (["dgamma", "dbeta"] if shape.sp_ln else [])


def _micro_step(blk, shape, g, X, dY, grads, ln):
    """forward + backward of one micro-batch; parameter gradients land in `grads` / `ln`.
    Returns the micro-batch's input gradient (a copy)."""
    dev = X.device
    T, H = X.shape
    if shape.sp_ln:
        Xn = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        mean = torch.empty((T,), dtype=torch.float32, device=dev)
        rstd = torch.empty((T,), dtype=torch.float32, device=dev)
        mlpb.mlpb_layernorm_sp_fwd(blk.handle, X, g["gamma"], g["beta"], Xn, mean, rstd)
        Xin = Xn
    else:
        Xin = X
    blk.forward(Xin, g["W1"], g["b1"], g["W2"], g["b2"])
    blk.backward(Xin, g["W1"], g["W2"], dY, grads)
    if shape.sp_ln:
        dX = torch.empty((T, H), dtype=torch.float32, device=dev)
        mlpb.mlpb_layernorm_sp_bwd(blk.handle, X, g["gamma"], mean, rstd, grads["dX"], dX,
                                   ln["dgamma"], ln["dbeta"], blk.workspace)
        return dX
    return grads["dX"].clone()


@pytest.mark.parametrize("shape,wid", SHAPES)
def test_two_micro_batches_accumulate(shape, wid):
    dev = torch.device("cuda:0")
    d = make_inputs(shape, wid)  # the whole batch; micro-batches are its two token halves
    exact, stored = oracle_pair(shape, d)
    names = _param_names(shape)
    scales = {k: float(np.sqrt(np.mean(exact[k] ** 2))) for k in names}
    main0 = make_main_grads({k: exact[k].shape for k in names}, wid, scales)

    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    Tm = shape.tokens // 2
    micro = shape.with_tokens(Tm)
    halves = [(g["X"][i * Tm:(i + 1) * Tm].contiguous(),
               g["dY"][i * Tm:(i + 1) * Tm].contiguous()) for i in range(2)]
    args = (Tm, shape.hidden, shape.ffn, shape.tp, shape.act, shape.bias, shape.sp_ln,
            shape.ln_eps)

    # overwrite mode: each micro-batch's own gradients
    ow = mlpb.MLPBlock(*args)
    per_mb, dx_ow = [], []
    for X, dY in halves:
        gr = ow.alloc_grads(g["W1"], g["W2"])
        ln = {k: torch.empty((shape.hidden,), dtype=torch.float32, device=dev)
              for k in ("dgamma", "dbeta")}
        dx_ow.append(_micro_step(ow, micro, g, X, dY, gr, ln))
        per_mb.append({**{k: v for k, v in gr.items() if v is not None}, **ln})
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(ow.handle) == 0
    ow.close()

    # accumulate mode into buffers holding main0
    acc = mlpb.MLPBlock(*args, flags=ACC)
    grads = acc.alloc_grads(g["W1"], g["W2"])
    for k in names:
        if k in grads:
            grads[k].copy_(main0[k])
    ln = {k: main0[k].to(dev) if shape.sp_ln else None for k in ("dgamma", "dbeta")}
    for i, (X, dY) in enumerate(halves):
        dx = _micro_step(acc, micro, g, X, dY, grads, ln)
        assert torch.equal(dx, dx_ow[i]), f"dX of micro-batch {i} is not overwritten"
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(acc.handle) == 0
    acc.close()
    final = {k: (ln[k] if k in ("dgamma", "dbeta") else grads[k]) for k in names}

    for k in names:
        start = main0[k].to(dev)
        want = (start + per_mb[0][k]) + per_mb[1][k]
        assert torch.equal(final[k], want), f"{k}: accumulated bits differ from (start+g1)+g2"
        # the oracle's concatenated-batch gradient, as accumulated from zeroed buffers
        ref = omlp.accumulate_param_grads({k: np.zeros(exact[k].shape)}, exact)[k]
        ref_st = omlp.accumulate_param_grads({k: np.zeros(stored[k].shape)}, stored)[k]
        gate(k, to_f64(final[k]) - to_f64(start), ref, ref_st)


def test_empty_micro_batch_leaves_main_grads():
    dev = torch.device("cuda:0")
    d = make_inputs(MLPShape(128, 256, 1024, 2, "gelu", True, sp_ln=True), 53)
    blk = mlpb.MLPBlock(0, 256, 1024, 2, "gelu", True, True, 1e-5, flags=ACC)
    W1, W2 = d["W1"].to(dev), d["W2"].to(dev)
    X = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    blk.forward(X, W1, d["b1"].to(dev), W2, d["b2"].to(dev))
    g = blk.alloc_grads(W1, W2)
    main0 = make_main_grads({k: tuple(g[k].shape) for k in ("dW1", "dW2", "db1", "db2")}, 53)
    for k, v in main0.items():
        g[k].copy_(v)
    blk.backward(X, W1, W2, torch.empty((0, 256), dtype=torch.bfloat16, device=dev), g)
    dgamma = torch.full((256,), 3.0, device=dev)
    dbeta = torch.full((256,), -2.0, device=dev)
    mlpb.mlpb_layernorm_sp_bwd(blk.handle, None, d["gamma"].to(dev), None, None, None, None,
                               dgamma, dbeta, None)
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(blk.handle) == 0
    for k, v in main0.items():
        assert torch.equal(g[k].cpu(), v), k
    assert bool((dgamma == 3.0).all()) and bool((dbeta == -2.0).all())
    blk.close()
