"""Shared helpers of the GPU parity tests: run the block through the C ABI, run the
oracle on the same seeded bf16 inputs, and compare with the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_inputs
from oracle import layernorm as oln
from oracle import mlp as omlp

# max|gpu - oracle| <= TOL * RMS(oracle), per output tensor, over the compared entries.
TOL = 2e-2


def to_f64(t):
    return None if t is None else t.detach().to(torch.float64).cpu().numpy()


def compare(name, got, ref, tol=TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(got).all(), f"{name}: non-finite GPU output"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    assert err <= tol * rms + 1e-30, f"{name}: max|gpu-oracle| {err:.4e} > {tol} * RMS {rms:.4e}"
    return err / rms if rms else 0.0


def pack_glu(G, U, t):
    """Unsharded G, U [T][F] -> the library's saved layout [T][t][2][Fs]."""
    T, F = G.shape
    Fs = F // t
    return np.stack([G.reshape(T, t, Fs), U.reshape(T, t, Fs)], axis=2).reshape(T, 2 * F)


def run_gpu(shape: MLPShape, d: dict, flags: int = 0, timing: bool = False):
    """Forward + backward (+ SP-LN around it when shape.sp_ln) through the C ABI."""
    dev = torch.device("cuda:0")
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    blk = mlpb.MLPBlock(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act, shape.bias,
                        shape.sp_ln, shape.ln_eps, flags)
    if timing:
        mlpb.mlpb_enable_timing(blk.handle)
    out = {}
    X = g["X"]
    if shape.sp_ln:
        T, H = shape.tokens, shape.hidden
        Xn = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        mean = torch.empty((T,), dtype=torch.float32, device=dev)
        rstd = torch.empty((T,), dtype=torch.float32, device=dev)
        mlpb.mlpb_layernorm_sp_fwd(blk.handle, X, g["gamma"], g["beta"], Xn, mean, rstd)
        out.update(Xn=Xn, mean=mean, rstd=rstd)
        X = Xn
    out["Y"] = blk.forward(X, g["W1"], g["b1"], g["W2"], g["b2"])
    grads = blk.backward(X, g["W1"], g["W2"], g["dY"])
    if shape.sp_ln:
        T, H = shape.tokens, shape.hidden
        dX = torch.empty((T, H), dtype=torch.float32, device=dev)
        dgamma = torch.empty((H,), dtype=torch.float32, device=dev)
        dbeta = torch.empty((H,), dtype=torch.float32, device=dev)
        mlpb.mlpb_layernorm_sp_bwd(blk.handle, g["X"], g["gamma"], out["mean"], out["rstd"],
                                   grads["dX"], dX, dgamma, dbeta, blk.workspace)
        out.update(dXn=grads["dX"], dX=dX, dgamma=dgamma, dbeta=dbeta)
        grads = {k: v for k, v in grads.items() if k != "dX"}
    out.update(grads)
    out["Z"], out["A"] = blk.Z, blk.A
    torch.cuda.synchronize()
    out["status"] = mlpb.mlpb_last_device_error(blk.handle)
    if timing:
        out["timings"] = mlpb.mlpb_read_timings(blk.handle)
    blk.close()
    return out


def oracle_full(shape: MLPShape, d: dict):
    f = {k: to_f64(v) for k, v in d.items()}
    if shape.sp_ln:
        fw = oln.block_forward(f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"],
                               f["W2"], f["b2"], shape.act, shape.tp)
        bw = oln.block_backward(f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"],
                                f["W2"], f["dY"], shape.act, shape.tp)
        return {**fw, **bw}
    fw = omlp.mlp_forward(f["X"], f["W1"], f["b1"], f["W2"], f["b2"], shape.act)
    bw = omlp.mlp_backward(f["X"], f["W1"], f["b1"], f["W2"], f["dY"], shape.act)
    return {**fw, **bw}


def check_full(shape: MLPShape, gpu: dict, ref: dict):
    """Every element of every output (and the saved activations) against the oracle."""
    assert gpu["status"] == 0, f"device error status {gpu['status']}"
    rel = {}
    names = ["Y", "dX", "dW1", "dW2"] + (["db1", "db2"] if shape.bias else [])
    if shape.sp_ln:
        names += ["dgamma", "dbeta", "dXn"]
    for k in names:
        rel[k] = compare(k, to_f64(gpu[k]), ref[k])
    # saved activations are bf16 tensor-core inputs: compared for diagnosis
    if shape.act == "swiglu":
        rel["Zsaved"] = compare("Zsaved", to_f64(gpu["Z"]), pack_glu(ref["G"], ref["U"], shape.tp))
    else:
        rel["Zsaved"] = compare("Zsaved", to_f64(gpu["Z"]), ref["Z"])
    rel["Asaved"] = compare("Asaved", to_f64(gpu["A"]), ref["A"])
    return rel


def inputs_for(shape: MLPShape, wid: int):
    return make_inputs(shape, wid)
