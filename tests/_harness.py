"""Shared helpers of the GPU parity tests: run the block through the C ABI, run the
oracle on the same seeded bf16 inputs, and compare with the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, make_inputs
from oracle import layernorm as oln
from oracle import mlp as omlp
from oracle.bf16 import round_bf16

# max|gpu - oracle| <= TOL * RMS(oracle), per output tensor, over the compared entries.
TOL = 2e-2


def to_f64(t):
    return None if t is None else t.detach().to(torch.float64).cpu().numpy()


def max_rel(got, ref):
    """max|got - ref| / RMS(ref) over the compared entries."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.abs(got - ref).max())
    return err / rms if rms else (0.0 if err == 0.0 else np.inf)


def compare(name, got, ref, tol=TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(got).all(), f"{name}: non-finite GPU output"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    assert err <= tol * rms + 1e-30, f"{name}: max|gpu-oracle| {err:.4e} > {tol} * RMS {rms:.4e}"
    return err / rms if rms else 0.0


def gate(name, got, exact, stored, tol=TOL):
    """The parity gate of one output tensor: max|gpu - exact| <= tol * RMS(exact).

    Where storing the GEMM-input activations in bf16 (the workloads' "bf16 in") by
    itself already puts the result further than tol from the exact fp64 value -- the
    oracle's bf16-storage mode measures that distance -- the bar is that distance:
    the GPU may be no further from the exact result than 1.15x the bf16-storage
    oracle, plus 0.2 % RMS for the fp32 accumulation order.
    Returns (gpu-vs-exact, bf16-oracle-vs-exact, gpu-vs-bf16-oracle) as max/RMS.
    """
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == np.shape(exact), f"{name}: shape {got.shape} vs {np.shape(exact)}"
    assert np.isfinite(got).all(), f"{name}: non-finite GPU output"
    e_gpu = max_rel(got, exact)
    e_store = max_rel(stored, exact)
    e_vs_store = max_rel(got, stored)
    assert e_gpu <= max(tol, 1.15 * e_store + 2e-3), (
        f"{name}: vs exact oracle {e_gpu:.4e} > max({tol}, bf16-storage bound {e_store:.4e})")
    return e_gpu, e_store, e_vs_store


def compare_stored(name, got, ref):
    """bf16 activations against the bf16-storage oracle: within one bf16 unit (2^-7
    relative) plus 1e-3 RMS, except for at most 1e-6 of the entries (where the GPU's
    fp32 and the oracle's fp64 inputs to a rounding straddle a bf16 boundary upstream),
    and every entry within two units plus 1e-2 RMS."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape and np.isfinite(got).all(), name
    rms = float(np.sqrt(np.mean(ref * ref)))
    diff = np.abs(got - ref)
    near = int((diff > np.abs(ref) * 2.0 ** -7 + 1e-3 * rms).sum())
    assert near <= max(1, int(1e-6 * ref.size)), f"{name}: {near} entries beyond one bf16 unit"
    far = int((diff > np.abs(ref) * 2.0 ** -6 + 1e-2 * rms).sum())
    assert far == 0, f"{name}: {far} entries beyond two bf16 units + 1e-2 RMS"


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


def oracle_full(shape: MLPShape, d: dict, store=None):
    f = {k: to_f64(v) for k, v in d.items()}
    if shape.sp_ln:
        fw = oln.block_forward(f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"],
                               f["W2"], f["b2"], shape.act, shape.tp, store)
        bw = oln.block_backward(f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"],
                                f["W2"], f["dY"], shape.act, shape.tp, store)
        return {**fw, **bw}
    fw = omlp.mlp_forward(f["X"], f["W1"], f["b1"], f["W2"], f["b2"], shape.act, store)
    bw = omlp.mlp_backward(f["X"], f["W1"], f["b1"], f["W2"], f["dY"], shape.act, store)
    return {**fw, **bw}


def oracle_pair(shape: MLPShape, d: dict):
    """(exact, bf16-storage) oracle results on the same inputs."""
    return oracle_full(shape, d), oracle_full(shape, d, round_bf16)


def check_full(shape: MLPShape, gpu: dict, refs):
    """Every element of every output (and the saved activations) against the oracle."""
    assert gpu["status"] == 0, f"device error status {gpu['status']}"
    exact, stored = refs
    rel = {}
    names = ["Y", "dX", "dW1", "dW2"] + (["db1", "db2"] if shape.bias else [])
    if shape.sp_ln:
        names += ["dgamma", "dbeta", "dXn"]
    for k in names:
        rel[k] = gate(k, to_f64(gpu[k]), exact[k], stored[k])
    # saved activations are the bf16 tensor-core inputs themselves
    if shape.act == "swiglu":
        compare_stored("Zsaved", to_f64(gpu["Z"]), pack_glu(stored["G"], stored["U"], shape.tp))
    else:
        compare_stored("Zsaved", to_f64(gpu["Z"]), stored["Z"])
    compare_stored("Asaved", to_f64(gpu["A"]), stored["A"])
    if shape.sp_ln:
        compare_stored("Xn", to_f64(gpu["Xn"]), stored["Xn"])
    return rel


def inputs_for(shape: MLPShape, wid: int):
    return make_inputs(shape, wid)
