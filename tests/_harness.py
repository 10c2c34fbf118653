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


def rms_rel(got, ref):
    """RMS(got - ref) / RMS(ref) over the compared entries."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.sqrt(np.mean((got - ref) ** 2)))
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


# RMS of the difference to the bf16-storage oracle, as a fraction of its RMS.  The two
# differ where the GPU's fp32 value and the oracle's fp64 value of a stored activation
# round to neighbouring bf16 numbers (one step, 2^-7 of the value at most): in a fraction
# p of the entries, p ~ the pre-rounding error over the bf16 spacing.  A fraction p of
# one-step changes moves an output sum by about sqrt(p) 2^-7 of its RMS; the fp32 GEMM
# error measured on this hardware (1-2 sqrt(K) 2^-24 of the RMS at the median) keeps p
# below 2 %, so <= 1.1e-3.
RMS_TOL = 2e-3


def gate(name, got, exact, stored, tol=TOL):
    """The parity gate of one output tensor, three bounds:

    * against the exact fp64 oracle: max|gpu - exact| <= tol * RMS wherever storing the
      activations in bf16 (the workloads' "bf16 in") leaves that reachable; where bf16
      storage by itself already puts the result further than tol from the exact value
      (the SwiGLU blocks' dW1, measured by the bf16-storage oracle), the GPU may be no
      further from it than 1.15x the bf16-storage oracle plus 0.2 % RMS.
    * against the bf16-storage oracle (the same block with every GEMM-input activation
      rounded to bf16, as the kernels store them), in RMS: RMS(gpu - stored) <= RMS_TOL *
      RMS -- ten times tighter than tol, and blind to nothing that touches many entries.
    * against the bf16-storage oracle, in max: max|gpu - stored| <= tol * RMS, unless bf16
      storage alone moves this tensor by more than tol / 2 (e_store): then a rounding that
      the GPU takes the other way (one bf16 step where the storage error is at most half
      of one) can move an entry by up to twice that, and the bound is 2 e_store + 0.2 %.
    Returns (gpu-vs-exact, bf16-oracle-vs-exact, gpu-vs-bf16-oracle max, ... RMS).
    """
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == np.shape(exact), f"{name}: shape {got.shape} vs {np.shape(exact)}"
    assert np.isfinite(got).all(), f"{name}: non-finite GPU output"
    e_gpu = max_rel(got, exact)
    e_store = max_rel(stored, exact)
    e_vs_store = max_rel(got, stored)
    r_vs_store = rms_rel(got, stored)
    assert e_gpu <= max(tol, 1.15 * e_store + 2e-3), (
        f"{name}: vs exact oracle {e_gpu:.4e} > max({tol}, bf16-storage bound {e_store:.4e})")
    assert r_vs_store <= RMS_TOL, (
        f"{name}: RMS vs bf16-storage oracle {r_vs_store:.3e} > {RMS_TOL}")
    bound = tol if e_store <= tol / 2 else max(tol, 2.0 * e_store + 2e-3)
    assert e_vs_store <= bound, (
        f"{name}: max vs bf16-storage oracle {e_vs_store:.4e} > {bound:.4e} "
        f"(bf16 storage alone {e_store:.4e})")
    return e_gpu, e_store, e_vs_store, r_vs_store


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
    return float((diff > 0).mean()) if diff.size else 0.0


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
        dX = torch.empty((T, H), dtype=mlpb.out_dtype(blk.cfg), device=dev)
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


def oracle_refs(shape: MLPShape, d: dict):
    """The exact and the bf16-storage oracle results (the pair check_full compares with)."""
    return oracle_pair(shape, d)


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
    # the fraction of each saved activation whose bf16 rounding went the other way
    if shape.act == "swiglu":
        zs = pack_glu(stored["G"], stored["U"], shape.tp)
    else:
        zs = stored["Z"]
    flips = {"Z": compare_stored("Zsaved", to_f64(gpu["Z"]), zs),
             "A": compare_stored("Asaved", to_f64(gpu["A"]), stored["A"])}
    if shape.sp_ln:
        flips["Xn"] = compare_stored("Xn", to_f64(gpu["Xn"]), stored["Xn"])
    rel["flips"] = tuple(round(v, 6) for v in flips.values())
    return rel


def fmt_rel(rel):
    """The gate values of check_full / gate, three significant digits, for printing."""
    return {k: tuple(float(f"{x:.3g}") for x in v) for k, v in rel.items()}


def inputs_for(shape: MLPShape, wid: int):
    return make_inputs(shape, wid)
