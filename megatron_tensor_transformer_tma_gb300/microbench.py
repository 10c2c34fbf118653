"""Bandwidth microbenchmark of the library's memory-bound entry points.

  python -m megatron_tensor_transformer_tma_gb300.microbench [--tokens T] [--hidden H]
         [--tp t] [--iters N]

Times, with CUDA events over N back-to-back calls on resident random inputs:
mlpb_layernorm_sp_fwd (reads X bf16, writes Xn bf16: 4 bytes per element),
mlpb_layernorm_sp_bwd (reads X bf16 and dXn fp32, writes dX fp32: 10 bytes per element),
mlpb_bias_grad_noalloc on a [T][H] bf16 matrix (2 bytes per element), and the LayerNorm
backward inside mlpb_branch_backward, which also reads the residual gradient (12 bytes
per element; its CUDA-event record, on a branch with a token-sized MLP), and prints one
JSON line with microseconds and GB/s per entry point.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import mlpb as m
from .build import build


def _time(fn, iters):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters * 1e3  # microseconds


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=8192)
    ap.add_argument("--hidden", type=int, default=8192)
    ap.add_argument("--tp", type=int, default=8)
    ap.add_argument("--iters", type=int, default=50)
    a = ap.parse_args(argv)
    build()
    T, H, t = a.tokens, a.hidden, a.tp
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    h = m.mlpb_create(m.make_config(T, H, 8 * t, t, "swiglu", False, True, 1e-5))
    X = torch.randn(T, H, device=dev, generator=g).to(torch.bfloat16)
    gm = (1 + 0.1 * torch.randn(H, device=dev, generator=g)).to(torch.bfloat16)
    bt = (0.02 * torch.randn(H, device=dev, generator=g)).to(torch.bfloat16)
    Xn = torch.empty_like(X)
    mean = torch.empty(T, device=dev)
    rstd = torch.empty(T, device=dev)
    dXn = torch.randn(T, H, device=dev, generator=g)
    dX = torch.empty(T, H, device=dev)
    dg = torch.empty(H, device=dev)
    db = torch.empty(H, device=dev)
    ws = torch.empty(m.mlpb_workspace_size(h), dtype=torch.uint8, device=dev)
    col = torch.empty(H, device=dev)
    fwd = _time(lambda: m.mlpb_layernorm_sp_fwd(h, X, gm, bt, Xn, mean, rstd), a.iters)
    bwd = _time(lambda: m.mlpb_layernorm_sp_bwd(h, X, gm, mean, rstd, dXn, dX, dg, db, ws),
                a.iters)
    cs = _time(lambda: m.mlpb_bias_grad_noalloc(X, col), a.iters)
    assert m.mlpb_last_device_error(h) == 0
    m.mlpb_destroy(h)
    # the branch's LayerNorm backward (dX = dY + LN'(dXn), in place), from its timing record
    br = m.MLPBranch(T, H, 8 * t, t, "swiglu", False)
    W1 = (0.02 * torch.randn(t, 2, 8, H, device=dev, generator=g)).to(torch.bfloat16)
    W2 = (0.02 * torch.randn(t, H, 8, device=dev, generator=g)).to(torch.bfloat16)
    dY = torch.randn(T, H, device=dev, generator=g).to(torch.bfloat16)
    grads = br.alloc_grads(W1, W2)
    for _ in range(3):
        br.forward(X, gm, bt, W1, None, W2, None)
        br.backward(X, gm, W1, W2, dY, grads)
    torch.cuda.synchronize()
    m.mlpb_enable_timing(br.handle, True)
    for _ in range(a.iters):
        br.forward(X, gm, bt, W1, None, W2, None)
        br.backward(X, gm, W1, W2, dY, grads)
    torch.cuda.synchronize()
    recs = [r for r in m.mlpb_read_timings(br.handle, 64 * a.iters) if r["name"] == "ln_bwd"]
    assert m.mlpb_last_device_error(br.handle) == 0
    br.close()
    res = sum(r["ms"] for r in recs) / len(recs) * 1e3
    n = T * H
    print(json.dumps({
        "tokens": T, "hidden": H, "tp": t,
        "ln_fwd_us": fwd, "ln_fwd_gbs": 4 * n / fwd / 1e3,
        "ln_bwd_us": bwd, "ln_bwd_gbs": 10 * n / bwd / 1e3,
        "bias_grad_us": cs, "bias_grad_gbs": 2 * n / cs / 1e3,
        "ln_bwd_residual_us": res, "ln_bwd_residual_gbs": 12 * n / res / 1e3,
    }))


if __name__ == "__main__":
    main()
