"""GPU parity of the C-ABI path against the fp64 oracle (element by element).

Shapes span several 128 x 256 tiles and ragged tails: Fs not a multiple of 64 or 128
(shard seams inside a K block and inside an N tile), H = 64 mod 128 (a ragged N tile in
fc2, dX, dW1 and dW2, which is computed as its transpose), t = 1 and t = 8, with and
without bias, GELU and SwiGLU, and the sequence-parallel pre-LN block.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, WORKLOADS, make_inputs, make_ln_grad
from oracle import layernorm as oln

from _harness import check_full, compare, fmt_rel, oracle_refs, run_gpu, to_f64

pytestmark = pytest.mark.gpu

SMALL = [
    pytest.param(WORKLOADS[1], 1, id="tiny-gelu-t2"),
    pytest.param(MLPShape(256, 512, 2048, 4, "gelu", True), 11, id="gelu-t4-multitile"),
    pytest.param(MLPShape(384, 320, 1536, 1, "gelu", False), 12, id="gelu-t1-nobias-raggedH"),
    pytest.param(MLPShape(256, 192, 704, 8, "swiglu", False), 13, id="swiglu-t8-Fs88-raggedH"),
    pytest.param(MLPShape(512, 256, 2752, 2, "swiglu", False), 14, id="swiglu-t2-Fs1376"),
    # Fs = 160: each shard's one 256-column N tile of the SwiGLU dgrad is 96 columns of
    # padding; 64-wide B boxes straddle the shard's end (a K-block of fc2 too)
    pytest.param(MLPShape(256, 192, 480, 3, "swiglu", False), 19, id="swiglu-t3-Fs160-seams"),
    pytest.param(MLPShape(256, 256, 1024, 8, "gelu", True), 15, id="gelu-t8-Fs128"),
    pytest.param(MLPShape(256, 384, 1024, 4, "swiglu", False, sp_ln=True), 16, id="sp-ln-swiglu-t4"),
    pytest.param(MLPShape(128, 128, 512, 2, "gelu", True, sp_ln=True), 17, id="sp-ln-gelu-t2"),
    # 80 pair tiles on 76 pairs: fc2 and dX split their 4 tail tiles' K range 4 ways
    pytest.param(MLPShape(1024, 5120, 2048, 2, "gelu", True), 18, id="gelu-tail-split"),
    # T = 640: five 128-row M tiles (the last pair's odd CTA has no rows), and db2's column
    # sums over two row ranges of 320; F = 1344 (21 chunks of 64: the MN-major 3-D maps)
    pytest.param(MLPShape(640, 320, 1344, 4, "gelu", True), 20, id="gelu-t4-T640-oddM"),
]


@pytest.mark.parametrize("shape,wid", SMALL)
def test_small_shapes_every_element(shape, wid):
    d = make_inputs(shape, wid)
    gpu = run_gpu(shape, d)
    print(shape, fmt_rel(check_full(shape, gpu, oracle_refs(shape, d))))


@pytest.mark.parametrize("tp", [1, 4])
def test_gelu_h1024_f4096_full(tp):
    shape = WORKLOADS[2].with_tp(tp)
    d = make_inputs(shape, 2)
    gpu = run_gpu(shape, d)
    print(shape, fmt_rel(check_full(shape, gpu, oracle_refs(shape, d))))


def test_deterministic_bitwise():
    shape = MLPShape(256, 320, 1408, 4, "gelu", True)
    d = make_inputs(shape, 21)
    a = run_gpu(shape, d)
    b = run_gpu(shape, d)
    for k in ("Y", "dX", "dW1", "dW2", "db1", "db2"):
        assert torch.equal(a[k], b[k]), k


def test_timing_records_and_serialised_schedule_are_bitwise_equal():
    """With per-kernel timing on, the backward runs on one stream: its outputs equal the
    two-stream schedule's bit for bit, and every launch has a record with its algorithmic
    flops and bytes."""
    shape = MLPShape(256, 512, 2048, 4, "gelu", True)
    d = make_inputs(shape, 22)
    a = run_gpu(shape, d)
    b = run_gpu(shape, d, timing=True)
    assert a["status"] == 0 and b["status"] == 0
    for k in ("Y", "dX", "dW1", "dW2", "db1", "db2", "Z", "A"):
        assert torch.equal(a[k], b[k]), k
    recs = b["timings"]
    assert [r["name"] for r in recs] == ["fc1_gelu", "fc2", "w2_transpose_db2", "dgrad_gelu",
                                         "wgrad_w2", "bias_sums", "wgrad_w1", "dgrad_x"]
    T, H, F = shape.tokens, shape.hidden, shape.ffn
    for r in recs:
        assert r["ms"] > 0.0 and r["bytes"] > 0.0 and r["kernels"] == 1
        if r["name"] in ("w2_transpose_db2", "bias_sums"):
            assert r["flops"] == 0.0
        else:
            assert r["flops"] == 2.0 * T * H * F


@pytest.mark.parametrize("T,H,t", [
    pytest.param(1024, 8192, 8, id="H8192-4-vectors-a-thread"),
    pytest.param(512, 16384, 4, id="H16384-max-8-vectors"),
    pytest.param(384, 12352, 3, id="H12352-8-vectors-ragged"),
    pytest.param(256, 3072, 2, id="H3072-2-vectors"),
    pytest.param(128, 64, 2, id="H64-min"),
])
def test_layernorm_sp_components(T, H, t):
    """K8 / K9 alone on seeded inputs (the upstream dXn is seeded, not produced here), for
    every register-block width the kernels instantiate (1, 2, 4, 8 vectors a thread)."""
    shape = MLPShape(T, H, 8 * t, t, "swiglu", False, sp_ln=True)
    d = make_inputs(shape, 31)
    dXn = make_ln_grad(shape, 31)
    dev = torch.device("cuda:0")
    h = mlpb.mlpb_create(mlpb.make_config(T, H, 8 * t, t, "swiglu", False, True, 1e-5))
    X, gm, bt = d["X"].to(dev), d["gamma"].to(dev), d["beta"].to(dev)
    Xn = torch.empty_like(X)
    mean = torch.empty(T, device=dev)
    rstd = torch.empty(T, device=dev)
    mlpb.mlpb_layernorm_sp_fwd(h, X, gm, bt, Xn, mean, rstd)
    ws = torch.empty(mlpb.mlpb_workspace_size(h), dtype=torch.uint8, device=dev)
    dX = torch.empty((T, H), device=dev)
    dg = torch.empty(H, device=dev)
    db = torch.empty(H, device=dev)
    mlpb.mlpb_layernorm_sp_bwd(h, X, gm, mean, rstd, dXn.to(dev), dX, dg, db, ws)
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(h) == 0
    mlpb.mlpb_destroy(h)
    x64, g64, b64 = to_f64(d["X"]), to_f64(d["gamma"]), to_f64(d["beta"])
    rXn, rmu, rrs = oln.layernorm_sp_fwd(x64, g64, b64, 1e-5, t)
    # Xn is bf16: within one bf16 rounding of the oracle plus 1e-3 RMS
    got = to_f64(Xn)
    assert np.all(np.abs(got - rXn) <= np.abs(rXn) * 2.0 ** -8 + 1e-3 * np.sqrt(np.mean(rXn ** 2)))
    # the mean is judged on the scale of the data it averages (rows have std ~1)
    assert np.abs(to_f64(mean) - rmu).max() <= 1e-5 * np.sqrt(np.mean(x64 ** 2))
    compare("rstd", to_f64(rstd), rrs, tol=1e-5)
    rdX, rdg, rdb = oln.layernorm_sp_bwd(x64, g64, rmu, rrs, to_f64(dXn), t)
    compare("ln_dX", to_f64(dX), rdX, tol=1e-4)
    compare("dgamma", to_f64(dg), rdg, tol=1e-4)
    compare("dbeta", to_f64(db), rdb, tol=1e-4)


def test_empty_batch_zero_grads():
    shape = MLPShape(0, 256, 1024, 2, "gelu", True)
    d = make_inputs(MLPShape(128, 256, 1024, 2, "gelu", True), 41)
    dev = torch.device("cuda:0")
    blk = mlpb.MLPBlock(0, 256, 1024, 2, "gelu", True)
    X = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    W1, W2 = d["W1"].to(dev), d["W2"].to(dev)
    Y = blk.forward(X, W1, d["b1"].to(dev), W2, d["b2"].to(dev))
    g = blk.alloc_grads(W1, W2)
    for v in g.values():
        v.fill_(7.0)
    blk.backward(X, W1, W2, torch.empty((0, 256), dtype=torch.bfloat16, device=dev), g)
    torch.cuda.synchronize()
    assert Y.shape == (0, 256)
    for k in ("dW1", "dW2", "db1", "db2"):
        assert torch.count_nonzero(g[k]).item() == 0, k
    blk.close()
    del shape


def test_host_validation_launches_nothing():
    dev = torch.device("cuda:0")
    blk = mlpb.MLPBlock(128, 256, 1024, 2, "gelu", True)
    X = torch.zeros((128 * 256 + 1,), dtype=torch.bfloat16, device=dev)[1:].view(128, 256)
    W1 = torch.zeros((2, 512, 256), dtype=torch.bfloat16, device=dev)
    W2 = torch.zeros((2, 256, 512), dtype=torch.bfloat16, device=dev)
    b1 = torch.zeros(1024, dtype=torch.bfloat16, device=dev)
    b2 = torch.zeros(256, dtype=torch.bfloat16, device=dev)
    with pytest.raises(mlpb.MLPBError) as e:
        blk.forward(X, W1, b1, W2, b2)  # X misaligned by 2 bytes
    assert e.value.status == mlpb.MLPB_EINVAL
    with pytest.raises(mlpb.MLPBError) as e:
        blk.forward(X.clone(), W1, None, W2, b2)  # bias config without b1
    assert e.value.status == mlpb.MLPB_EINVAL
    assert mlpb.mlpb_last_device_error(blk.handle) == 0
    blk.close()


def test_bounded_wait_reports_timeout_and_context_survives():
    """The producer skips one arrive (a flag nothing else sets); the consumer's bounded
    wait expires, the kernel drains, frees tensor memory and returns; the host reads
    MLPB_ETIMEOUT, and the next call on a fresh handle is correct."""
    shape = WORKLOADS[1]
    d = make_inputs(shape, 1)
    bad = run_gpu(shape, d, flags=mlpb.MLPB_FLAG_FAULT_INJECT)
    assert bad["status"] == mlpb.MLPB_ETIMEOUT
    good = run_gpu(shape, d)
    check_full(shape, good, oracle_refs(shape, d))
