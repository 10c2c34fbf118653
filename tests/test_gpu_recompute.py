"""GPU parity of selective activation recomputation (MLPB_FLAG_RECOMPUTE_ACT).

The forward runs as usual; the A buffer is then filled with NaN, so that a backward that
read the forward's A would fail.  With the flag the dgrad epilogue rewrites A from the
saved Z (G, U) and dW2 consumes it.  Checked:
  * every gradient against the fp64 oracle within the parity gate, the bf16-storage
    oracle being the recomputing one (A = store(act(store(Z))));
  * the rewritten A against that oracle's A, bf16 unit by unit;
  * dX, dW1, db1, db2 bit-equal to the stored-A backward (recomputation moves dW2 only);
  * dW2 bit-equal to the stored-A backward run on the rewritten A.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import MLPShape, WORKLOADS, make_inputs, reduced_tokens
from oracle import mlp as omlp
from oracle.bf16 import round_bf16

from _harness import gate, to_f64

pytestmark = pytest.mark.gpu

RECOMPUTE = mlpb.MLPB_FLAG_RECOMPUTE_ACT

SHAPES = [
    pytest.param(MLPShape(384, 320, 1408, 4, "gelu", True), 81, id="gelu-t4-bias-ragged"),
    pytest.param(MLPShape(256, 192, 704, 8, "swiglu", False), 82, id="swiglu-t8-Fs88"),
    pytest.param(reduced_tokens(WORKLOADS[3], 512), 3, id="gelu-H5120-F20480-t8-T512"),
    pytest.param(reduced_tokens(WORKLOADS[4], 512), 4, id="swiglu-H4096-F11008-t8-T512"),
]


def _run(shape, g, flags, poison):
    blk = mlpb.MLPBlock(shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.act, shape.bias,
                        flags=flags)
    Y = blk.forward(g["X"], g["W1"], g["b1"], g["W2"], g["b2"])
    A_fwd = blk.A.clone()
    if poison:
        blk.A.fill_(float("nan"))
    grads = blk.backward(g["X"], g["W1"], g["W2"], g["dY"])
    torch.cuda.synchronize()
    assert mlpb.mlpb_last_device_error(blk.handle) == 0
    out = {"Y": Y, "A_fwd": A_fwd, "A": blk.A.clone(), "Z": blk.Z.clone(), **grads}
    return blk, out


@pytest.mark.parametrize("shape,wid", SHAPES)
def test_recompute_matches_oracle_and_stored_path(shape, wid):
    dev = torch.device("cuda:0")
    d = make_inputs(shape, wid)
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    blk_re, re = _run(shape, g, RECOMPUTE, poison=True)
    blk_re.close()
    blk_st, st = _run(shape, g, 0, poison=False)

    names = ["dX", "dW1", "db1", "db2"] if shape.bias else ["dX", "dW1"]
    for k in names:
        assert torch.equal(re[k], st[k]), f"{k} differs from the stored-A backward"
    # dW2 of the stored-A path, run on the rewritten A, is the recomputing path's dW2
    blk_st.A.copy_(re["A"])
    again = blk_st.backward(g["X"], g["W1"], g["W2"], g["dY"])
    torch.cuda.synchronize()
    assert torch.equal(again["dW2"], re["dW2"])
    blk_st.close()

    f = {k: to_f64(v) for k, v in d.items()}
    a = (f["X"], f["W1"], f["b1"], f["W2"], f["dY"], shape.act)
    exact = omlp.mlp_backward(*a)
    stored = omlp.mlp_backward(*a, store=round_bf16, recompute=True)
    for k in ["dX", "dW1", "dW2"] + (["db1", "db2"] if shape.bias else []):
        gate(k, to_f64(re[k]), exact[k], stored[k])
    fw = omlp.mlp_forward(f["X"], f["W1"], f["b1"], f["W2"], None, shape.act, round_bf16)
    check_recomputed_A(to_f64(re["A"]), fw, shape.act, shape.hidden)
    assert not torch.isnan(re["A"]).any()


def _unit(x):
    """One bf16 unit (2^-7 of the binade) at |x|; the subnormal quantum below it."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.where(x == 0.0, 2.0 ** -133, np.ldexp(1.0, np.maximum(e, -125) - 8))


def check_recomputed_A(got, fw, act, K):
    """A rewritten from the GPU's saved bf16 Z against A rewritten from the oracle's.

    The GPU's Z (G, U) comes from an fp32 accumulation of K = H products, the oracle's
    from an exact one; after rounding to bf16 the two may differ by one bf16 unit (next
    to a rounding boundary) plus the fp32 accumulation error itself, which matters only
    near zero: at most about sqrt(K) 2^-24 RMS(Z) in a random walk, taken here with a 4x
    margin.  The activation carries an input difference through its derivative, which can
    be many units of A where A is small (GELU's negative tail).  Bound per entry:
    |dA/dinput| x (one unit + the accumulation error) for each input, plus two units of A,
    plus the activation's own fp32 evaluation error.
    """
    def dev(x):
        return _unit(x) + 2.0 ** -22 * np.sqrt(K) * float(np.sqrt(np.mean(x * x)))

    if act == "swiglu":
        G, U = fw["G"], fw["U"]
        ref = round_bf16(omlp.silu(G) * U)
        slack = np.abs(U * omlp.silu_grad(G)) * dev(G) + np.abs(omlp.silu(G)) * dev(U)
    else:
        Z = fw["Z"]
        ref = round_bf16(omlp.gelu_tanh(Z))
        slack = np.abs(omlp.gelu_tanh_grad(Z)) * dev(Z)
    # fp32 evaluation of the activation: a few fp32 units on the data's scale (this also
    # covers tails where exp() under- or overflows and A is far below one fp32 unit)
    floor = 2.0 ** -20 * float(np.sqrt(np.mean(ref * ref)))
    bound = slack + 2.0 * _unit(ref) + floor
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (
        f"recomputed A: {int(bad.sum())} entries beyond the bound; worst "
        f"{float((np.abs(got - ref) / bound).max()):.3f} x bound")
    # and the bulk agrees to within one unit
    near = np.abs(got - ref) <= _unit(ref)
    assert near.mean() > 0.999, near.mean()
