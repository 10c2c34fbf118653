"""Parity at the full workload sizes, in the launch configuration the benchmark times.

For the GELU T8192/H5120/F20480/t8, SwiGLU T16384/H4096/F11008/t8 and SP pre-LN
SwiGLU T8192/H8192/F28672/t8 blocks:
  * every element at the same H, F and t with T = 512 tokens;
  * at full T, the outputs the oracle can compute one by one: 128 seeded token rows
    of Y and dX (rows 0, T-1 and every sequence shard's edges included), 64 seeded
    ffn features of dW1, dW2 and db1 (every shard seam included), and all of db2.
    The last shard's seams lie in the last M tiles, which the tail split of fc2, dX and
    dW1 cuts into K-ranges, so the sampled rows and features cross split tiles.
"""
import numpy as np
import pytest
import torch

from inputs import WORKLOADS, make_inputs, reduced_tokens, sample_ffn_cols, sample_rows
from oracle import layernorm as oln
from oracle import mlp as omlp
from oracle.bf16 import round_bf16

from _harness import check_full, fmt_rel, gate, oracle_refs, run_gpu, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BIG = [pytest.param(3, id="gelu-H5120-F20480-t8"), pytest.param(4, id="swiglu-H4096-F11008-t8"),
       pytest.param(5, id="sp-ln-swiglu-H8192-F28672-t8")]


@pytest.mark.parametrize("wid", BIG)
def test_reduced_tokens_every_element(wid):
    shape = reduced_tokens(WORKLOADS[wid], 512)
    d = make_inputs(shape, wid)
    gpu = run_gpu(shape, d)
    rel = check_full(shape, gpu, oracle_refs(shape, d))
    print(wid, fmt_rel(rel))


def _sampled_oracle(shape, f, rows, cols, store):
    if shape.sp_ln:
        r = oln.block_rows(f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"], f["W2"],
                           f["b2"], f["dY"], rows, shape.act, store)
        c = oln.block_ffn_cols(f["X"], f["gamma"], f["beta"], shape.ln_eps, f["W1"], f["b1"],
                               f["W2"], f["dY"], cols, shape.act, store)
    else:
        r = omlp.mlp_rows(f["X"], f["W1"], f["b1"], f["W2"], f["b2"], f["dY"], rows, shape.act,
                          store)
        c = omlp.mlp_ffn_cols(f["X"], f["W1"], f["b1"], f["W2"], f["dY"], cols, shape.act, store)
    return r, c


@pytest.mark.parametrize("wid", BIG)
def test_full_tokens_sampled(wid):
    shape = WORKLOADS[wid]
    d = make_inputs(shape, wid)
    gpu = run_gpu(shape, d)
    assert gpu["status"] == 0
    rows = sample_rows(shape, wid).numpy()
    cols = sample_ffn_cols(shape, wid).numpy()
    t, Fs = shape.tp, shape.fs
    ci, cj = cols // Fs, cols % Fs
    got = {
        "Y": to_f64(gpu["Y"][torch.from_numpy(rows).cuda()]),
        "dX": to_f64(gpu["dX"][torch.from_numpy(rows).cuda()]),
        "dW2": to_f64(gpu["dW2"][torch.from_numpy(ci).cuda(), :, torch.from_numpy(cj).cuda()]),
    }
    if shape.act == "swiglu":
        got["dW1"] = to_f64(gpu["dW1"][torch.from_numpy(ci).cuda(), :, torch.from_numpy(cj).cuda()])
    else:
        got["dW1"] = to_f64(gpu["dW1"][torch.from_numpy(ci).cuda(), torch.from_numpy(cj).cuda()])
    if shape.bias:
        got["db1"] = to_f64(gpu["db1"][torch.from_numpy(cols).cuda()])
        got["db2"] = to_f64(gpu["db2"])
    del gpu
    torch.cuda.empty_cache()
    f = {k: to_f64(v) for k, v in d.items()}
    ex_r, ex_c = _sampled_oracle(shape, f, rows, cols, None)
    st_r, st_c = _sampled_oracle(shape, f, rows, cols, round_bf16)
    rel = {}
    for k in ("Y", "dX"):
        rel[k] = gate(k, got[k], ex_r[k], st_r[k])
    for k in ("dW2", "dW1") + (("db1",) if shape.bias else ()):
        rel[k] = gate(k, got[k], ex_c[k], st_c[k])
    if shape.bias:
        db2 = f["dY"].sum(axis=0)
        rel["db2"] = gate("db2", got["db2"], db2, db2)
    print(wid, fmt_rel(rel))
