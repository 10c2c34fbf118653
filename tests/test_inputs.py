"""The seeded input generator: deterministic, right shapes, bf16, documented spreads."""
import torch

from inputs import WORKLOADS, make_inputs, reduced_tokens, sample_ffn_cols, sample_rows, workload


def test_inputs_are_deterministic_and_bf16():
    s = WORKLOADS[1]
    a, b = make_inputs(s, 1), make_inputs(s, 1)
    for k, v in a.items():
        if v is None:
            continue
        assert v.dtype == torch.bfloat16
        assert torch.equal(v, b[k]), k
    assert a["W1"].shape == (2, 512, 256) and a["W2"].shape == (2, 256, 512)
    assert a["X"].shape == (128, 256) and a["b1"].shape == (1024,)


def test_spreads_match_recipe():
    s = reduced_tokens(WORKLOADS[2], 1024)
    d = make_inputs(s, 2)
    assert abs(d["X"].float().std().item() - 1.0) < 0.02
    assert abs(d["W1"].float().std().item() - 0.02) < 0.001
    assert abs(d["b2"].float().std().item() - 0.02) < 0.004


def test_swiglu_and_ln_layouts():
    s = reduced_tokens(WORKLOADS[5], 256).__class__(256, 512, 1024, 8, "swiglu", False, sp_ln=True)
    d = make_inputs(s, 5)
    assert d["W1"].shape == (8, 2, 128, 512)
    assert d["b1"] is None and d["b2"] is None
    assert abs(d["gamma"].float().mean().item() - 1.0) < 0.02


def test_samples_cover_seams():
    s = workload(4)
    cols = sample_ffn_cols(s, 4).tolist()
    for i in range(s.tp):
        assert i * s.fs in cols and i * s.fs + s.fs - 1 in cols
    s5 = workload(5)
    rows = sample_rows(s5, 5).tolist()
    ts = s5.tokens // s5.tp
    for sh in range(s5.tp):
        assert sh * ts in rows and sh * ts + ts - 1 in rows
    assert rows == sorted(set(rows))


def test_gemm_flop_counts():
    assert WORKLOADS[3].gemm_flops() == 6 * 2 * 8192 * 5120 * 20480
    assert WORKLOADS[4].gemm_flops() == 2 * 16384 * 4096 * (2 * 11008 + 11008) * 3
