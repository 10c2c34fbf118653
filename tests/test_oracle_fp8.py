"""Pins of the FP8 (E4M3) oracle against the number format and library conversions.

* round_e4m3 against torch's float8_e4m3fn conversion (a library routine) on values
  spread over every binade, subnormals and ties included, and on the format itself:
  every one of the 254 finite codes is a fixed point, every midpoint between two
  neighbours goes to the one with an even code;
* round_e4m3 against a table of values and codes that the format's definition in the
  OCP 8-bit floating point specification fixes (tests/golden/e4m3_ofp8.txt: the extreme
  normals and subnormals, ties to even in both directions, saturation), each code also
  decoded here bit by bit and, below 480, converted by torch;
* the scale exponent against its defining inequality;
* a quantized GEMM against the same product formed from torch's E4M3 codes;
* the FP8 block against the exact block within the error the format allows, and
  planted mistakes (truncation instead of rounding, a scale off by one power of two,
  a missing rescale) that the pins catch.
"""
import os

import numpy as np
import pytest
import torch

from oracle import fp8
from oracle import layernorm as oln
from oracle import mlp


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).float() \
        .double().numpy()


def _all_finite_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    v = codes.float().double().numpy()
    return np.unique(v[np.isfinite(v)])


def test_round_e4m3_matches_torch_conversion():
    r = np.random.default_rng(5)
    mags = np.ldexp(r.uniform(1.0, 2.0, 200000), r.integers(-14, 9, 200000))
    x = np.concatenate([mags, -mags, r.uniform(-2 ** -6, 2 ** -6, 20000)])
    x = x[np.abs(x) <= 448.0].astype(np.float32).astype(np.float64)  # torch converts fp32
    assert np.array_equal(fp8.round_e4m3(x), _torch_e4m3(x))


def _golden_e4m3():
    """Rows (input, E4M3 value, code, torch agrees) of tests/golden/e4m3_ofp8.txt."""
    def num(tok):
        return float.fromhex(tok) if "x" in tok.lower() else float(tok)
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "e4m3_ofp8.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, v, c, t = line.split()
                rows.append((num(a), num(v), int(c, 16), t == "1"))
    return rows


def _decode_e4m3(code):
    """An E4M3 code's value from the bit fields: sign, exponent (bias 7), mantissa."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    return sign * (2.0 ** (e - 7) * (1 + m / 8) if e else 2.0 ** -6 * (m / 8))


def test_round_e4m3_matches_the_format_table():
    rows = _golden_e4m3()
    assert len(rows) >= 20
    x = np.array([r[0] for r in rows])
    assert np.array_equal(fp8.round_e4m3(x), np.array([r[1] for r in rows]))
    for a, v, code, torch_agrees in rows:
        assert _decode_e4m3(code) == v, (a, hex(code))
        if torch_agrees:
            got = torch.tensor([a], dtype=torch.float32).to(torch.float8_e4m3fn) \
                .view(torch.uint8).item()
            assert got == code, (a, hex(got), hex(code))


def test_round_e4m3_fixed_points_and_ties_to_even():
    v = _all_finite_codes()
    assert v.size == 253 and v.max() == 448.0 and v.min() == -448.0  # +-0 merged
    assert np.array_equal(fp8.round_e4m3(v), v)
    pos = v[v >= 0]
    mid = (pos[:-1] + pos[1:]) / 2
    got = fp8.round_e4m3(mid)
    codes = torch.from_numpy(pos.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    even = {float(a): int(c) % 2 == 0 for a, c in zip(pos, codes.numpy())}
    for m, g, lo, hi in zip(mid, got, pos[:-1], pos[1:]):
        assert g in (lo, hi)
        assert even[float(g)], (m, g)
    assert fp8.round_e4m3(2.0 ** -10) == 0.0 and fp8.round_e4m3(3 * 2.0 ** -11) == 2.0 ** -9
    assert fp8.round_e4m3(1000.0) == 448.0 and fp8.round_e4m3(-1e9) == -448.0


def test_scale_exponent_definition():
    assert fp8.scale_exponent(0.0) == 0
    assert fp8.scale_exponent(448.0) == 0
    assert fp8.scale_exponent(1.75) == 8
    assert fp8.scale_exponent(1.0) == 8
    assert fp8.scale_exponent(448.00001) == -1
    r = np.random.default_rng(6)
    for a in np.ldexp(r.uniform(0.5, 1.0, 2000), r.integers(-40, 40, 2000)):
        k = fp8.scale_exponent(a)
        assert a * 2.0 ** k <= 448.0 < a * 2.0 ** (k + 1), (a, k)


def test_quantize_error_and_exact_grid():
    r = np.random.default_rng(7)
    x = r.standard_normal((64, 96))
    d, q, k = fp8.quantize(x)
    assert np.abs(q).max() <= 448.0 and np.array_equal(d, np.ldexp(q, -k))
    big = np.abs(x) * 2.0 ** k >= 2.0 ** -6          # normal range after scaling
    rel = np.abs(d - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-15             # half a unit of 3 mantissa bits
    grid = np.ldexp(np.rint(np.ldexp(x, 2)), -2)      # values on a 0.25 grid are exact
    grid = np.clip(grid, -3.5, 3.5)
    assert np.array_equal(fp8.deq(grid), grid)


def test_quantized_gemm_matches_torch_codes():
    r = np.random.default_rng(8)
    a, b = r.standard_normal((48, 80)), 0.02 * r.standard_normal((32, 80))
    ka, kb = fp8.scale_exponent(np.abs(a).max()), fp8.scale_exponent(np.abs(b).max())
    qa, qb = _torch_e4m3(np.ldexp(a, ka)), _torch_e4m3(np.ldexp(b, kb))
    want = (qa @ qb.T) * 2.0 ** -(ka + kb)
    got = fp8.deq(a) @ fp8.deq(b).T
    assert np.allclose(got, want, rtol=1e-13, atol=0)


def _inputs(T, H, F, t, act, bias, seed):
    r = np.random.default_rng(seed)
    Fs = F // t
    w1 = (t, 2, Fs, H) if act == "swiglu" else (t, Fs, H)
    return dict(X=r.standard_normal((T, H)), W1=0.02 * r.standard_normal(w1),
                b1=0.02 * r.standard_normal(F) if bias else None,
                W2=0.02 * r.standard_normal((t, H, Fs)),
                b2=0.02 * r.standard_normal(H) if bias else None, dY=r.standard_normal((T, H)))


def _rms_rel(a, b):
    return float(np.sqrt(np.mean((a - b) ** 2) / np.mean(b ** 2)))


@pytest.mark.parametrize("act,bias", [("gelu", True), ("swiglu", False)])
def test_fp8_block_within_format_error_of_exact_block(act, bias):
    """Each E4M3 operand carries a relative rounding error of at most 2^-4 (uniform-ish,
    RMS about 2^-4 / sqrt(3) ~ 3.6 %); a GEMM of two such operands is off by about
    sqrt(2) x that in RMS, ~5 %, and the backward chains two GEMMs.  So every output must
    be within 12 % RMS of the exact block, and -- the scales being undone -- above 0.5 %."""
    d = _inputs(64, 128, 256, 2, act, bias, 9)
    a = (d["X"], d["W1"], d["b1"], d["W2"])
    f8 = {**fp8.mlp_forward_fp8(*a, d["b2"], act), **fp8.mlp_backward_fp8(*a, d["dY"], act)}
    ex = {**mlp.mlp_forward(*a, d["b2"], act), **mlp.mlp_backward(*a, d["dY"], act)}
    for k in ("Y", "dX", "dW1", "dW2"):
        e = _rms_rel(f8[k], ex[k])
        assert 5e-3 < e < 0.12, (k, e)
    if bias:  # db2 sees dY itself; db1 the bf16 dZ of the fp8 dgrad
        assert np.array_equal(f8["db2"], ex["db2"])
        assert _rms_rel(f8["db1"], ex["db1"]) < 0.12


@pytest.mark.parametrize("act,bias", [("swiglu", False), ("gelu", True)])
def test_fp8_pre_ln_block_within_format_error_and_wired_to_its_own_dxn(act, bias):
    """block_fp8, the pre-LN block with E4M3 GEMMs, against the exact pre-LN block: every
    output that passes through a GEMM within the format's error (above 0.5 % and under
    12 % RMS, as for the MLP alone), Xn within one bf16 rounding (2^-8 relative) of the
    exact LayerNorm output, and the LayerNorm backward applied to the block's own dXn: each row of dX
    sums to zero, dbeta is the column sum of dXn."""
    d = _inputs(64, 128, 256, 2, act, bias, 11)
    r = np.random.default_rng(12)
    gamma, beta, eps = 1 + 0.1 * r.standard_normal(128), 0.02 * r.standard_normal(128), 1e-5
    f8 = fp8.block_fp8(d["X"], gamma, beta, eps, d["W1"], d["b1"], d["W2"], d["b2"], d["dY"],
                       act)
    ex = {**oln.block_forward(d["X"], gamma, beta, eps, d["W1"], d["b1"], d["W2"], d["b2"],
                              act, 2),
          **oln.block_backward(d["X"], gamma, beta, eps, d["W1"], d["b1"], d["W2"], d["dY"],
                               act, 2)}
    for k in ("Y", "dX", "dXn", "dW1", "dW2", "dgamma", "dbeta"):
        e = _rms_rel(f8[k], ex[k])
        assert 5e-3 < e < 0.12, (k, e)
    assert np.all(np.abs(f8["Xn"] - ex["Xn"]) <= np.abs(ex["Xn"]) * 2.0 ** -8)  # bf16 u
    scale = np.abs(f8["dX"]).max()
    assert np.all(np.abs(f8["dX"].sum(axis=1)) <= 1e-12 * 128 * scale)
    assert np.allclose(f8["dbeta"], f8["dXn"].sum(axis=0), rtol=1e-12, atol=0)


def test_fp8_block_identity_on_exact_grid():
    """With the identity activation and every operand (A too) on a grid E4M3 holds
    exactly at its tensor's scale, quantization changes nothing: Y equals the exact Y."""
    r = np.random.default_rng(10)
    X = np.ldexp(r.integers(-4, 5, (16, 64)), -2)          # multiples of 1/4, |x| <= 1
    W1 = np.zeros((2, 16, 64))
    for i in range(2):                                      # one 1/2 per row: Z = X[:, j]/2
        W1[i, np.arange(16), np.arange(16) + 16 * i] = 0.5
    W2 = np.ldexp(r.integers(-3, 4, (2, 32, 16)), -3)
    got = fp8.mlp_forward_fp8(X, W1, None, W2, None, "identity")["Y"]
    want = mlp.mlp_forward(X, W1, None, W2, None, "identity")["Y"]
    assert np.array_equal(got, want)


def _pins_pass():
    try:
        test_round_e4m3_matches_torch_conversion()
        test_round_e4m3_fixed_points_and_ties_to_even()
        test_scale_exponent_definition()
        test_quantize_error_and_exact_grid()
        test_quantized_gemm_matches_torch_codes()
        test_fp8_block_within_format_error_of_exact_block("gelu", True)
    except AssertionError:
        return False
    return True


def _mut_round_truncates(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.clip(np.ldexp(np.trunc(np.ldexp(m, 4)), e - 4), -448.0, 448.0)


def _mut_scale_one_too_high(amax):
    return 0 if amax == 0 else int(np.floor(np.log2(448.0 / amax))) + 1


def _mut_quantize_no_rescale(x):
    x = np.asarray(x, dtype=np.float64)
    k = fp8.scale_exponent(np.abs(x).max())
    q = fp8.round_e4m3(np.ldexp(x, k))
    return q, q, k


@pytest.mark.parametrize("attr,mutant", [
    ("round_e4m3", _mut_round_truncates),
    ("scale_exponent", _mut_scale_one_too_high),
    ("quantize", _mut_quantize_no_rescale),
])
def test_planted_fp8_mistake_is_caught(monkeypatch, attr, mutant):
    assert _pins_pass()
    monkeypatch.setattr(fp8, attr, mutant)
    assert not _pins_pass()
