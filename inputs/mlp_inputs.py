"""Workload shapes and seeded input draws for the MLP block.

Shapes follow the five workloads the block is measured on (a tiny GELU block,
two GELU blocks, a SwiGLU block and a sequence-parallel pre-LN SwiGLU block).
Distributions: X, dY ~ N(0, 1); weights and biases ~ N(0, 0.02^2);
LayerNorm gamma ~ 1 + N(0, 0.1^2), beta ~ N(0, 0.02^2).  Every tensor is
drawn in fp32 on the CPU with a ``torch.Generator`` seeded per tensor and
rounded once to bf16 (round to nearest even); the oracle and the GPU consume
exactly those bf16 values.

Layouts (shard-major, as each tensor-parallel rank would hold its slice):
  X, dY        [T, H]
  W1 (GELU)    [t, Fs, H]         W1 (SwiGLU) [t, 2, Fs, H]  (gate, then up)
  b1           [F]                (shard i owns b1[i*Fs:(i+1)*Fs])
  W2           [t, H, Fs]
  b2           [H]
  gamma, beta  [H]
"""
from __future__ import annotations

import dataclasses

import torch

SEED_BASE = 20261202

# tensor index k in the per-tensor seed ``SEED_BASE + 1000*workload + k``
_K = {"X": 0, "W1": 1, "b1": 2, "W2": 3, "b2": 4, "dY": 5, "gamma": 6,
      "beta": 7, "dXn": 8, "rows": 9, "cols": 10, "main": 11}


@dataclasses.dataclass(frozen=True)
class MLPShape:
    tokens: int
    hidden: int
    ffn: int
    tp: int
    act: str = "gelu"          # "gelu" (tanh form) or "swiglu"
    bias: bool = True
    sp_ln: bool = False        # sequence-parallel pre-LayerNorm in front of fc1
    ln_eps: float = 1e-5
    name: str = ""

    @property
    def fs(self) -> int:
        return self.ffn // self.tp

    @property
    def f1(self) -> int:
        """Output width of fc1: F for GELU, 2F (gate and up) for SwiGLU."""
        return 2 * self.ffn if self.act == "swiglu" else self.ffn

    def gemm_flops(self) -> int:
        """fwd+bwd GEMM flops: fc1, fc2, dA, dX, dW1, dW2."""
        T, H, F, F1 = self.tokens, self.hidden, self.ffn, self.f1
        return 2 * T * H * (F1 + F) * 3

    def with_tokens(self, tokens: int) -> "MLPShape":
        return dataclasses.replace(self, tokens=tokens)

    def with_tp(self, tp: int) -> "MLPShape":
        return dataclasses.replace(self, tp=tp)


WORKLOADS = {
    1: MLPShape(128, 256, 1024, 2, "gelu", True, name="tiny-gelu T128 H256 F1024 t2"),
    2: MLPShape(8192, 1024, 4096, 4, "gelu", True, name="gelu T8192 H1024 F4096 t4"),
    3: MLPShape(8192, 5120, 20480, 8, "gelu", True, name="gelu T8192 H5120 F20480 t8"),
    4: MLPShape(16384, 4096, 11008, 8, "swiglu", False,
                name="swiglu T16384 H4096 F11008 t8"),
    5: MLPShape(8192, 8192, 28672, 8, "swiglu", False, sp_ln=True, ln_eps=1e-5,
                name="sp-preln-swiglu T8192 H8192 F28672 t8"),
}


def workload(k: int, tp: int | None = None) -> MLPShape:
    s = WORKLOADS[k]
    return s if tp is None else s.with_tp(tp)


def _gen(wid: int, key: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + 1000 * wid + _K[key])
    return g


def _normal(shape, wid, key, std, mean=0.0):
    x = torch.randn(shape, generator=_gen(wid, key), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def make_inputs(shape: MLPShape, wid: int) -> dict:
    """All bf16 inputs of one forward+backward step, on the CPU."""
    T, H, F, t, Fs = shape.tokens, shape.hidden, shape.ffn, shape.tp, shape.fs
    if F % t:
        raise ValueError("ffn must be divisible by the tensor-parallel degree")
    w1_shape = (t, 2, Fs, H) if shape.act == "swiglu" else (t, Fs, H)
    d = {
        "X": _normal((T, H), wid, "X", 1.0),
        "W1": _normal(w1_shape, wid, "W1", 0.02),
        "W2": _normal((t, H, Fs), wid, "W2", 0.02),
        "dY": _normal((T, H), wid, "dY", 1.0),
        "b1": _normal((F,), wid, "b1", 0.02) if shape.bias else None,
        "b2": _normal((H,), wid, "b2", 0.02) if shape.bias else None,
    }
    if shape.sp_ln:
        d["gamma"] = _normal((H,), wid, "gamma", 0.1, mean=1.0)
        d["beta"] = _normal((H,), wid, "beta", 0.02)
    return d


def make_ln_grad(shape: MLPShape, wid: int) -> torch.Tensor:
    """A seeded fp32 upstream gradient for a stand-alone LayerNorm backward."""
    g = _gen(wid, "dXn")
    return torch.randn((shape.tokens, shape.hidden), generator=g, dtype=torch.float32)


def make_main_grads(shapes: dict, wid: int, scales: dict | None = None) -> dict:
    """Seeded fp32 starting contents of main-grad buffers (the state a gradient-
    accumulating backward adds into): one standard-normal tensor per name, in sorted
    name order from one generator, times ``scales[name]`` (default 1)."""
    g = _gen(wid, "main")
    out = {}
    for k in sorted(shapes):
        x = torch.randn(shapes[k], generator=g, dtype=torch.float32)
        out[k] = x.mul_(float((scales or {}).get(k, 1.0)))
    return out


def make_bf16(shape, seed: int, std: float = 1.0, log2_spread: int = 0) -> torch.Tensor:
    """A seeded bf16 tensor: N(0, std^2) values, each multiplied by 2^u with u uniform
    on the integers [-log2_spread, log2_spread] (a wide dynamic range when > 0)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + 7919 * seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32) * std
    if log2_spread:
        e = torch.randint(-log2_spread, log2_spread + 1, shape, generator=g)
        x = torch.ldexp(x, e)
    return x.to(torch.bfloat16)


def reduced_tokens(shape: MLPShape, tokens: int = 512) -> MLPShape:
    """Same H, F, t and activation with fewer tokens (a multiple of 128 and of t)."""
    return shape.with_tokens(min(shape.tokens, tokens))


def sample_rows(shape: MLPShape, wid: int, n: int = 128) -> torch.Tensor:
    """Seeded token rows, always including 0, T-1 and each seq shard's edges."""
    T = shape.tokens
    must = {0, T - 1}
    if shape.sp_ln:
        ts = T // shape.tp
        for s in range(shape.tp):
            must |= {s * ts, s * ts + ts - 1}
    perm = torch.randperm(T, generator=_gen(wid, "rows"))[:n].tolist()
    rows = sorted(must | set(perm[: max(0, n - len(must))]))
    return torch.tensor(rows, dtype=torch.int64)


def sample_ffn_cols(shape: MLPShape, wid: int, n: int = 64) -> torch.Tensor:
    """Seeded ffn indices f in [0, F), always including every shard's seams."""
    F, Fs = shape.ffn, shape.fs
    must = set()
    for i in range(shape.tp):
        must |= {i * Fs, i * Fs + Fs - 1}
    perm = torch.randperm(F, generator=_gen(wid, "cols"))[:n].tolist()
    cols = sorted(must | set(perm[: max(0, n - len(must))]))
    return torch.tensor(cols, dtype=torch.int64)


# ---------------------------------------------------------------- edge cases
# Seeds of the edge-case draws: SEED_BASE + 1000 * wid + 500 + k (k as in _K), apart from
# the workloads' own seeds.
def _edge_gen(wid: int, key: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + 1000 * wid + 500 + _K[key])
    return g


def make_saturating_inputs(shape: MLPShape, wid: int, z_std: float = 24.0) -> dict:
    """The block's inputs with fc1's weights drawn at std z_std / sqrt(H), so that the
    pre-activations Z (or G, U) have std ~ z_std: over a few hundred thousand entries
    |Z| reaches ~4.5 z_std, deep into the saturated tails of GELU and SiLU (past the
    point where exp(|x|) overflows fp32).  Everything else as make_inputs."""
    d = make_inputs(shape, wid)
    t, Fs, H = shape.tp, shape.fs, shape.hidden
    w1_shape = (t, 2, Fs, H) if shape.act == "swiglu" else (t, Fs, H)
    w = torch.randn(w1_shape, generator=_edge_gen(wid, "W1"), dtype=torch.float32)
    d["W1"] = w.mul_(z_std / float(H) ** 0.5).to(torch.bfloat16)
    return d


def make_zero_block_inputs(shape: MLPShape, wid: int) -> dict:
    """make_inputs with exact-zero blocks: X rows [64, 192) (crossing a 128-row tile
    boundary) and X columns [0, 32); dY rows [100, 228) and dY columns [32, 96)."""
    d = make_inputs(shape, wid)
    T, H = shape.tokens, shape.hidden
    X, dY = d["X"].clone(), d["dY"].clone()
    X[64:min(192, T)] = 0
    X[:, :min(32, H)] = 0
    dY[100:min(228, T)] = 0
    dY[:, 32:min(96, H)] = 0
    d["X"], d["dY"] = X, dY
    return d


LN_EDGE_KINDS = ("normal", "constant", "offset", "outlier")


def make_ln_edge_rows(T: int, H: int, wid: int) -> torch.Tensor:
    """A bf16 [T, H] LayerNorm input whose row r is of kind LN_EDGE_KINDS[r % 4]:
    normal N(0,1); constant (one N(0,1) value repeated: variance 0); offset (1e3 + N(0,1):
    a common offset 1000x the spread); outlier (N(0,1) with the first element set to 50,
    a 50-sigma value where a row's statistics start)."""
    g = _edge_gen(wid, "X")
    x = torch.randn((T, H), generator=g, dtype=torch.float32)
    c = torch.randn((T,), generator=g, dtype=torch.float32)
    kind = torch.arange(T) % 4
    x[kind == 1] = c[kind == 1][:, None].expand(-1, H)
    x[kind == 2] += 1000.0
    x[kind == 3, 0] = 50.0
    return x.to(torch.bfloat16)
