"""ctypes binding of libmlpb (the C ABI declared in include/mlpb.h).

Argument marshalling only: torch tensors are checked for dtype, shape, device and
contiguity and passed as raw device pointers with the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no fallback.
Loading fails loudly when libmlpb.so has not been built.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libmlpb.so")

MLPB_OK = 0
MLPB_EINVAL = -1
MLPB_EUNSUPPORTED = -2
MLPB_ECUDA = -3
MLPB_ETIMEOUT = -4
MLPB_ENOMEM = -5

MLPB_ACT_GELU_TANH = 0
MLPB_ACT_SWIGLU = 1
MLPB_FLAG_FAULT_INJECT = 0x1
MLPB_FLAG_ACCUMULATE_GRADS = 0x2
MLPB_FLAG_RECOMPUTE_ACT = 0x4
MLPB_FLAG_FP8 = 0x8
MLPB_FLAG_BF16_OUT = 0x10
MLPB_FLAG_EMULATE_COPIES = 0x20

# Every symbol include/mlpb.h declares.
EXPORTED = (
    "mlpb_create", "mlpb_destroy", "mlpb_workspace_size", "mlpb_saved_size", "mlpb_forward",
    "mlpb_backward", "mlpb_layernorm_sp_fwd", "mlpb_layernorm_sp_bwd", "mlpb_last_device_error",
    "mlpb_enable_timing", "mlpb_read_timings", "mlpb_status_str", "mlpb_bias_grad_noalloc",
    "mlpb_branch_forward", "mlpb_branch_backward", "mlpb_quantize_e4m3",
)


class mlpb_config(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64),
        ("tp", ctypes.c_int32), ("act", ctypes.c_int32), ("has_bias", ctypes.c_int32),
        ("seq_parallel_ln", ctypes.c_int32), ("ln_eps", ctypes.c_float), ("flags", ctypes.c_uint32),
    ]


class mlpb_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("ms", ctypes.c_float), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double), ("kernels", ctypes.c_int32)]


class MLPBError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmlpb.so and declares its signatures (idempotent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(the MLP block has no non-CUDA implementation)")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    H = ctypes.c_void_p
    sig = {
        "mlpb_create": (I, [ctypes.POINTER(mlpb_config), ctypes.POINTER(H)]),
        "mlpb_destroy": (None, [H]),
        "mlpb_workspace_size": (I, [H, ctypes.POINTER(Z)]),
        "mlpb_saved_size": (I, [H, ctypes.POINTER(Z), ctypes.POINTER(Z)]),
        "mlpb_forward": (I, [H, P, P, P, P, P, P, P, P, P, P]),
        "mlpb_backward": (I, [H, P, P, P, P, P, P, P, P, P, P, P, P, P]),
        "mlpb_layernorm_sp_fwd": (I, [H, P, P, P, P, P, P, P]),
        "mlpb_layernorm_sp_bwd": (I, [H, P, P, P, P, P, P, P, P, P, P]),
        "mlpb_last_device_error": (I, [H, P]),
        "mlpb_enable_timing": (I, [H, I]),
        "mlpb_read_timings": (I, [H, ctypes.POINTER(mlpb_kernel_time), I, ctypes.POINTER(I)]),
        "mlpb_status_str": (ctypes.c_char_p, [I]),
        "mlpb_bias_grad_noalloc": (I, [P, ctypes.c_int64, ctypes.c_int64, P, P]),
        "mlpb_branch_forward": (I, [H] + [P] * 15),
        "mlpb_branch_backward": (I, [H] + [P] * 19),
        "mlpb_quantize_e4m3": (I, [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P, P, P,
                                   P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load_library().mlpb_status_str(status).decode()


def _check(status: int, where: str):
    if status != MLPB_OK:
        raise MLPBError(status, where)


def _ptr(t, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclasses.dataclass
class Handle:
    ptr: int
    cfg: mlpb_config

    @property
    def shape(self):
        c = self.cfg
        return c.tokens, c.hidden, c.ffn, c.tp


def make_config(tokens, hidden, ffn, tp, act="gelu", has_bias=True, seq_parallel_ln=False,
                ln_eps=1e-5, flags=0) -> mlpb_config:
    return mlpb_config(tokens, hidden, ffn, tp,
                       MLPB_ACT_SWIGLU if act == "swiglu" else MLPB_ACT_GELU_TANH,
                       1 if has_bias else 0, 1 if seq_parallel_ln else 0, ln_eps, flags)


def mlpb_create(cfg: mlpb_config) -> Handle:
    h = ctypes.c_void_p()
    _check(load_library().mlpb_create(ctypes.byref(cfg), ctypes.byref(h)), "mlpb_create")
    return Handle(h.value, cfg)


def mlpb_destroy(h: Handle):
    if h is not None and h.ptr:
        load_library().mlpb_destroy(h.ptr)
        h.ptr = 0


def mlpb_workspace_size(h: Handle) -> int:
    n = ctypes.c_size_t()
    _check(load_library().mlpb_workspace_size(h.ptr, ctypes.byref(n)), "mlpb_workspace_size")
    return n.value


def mlpb_saved_size(h: Handle):
    z, a = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().mlpb_saved_size(h.ptr, ctypes.byref(z), ctypes.byref(a)),
           "mlpb_saved_size")
    return z.value, a.value


def out_dtype(c):
    """dtype of Y, dX (and the LayerNorm backward's dXn): bf16 under MLPB_FLAG_BF16_OUT."""
    return torch.bfloat16 if c.flags & MLPB_FLAG_BF16_OUT else torch.float32


def _w1_shape(c):
    fs = c.ffn // c.tp
    return (c.tp, 2, fs, c.hidden) if c.act == MLPB_ACT_SWIGLU else (c.tp, fs, c.hidden)


def mlpb_forward(h: Handle, X, W1, b1, W2, b2, Y, Zsaved, Asaved, workspace=None, stream=None):
    c = h.cfg
    T, Hd, F, t = c.tokens, c.hidden, c.ffn, c.tp
    bf = torch.bfloat16
    f1 = 2 * F if c.act == MLPB_ACT_SWIGLU else F
    args = [
        _ptr(X, bf, (T, Hd), "X"), _ptr(W1, bf, _w1_shape(c), "W1"), _ptr(b1, bf, (F,), "b1"),
        _ptr(W2, bf, (t, Hd, F // t), "W2"), _ptr(b2, bf, (Hd,), "b2"),
        _ptr(Y, out_dtype(c), (T, Hd), "Y"), _ptr(Zsaved, bf, (T, f1), "Zsaved"),
        _ptr(Asaved, bf, (T, F), "Asaved"), _ptr(workspace, None, None, "workspace"),
    ]
    _check(load_library().mlpb_forward(h.ptr, *args, _stream(stream)), "mlpb_forward")


def mlpb_backward(h: Handle, X, W1, W2, Zsaved, Asaved, dY, dX, dW1, dW2, db1, db2, workspace,
                  stream=None):
    c = h.cfg
    T, Hd, F, t = c.tokens, c.hidden, c.ffn, c.tp
    bf, f32 = torch.bfloat16, torch.float32
    f1 = 2 * F if c.act == MLPB_ACT_SWIGLU else F
    args = [
        _ptr(X, bf, (T, Hd), "X"), _ptr(W1, bf, _w1_shape(c), "W1"),
        _ptr(W2, bf, (t, Hd, F // t), "W2"), _ptr(Zsaved, bf, (T, f1), "Zsaved"),
        _ptr(Asaved, bf, (T, F), "Asaved"), _ptr(dY, bf, (T, Hd), "dY"),
        _ptr(dX, out_dtype(c), (T, Hd), "dX"), _ptr(dW1, f32, _w1_shape(c), "dW1"),
        _ptr(dW2, f32, (t, Hd, F // t), "dW2"), _ptr(db1, f32, (F,), "db1"),
        _ptr(db2, f32, (Hd,), "db2"), _ptr(workspace, None, None, "workspace"),
    ]
    _check(load_library().mlpb_backward(h.ptr, *args, _stream(stream)), "mlpb_backward")


def mlpb_layernorm_sp_fwd(h: Handle, X, gamma, beta, Xn, mean, rstd, stream=None):
    c = h.cfg
    T, Hd = c.tokens, c.hidden
    bf, f32 = torch.bfloat16, torch.float32
    args = [_ptr(X, bf, (T, Hd), "X"), _ptr(gamma, bf, (Hd,), "gamma"),
            _ptr(beta, bf, (Hd,), "beta"), _ptr(Xn, bf, (T, Hd), "Xn"),
            _ptr(mean, f32, (T,), "mean"), _ptr(rstd, f32, (T,), "rstd")]
    _check(load_library().mlpb_layernorm_sp_fwd(h.ptr, *args, _stream(stream)),
           "mlpb_layernorm_sp_fwd")


def mlpb_layernorm_sp_bwd(h: Handle, X, gamma, mean, rstd, dXn, dX, dgamma, dbeta, workspace,
                          stream=None):
    c = h.cfg
    T, Hd = c.tokens, c.hidden
    bf, f32 = torch.bfloat16, torch.float32
    args = [_ptr(X, bf, (T, Hd), "X"), _ptr(gamma, bf, (Hd,), "gamma"),
            _ptr(mean, f32, (T,), "mean"), _ptr(rstd, f32, (T,), "rstd"),
            _ptr(dXn, out_dtype(c), (T, Hd), "dXn"), _ptr(dX, out_dtype(c), (T, Hd), "dX"),
            _ptr(dgamma, f32, (Hd,), "dgamma"), _ptr(dbeta, f32, (Hd,), "dbeta"),
            _ptr(workspace, None, None, "workspace")]
    _check(load_library().mlpb_layernorm_sp_bwd(h.ptr, *args, _stream(stream)),
           "mlpb_layernorm_sp_bwd")


def mlpb_branch_forward(h: Handle, X, gamma, beta, W1, b1, W2, b2, Y, Xn, mean, rstd, Zsaved,
                        Asaved, workspace=None, stream=None):
    c = h.cfg
    T, Hd, F, t = c.tokens, c.hidden, c.ffn, c.tp
    bf, f32 = torch.bfloat16, torch.float32
    f1 = 2 * F if c.act == MLPB_ACT_SWIGLU else F
    args = [
        _ptr(X, bf, (T, Hd), "X"), _ptr(gamma, bf, (Hd,), "gamma"), _ptr(beta, bf, (Hd,), "beta"),
        _ptr(W1, bf, _w1_shape(c), "W1"), _ptr(b1, bf, (F,), "b1"),
        _ptr(W2, bf, (t, Hd, F // t), "W2"), _ptr(b2, bf, (Hd,), "b2"),
        _ptr(Y, out_dtype(c), (T, Hd), "Y"), _ptr(Xn, bf, (T, Hd), "Xn"),
        _ptr(mean, f32, (T,), "mean"),
        _ptr(rstd, f32, (T,), "rstd"), _ptr(Zsaved, bf, (T, f1), "Zsaved"),
        _ptr(Asaved, bf, (T, F), "Asaved"), _ptr(workspace, None, None, "workspace"),
    ]
    _check(load_library().mlpb_branch_forward(h.ptr, *args, _stream(stream)),
           "mlpb_branch_forward")


def mlpb_branch_backward(h: Handle, X, gamma, W1, W2, Xn, mean, rstd, Zsaved, Asaved, dY, dX,
                         dW1, dW2, db1, db2, dgamma, dbeta, workspace, stream=None):
    c = h.cfg
    T, Hd, F, t = c.tokens, c.hidden, c.ffn, c.tp
    bf, f32 = torch.bfloat16, torch.float32
    f1 = 2 * F if c.act == MLPB_ACT_SWIGLU else F
    args = [
        _ptr(X, bf, (T, Hd), "X"), _ptr(gamma, bf, (Hd,), "gamma"),
        _ptr(W1, bf, _w1_shape(c), "W1"), _ptr(W2, bf, (t, Hd, F // t), "W2"),
        _ptr(Xn, bf, (T, Hd), "Xn"), _ptr(mean, f32, (T,), "mean"), _ptr(rstd, f32, (T,), "rstd"),
        _ptr(Zsaved, bf, (T, f1), "Zsaved"), _ptr(Asaved, bf, (T, F), "Asaved"),
        _ptr(dY, bf, (T, Hd), "dY"), _ptr(dX, out_dtype(c), (T, Hd), "dX"),
        _ptr(dW1, f32, _w1_shape(c), "dW1"), _ptr(dW2, f32, (t, Hd, F // t), "dW2"),
        _ptr(db1, f32, (F,), "db1"), _ptr(db2, f32, (Hd,), "db2"),
        _ptr(dgamma, f32, (Hd,), "dgamma"), _ptr(dbeta, f32, (Hd,), "dbeta"),
        _ptr(workspace, None, None, "workspace"),
    ]
    _check(load_library().mlpb_branch_backward(h.ptr, *args, _stream(stream)),
           "mlpb_branch_backward")


def mlpb_quantize_e4m3(inp, q=None, qt=None, amax=None, scale_exp=None, stream=None):
    """E4M3 codes (uint8 tensors) of a bf16 CUDA tensor [rows][cols] or [batches][rows][cols]
    with one power-of-two scale; q in the input's layout, qt with the last two dimensions
    swapped.  Returns (amax bits as an int32 CUDA tensor, scale exponent int32 CUDA tensor)."""
    shape = tuple(inp.shape)
    b, r, c = (1,) + shape if len(shape) == 2 else shape
    dev = inp.device
    if amax is None:
        amax = torch.empty(1, dtype=torch.int32, device=dev)
    if scale_exp is None:
        scale_exp = torch.empty(1, dtype=torch.int32, device=dev)
    args = [_ptr(inp, torch.bfloat16, None, "in"), b, r, c,
            _ptr(q, torch.uint8, shape, "q"),
            _ptr(qt, torch.uint8, shape[:-2] + (c, r), "qt"),
            _ptr(amax, torch.int32, (1,), "amax"), _ptr(scale_exp, torch.int32, (1,), "scale_exp")]
    _check(load_library().mlpb_quantize_e4m3(*args, _stream(stream)), "mlpb_quantize_e4m3")
    return amax, scale_exp


def mlpb_last_device_error(h: Handle, stream=None) -> int:
    """Returns the status code (MLPB_OK, MLPB_ETIMEOUT, MLPB_ECUDA) without raising."""
    return load_library().mlpb_last_device_error(h.ptr, _stream(stream))


def mlpb_enable_timing(h: Handle, enable: bool = True):
    _check(load_library().mlpb_enable_timing(h.ptr, 1 if enable else 0), "mlpb_enable_timing")


def mlpb_read_timings(h: Handle, capacity: int = 64):
    buf = (mlpb_kernel_time * capacity)()
    n = ctypes.c_int()
    _check(load_library().mlpb_read_timings(h.ptr, buf, capacity, ctypes.byref(n)),
           "mlpb_read_timings")
    return [dict(name=buf[i].name.decode(), ms=buf[i].ms, flops=buf[i].flops,
                 bytes=buf[i].bytes, kernels=buf[i].kernels) for i in range(n.value)]


def mlpb_bias_grad_noalloc(inp, out, stream=None):
    """Column sums of a bf16 [rows][cols] CUDA tensor into the fp32 [cols] tensor `out`,
    with no device allocation (the library's fixed scratch array; see include/mlpb.h)."""
    rows, cols = inp.shape
    args = [_ptr(inp, torch.bfloat16, None, "in"), rows, cols,
            _ptr(out, torch.float32, (cols,), "out")]
    if out.device != inp.device:
        raise ValueError(f"in is on {inp.device} but out on {out.device}")
    # the library picks its scratch array and SM count from the current device, and the
    # stream must belong to that device too: make the tensors' device current
    with torch.cuda.device(inp.device):
        _check(load_library().mlpb_bias_grad_noalloc(*args, _stream(stream)),
               "mlpb_bias_grad_noalloc")


class MLPBlock:
    """Owns a handle plus the saved-activation and workspace buffers of one block shape.

    Convenience for callers that let torch allocate: forward() returns Y, backward()
    returns the gradient dict.  The arithmetic all happens in libmlpb.
    """

    def __init__(self, tokens, hidden, ffn, tp, act="gelu", has_bias=True,
                 seq_parallel_ln=False, ln_eps=1e-5, flags=0, device="cuda"):
        self.cfg = make_config(tokens, hidden, ffn, tp, act, has_bias, seq_parallel_ln, ln_eps,
                               flags)
        self.handle = mlpb_create(self.cfg)
        self.device = torch.device(device)
        f1 = 2 * ffn if act == "swiglu" else ffn
        self.act = act
        self.Z = torch.empty((tokens, f1), dtype=torch.bfloat16, device=self.device)
        self.A = torch.empty((tokens, ffn), dtype=torch.bfloat16, device=self.device)
        self.workspace = torch.empty(mlpb_workspace_size(self.handle), dtype=torch.uint8,
                                     device=self.device)

    def close(self):
        mlpb_destroy(self.handle)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, X, W1, b1, W2, b2, Y=None, stream=None):
        if Y is None:
            Y = torch.empty((self.cfg.tokens, self.cfg.hidden), dtype=out_dtype(self.cfg),
                            device=self.device)
        mlpb_forward(self.handle, X, W1, b1, W2, b2, Y, self.Z, self.A, self.workspace, stream)
        return Y

    def alloc_grads(self, W1, W2):
        """dX plus the parameter-gradient buffers; zeroed main-grad buffers when the handle
        accumulates (MLPB_FLAG_ACCUMULATE_GRADS)."""
        c = self.cfg
        has_b = bool(c.has_bias)
        new = torch.zeros if c.flags & MLPB_FLAG_ACCUMULATE_GRADS else torch.empty
        f32 = dict(dtype=torch.float32, device=self.device)
        return dict(
            dX=torch.empty((c.tokens, c.hidden), dtype=out_dtype(c), device=self.device),
            dW1=new(W1.shape, **f32),
            dW2=new(W2.shape, **f32),
            db1=new((c.ffn,), **f32) if has_b else None,
            db2=new((c.hidden,), **f32) if has_b else None,
        )

    def backward(self, X, W1, W2, dY, grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads(W1, W2)
        mlpb_backward(self.handle, X, W1, W2, self.Z, self.A, dY, g["dX"], g["dW1"], g["dW2"],
                      g["db1"], g["db2"], self.workspace, stream)
        return g


class MLPBranch(MLPBlock):
    """The sequence-parallel pre-norm MLP branch Y = X + MLP(LN(X)) of one shape: an
    MLPBlock whose handle has the LayerNorm enabled, plus the saved Xn, mean and rstd."""

    def __init__(self, tokens, hidden, ffn, tp, act="gelu", has_bias=True, ln_eps=1e-5,
                 flags=0, device="cuda"):
        super().__init__(tokens, hidden, ffn, tp, act, has_bias, True, ln_eps, flags, device)
        self.Xn = torch.empty((tokens, hidden), dtype=torch.bfloat16, device=self.device)
        self.mean = torch.empty((tokens,), dtype=torch.float32, device=self.device)
        self.rstd = torch.empty((tokens,), dtype=torch.float32, device=self.device)

    def forward(self, X, gamma, beta, W1, b1, W2, b2, Y=None, stream=None):
        if Y is None:
            Y = torch.empty((self.cfg.tokens, self.cfg.hidden), dtype=out_dtype(self.cfg),
                            device=self.device)
        mlpb_branch_forward(self.handle, X, gamma, beta, W1, b1, W2, b2, Y, self.Xn, self.mean,
                            self.rstd, self.Z, self.A, self.workspace, stream)
        return Y

    def alloc_grads(self, W1, W2):
        g = super().alloc_grads(W1, W2)
        new = torch.zeros if self.cfg.flags & MLPB_FLAG_ACCUMULATE_GRADS else torch.empty
        g["dgamma"] = new((self.cfg.hidden,), dtype=torch.float32, device=self.device)
        g["dbeta"] = new((self.cfg.hidden,), dtype=torch.float32, device=self.device)
        return g

    def backward(self, X, gamma, W1, W2, dY, grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads(W1, W2)
        mlpb_branch_backward(self.handle, X, gamma, W1, W2, self.Xn, self.mean, self.rstd, self.Z,
                             self.A, dY, g["dX"], g["dW1"], g["dW2"], g["db1"], g["db2"],
                             g["dgamma"], g["dbeta"], self.workspace, stream)
        return g
