"""The C ABI without a GPU: the library builds, loads, exports every symbol the header
declares, and rejects bad configurations before touching the device."""
import ctypes
import os
import re

import pytest

import megatron_tensor_transformer_tma_gb300 as mlpb
from megatron_tensor_transformer_tma_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mlpb.load_library()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "mlpb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mlpb_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    declared = _header_functions()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(mlpb.EXPORTED) == declared


def test_status_strings(lib):
    for code in range(0, -6, -1):
        assert mlpb.status_str(code) not in ("", "unknown status")
    assert mlpb.status_str(-99) == "unknown status"


@pytest.mark.parametrize("kw,status", [
    (dict(tokens=100), mlpb.MLPB_EUNSUPPORTED),          # T % 128
    (dict(hidden=96), mlpb.MLPB_EUNSUPPORTED),           # H % 64
    (dict(ffn=1000, tp=3), mlpb.MLPB_EUNSUPPORTED),      # F % t
    (dict(ffn=1028, tp=2), mlpb.MLPB_EUNSUPPORTED),      # (F/t) % 8
    (dict(act="swiglu", has_bias=True), mlpb.MLPB_EUNSUPPORTED),
    (dict(tokens=256, tp=3, ffn=768, seq_parallel_ln=True), mlpb.MLPB_EUNSUPPORTED),
    (dict(tp=0), mlpb.MLPB_EINVAL),
    (dict(hidden=0), mlpb.MLPB_EINVAL),
    (dict(tokens=-128), mlpb.MLPB_EINVAL),
    (dict(flags=0x80), mlpb.MLPB_EINVAL),
    (dict(flags=mlpb.MLPB_FLAG_FP8, ffn=1040), mlpb.MLPB_EUNSUPPORTED),  # F/t % 16
    (dict(flags=mlpb.MLPB_FLAG_FP8 | mlpb.MLPB_FLAG_RECOMPUTE_ACT), mlpb.MLPB_EUNSUPPORTED),
    (dict(seq_parallel_ln=True, ln_eps=0.0), mlpb.MLPB_EINVAL),
])
def test_create_rejects_bad_configs(lib, kw, status):
    args = dict(tokens=128, hidden=256, ffn=1024, tp=2, act="gelu", has_bias=True)
    args.update(kw)
    cfg = mlpb.make_config(**args)
    h = ctypes.c_void_p()
    assert lib.mlpb_create(ctypes.byref(cfg), ctypes.byref(h)) == status
    assert not h.value


def test_accumulate_flag_passes_config_validation(lib):
    """Without a GPU, a valid config fails only at the device query (ECUDA), so a flag
    that validation accepts shows as not-EINVAL and an unknown one as EINVAL."""
    for flags, ok in ((mlpb.MLPB_FLAG_ACCUMULATE_GRADS, True),
                      (mlpb.MLPB_FLAG_ACCUMULATE_GRADS | mlpb.MLPB_FLAG_FAULT_INJECT, True),
                      (mlpb.MLPB_FLAG_RECOMPUTE_ACT, True),
                      (mlpb.MLPB_FLAG_FP8, True),
                      (mlpb.MLPB_FLAG_BF16_OUT, True),
                      (mlpb.MLPB_FLAG_BF16_OUT | mlpb.MLPB_FLAG_FP8, True),
                      (0x40, False)):
        cfg = mlpb.make_config(128, 256, 1024, 2, "gelu", True, flags=flags)
        h = ctypes.c_void_p()
        st = lib.mlpb_create(ctypes.byref(cfg), ctypes.byref(h))
        if ok:
            assert st != mlpb.MLPB_EINVAL
            lib.mlpb_destroy(h)
        else:
            assert st == mlpb.MLPB_EINVAL and not h.value


def test_header_flag_values_match_binding():
    src = open(os.path.join(ROOT, "include", "mlpb.h")).read()
    for name in ("MLPB_FLAG_FAULT_INJECT", "MLPB_FLAG_ACCUMULATE_GRADS",
                 "MLPB_FLAG_RECOMPUTE_ACT", "MLPB_FLAG_FP8", "MLPB_FLAG_BF16_OUT",
                 "MLPB_FLAG_EMULATE_COPIES"):
        m = re.search(rf"#define\s+{name}\s+(0x[0-9a-fA-F]+)u", src)
        assert m and int(m.group(1), 16) == getattr(mlpb, name), name


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.mlpb_create(None, ctypes.byref(h)) == mlpb.MLPB_EINVAL
    n = ctypes.c_size_t()
    assert lib.mlpb_workspace_size(None, ctypes.byref(n)) == mlpb.MLPB_EINVAL
    assert lib.mlpb_forward(None, *([None] * 10)) == mlpb.MLPB_EINVAL
    assert lib.mlpb_backward(None, *([None] * 13)) == mlpb.MLPB_EINVAL
    lib.mlpb_destroy(None)


def test_other_entry_points_reject_bad_arguments_before_the_device(lib):
    """Null handles, null or misaligned pointers and unsupported sizes are refused on the
    host; the pointers below are never dereferenced (validation returns first)."""
    E, U = mlpb.MLPB_EINVAL, mlpb.MLPB_EUNSUPPORTED
    assert lib.mlpb_branch_forward(None, *([None] * 15)) == E
    assert lib.mlpb_branch_backward(None, *([None] * 19)) == E
    assert lib.mlpb_enable_timing(None, 1) == E
    count = ctypes.c_int()
    assert lib.mlpb_read_timings(None, None, 0, ctypes.byref(count)) == E
    assert lib.mlpb_last_device_error(None, None) == E
    a, b = 0x10000, 0x20000  # 16-byte aligned stand-ins
    # allocation-free column sum
    assert lib.mlpb_bias_grad_noalloc(None, 64, 256, b, None) == E      # rows > 0, no input
    assert lib.mlpb_bias_grad_noalloc(a, 64, 256, None, None) == E      # no output
    assert lib.mlpb_bias_grad_noalloc(a, -1, 256, b, None) == E
    assert lib.mlpb_bias_grad_noalloc(a, 64, 0, b, None) == E
    assert lib.mlpb_bias_grad_noalloc(a, 64, 260, b, None) == U         # cols % 8
    assert lib.mlpb_bias_grad_noalloc(a, 64, 1048576 + 8, b, None) == U  # beyond the scratch
    assert lib.mlpb_bias_grad_noalloc(a + 4, 64, 256, b, None) == E     # misaligned input
    assert lib.mlpb_bias_grad_noalloc(a, 64, 256, b + 8, None) == E     # misaligned output
    # E4M3 quantization
    q = lib.mlpb_quantize_e4m3
    assert q(a, 1, 64, 64, b, None, None, None, None) == E          # no amax word
    assert q(a, 1, 64, 64, None, None, b, None, None) == E          # neither q nor qt
    assert q(a, -1, 64, 64, b, None, b, None, None) == E
    assert q(a, 1, 72, 64, b, None, b, None, None) == U             # rows % 16
    assert q(a, 1, 64, 40, b, None, b, None, None) == U             # cols % 16
    assert q(None, 1, 64, 64, b, None, b, None, None) == E          # no input
    assert q(a + 8, 1, 64, 64, b, None, b, None, None) == E         # misaligned input
    assert q(a, 1, 64, 64, b, None, b + 2, None, None) == E         # misaligned amax
    assert q(a, 65536, 16, 16, b, None, b, None, None) == U         # grid z limit


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        mlpb.mlpb._ptr(torch.zeros(4), name="X")


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without libmlpb.so the binding raises: there is no other implementation to fall
    back to."""
    monkeypatch.setattr(mlpb.mlpb, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        mlpb.mlpb.load_library(str(tmp_path / "libmlpb.so"))
