"""GPU parity of mlpb_quantize_e4m3: E4M3 codes, scale exponent and amax bit for bit
against the FP8 oracle (quantization is integer work: exact equality is the bar)."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_tma_gb300 as mlpb
from inputs import make_bf16
from oracle import fp8

pytestmark = pytest.mark.gpu

CASES = [
    pytest.param((512, 5120), 1.0, 0, id="activation-like-512x5120"),
    pytest.param((80, 144), 1.0, 0, id="ragged-tiles-80x144"),
    pytest.param((8, 256, 352), 0.02, 0, id="batched-weight-like-8x256x352"),
    pytest.param((128, 256), 1.0, 24, id="wide-range-subnormal-codes"),
    pytest.param((64, 64), 3.0e4, 0, id="large-values-negative-exponent"),
]


def _decode(codes):
    return codes.view(torch.float8_e4m3fn).float().double().cpu().numpy()


@pytest.mark.parametrize("shape,std,spread", CASES)
def test_codes_scale_and_amax_bit_exact(shape, std, spread):
    x = make_bf16(shape, len(shape) * 1000 + shape[-1], std, spread)
    dev = torch.device("cuda:0")
    xd = x.to(dev)
    tshape = shape[:-2] + (shape[-1], shape[-2])
    q = torch.empty(shape, dtype=torch.uint8, device=dev)
    qt = torch.empty(tshape, dtype=torch.uint8, device=dev)
    for _ in range(2):  # the second call must not see the first call's amax
        amax, k = mlpb.mlpb_quantize_e4m3(xd, q, qt)
        torch.cuda.synchronize()
    xo = x.double().numpy()
    _, q_ref, k_ref = fp8.quantize(xo)
    assert int(k.item()) == k_ref
    amax_ref = np.float32(np.abs(xo).max())
    assert int(amax.item()) == int(amax_ref.view(np.int32))
    assert np.array_equal(_decode(q), q_ref)
    assert np.array_equal(_decode(qt), np.swapaxes(q_ref, -1, -2))
    # q alone and qt alone give the same codes
    q2 = torch.empty_like(q)
    mlpb.mlpb_quantize_e4m3(xd, q=q2)
    qt2 = torch.empty_like(qt)
    mlpb.mlpb_quantize_e4m3(xd, qt=qt2)
    torch.cuda.synchronize()
    assert torch.equal(q2, q) and torch.equal(qt2, qt)


def test_all_zero_tensor_and_argument_errors():
    dev = torch.device("cuda:0")
    x = torch.zeros((32, 48), dtype=torch.bfloat16, device=dev)
    q = torch.full((32, 48), 7, dtype=torch.uint8, device=dev)
    amax, k = mlpb.mlpb_quantize_e4m3(x, q)
    torch.cuda.synchronize()
    assert int(k.item()) == 0 and int(amax.item()) == 0 and int(q.sum().item()) == 0
    with pytest.raises(mlpb.MLPBError) as e:
        mlpb.mlpb_quantize_e4m3(torch.zeros((24, 48), dtype=torch.bfloat16, device=dev),
                                torch.empty((24, 48), dtype=torch.uint8, device=dev))
    assert e.value.status == mlpb.MLPB_EUNSUPPORTED  # rows % 16
    with pytest.raises(mlpb.MLPBError) as e:
        mlpb.mlpb_quantize_e4m3(x)                    # neither q nor qt
    assert e.value.status == mlpb.MLPB_EINVAL
