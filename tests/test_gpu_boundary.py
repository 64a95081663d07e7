"""Checks at the GEMM boundary: nvfp4_dequantize_ex (BF16 output, inverse RHT) against the
oracle bit for bit, and the property that makes the columnwise RHT harmless to a weight-gradient
GEMM: 0.25 H16 d is orthogonal, so the product of two RHT-quantized columnwise operands (same
sign mask along the contraction) equals the product of their inverse-transformed
reconstructions, and approximates X^T W within the quantization error.

The codes fed to the GPU dequantization come from the oracle, so no expected value depends on
the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import api, workloads

pytestmark = pytest.mark.gpu


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


@pytest.mark.parametrize("inverse_rht", [False, True])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("shape,mask", [((64, 48), 0x1234), ((320, 1040), 0xB3C5),
                                        ((8192, 4096), 0x5A3C)])
def test_dequantize_ex_matches_oracle(shape, mask, inverse_rht, bf16):
    dev = _cuda()
    M, N = shape
    x = workloads.normal_with_outliers(M, N, seed=M + N, fraction=0.002, gain=40.0)
    cc, cs, gs = oracle.quantize_colwise(x, rht=True, sign_mask=mask)   # codes [N][M/2]
    got = api.nvfp4_dequantize_ex(torch.from_numpy(cc).to(dev), torch.from_numpy(cs).to(dev),
                                  torch.from_numpy(gs).to(dev), inverse_rht=inverse_rht,
                                  sign_mask=mask, bf16=bf16)
    torch.cuda.synchronize()
    ref = oracle.dequantize_ex(cc, cs, gs[1], inverse_rht=inverse_rht, sign_mask=mask, bf16=bf16)
    g = got.cpu().view(torch.int16).numpy().view(np.uint16) if bf16 else \
        got.cpu().numpy().view(np.uint32)
    r = ref if bf16 else ref.view(np.uint32)
    assert g.shape == r.shape
    assert np.array_equal(g, r), int((g != r).sum())


def test_rht_columnwise_gemm_equals_the_product_of_reconstructions():
    """X [M, K] and W [M, N] quantized columnwise with the RHT along M: cuBLASLt's NVFP4 GEMM of
    the codes = (inverse-RHT reconstruction of X)^T (that of W) to FP32 rounding, and close to
    X^T W itself."""
    dev = _cuda()
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no FP4 dtype")
    M, K, N = 512, 256, 128
    mask = 0x6A5C
    x = workloads.normal(M, K, 1.0, seed=91).to(dev)
    w = workloads.laplace(M, N, 0.1, seed=92).to(dev)
    qx = api.nvfp4_quantize(x, rowwise=False, columnwise=True, rht_col=True, sign_mask=mask)
    qw = api.nvfp4_quantize(w, rowwise=False, columnwise=True, rht_col=True, sign_mask=mask)
    try:
        out = torch._scaled_mm(qx["col_codes"].view(torch.float4_e2m1fn_x2),
                               qw["col_codes"].view(torch.float4_e2m1fn_x2).t(),
                               api.nvfp4_swizzle_scales(qx["col_scales"]).view(torch.float8_e4m3fn),
                               api.nvfp4_swizzle_scales(qw["col_scales"]).view(torch.float8_e4m3fn),
                               out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError) as e:
        pytest.skip("NVFP4 scaled_mm unavailable: %s" % str(e)[:120])
    got = out.double() * (float(qx["col_gscale"][1]) * float(qw["col_gscale"][1]))
    rx = api.nvfp4_dequantize_ex(qx["col_codes"], qx["col_scales"], qx["col_gscale"],
                                 inverse_rht=True, sign_mask=mask).double()   # [K, M]
    rw = api.nvfp4_dequantize_ex(qw["col_codes"], qw["col_scales"], qw["col_gscale"],
                                 inverse_rht=True, sign_mask=mask).double()   # [N, M]
    ref = rx @ rw.t()
    rel = ((got - ref).abs().max() / ref.abs().max()).item()
    assert rel < 1e-5, rel
    exact = x.double().t() @ w.double()
    err = ((got - exact).norm() / exact.norm()).item()
    assert err < 0.25, err  # two operands at ~20 dB SQNR each: ~0.14 expected
