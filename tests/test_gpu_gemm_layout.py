"""The scale layout of the tensor-core block-scaled GEMMs (nvfp4_swizzle_scales), and an
independent check of the codes' packing and scale semantics: cuBLASLt's NVFP4 GEMM (through
torch._scaled_mm) run on this library's codes and tiled scales must give the product of the
dequantized tensors. A wrong nibble order, scale encoding or layout would make it disagree."""
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


@pytest.mark.parametrize("R,C", [(128, 4), (200, 10), (33, 3), (1, 1), (4096, 448), (300, 17)])
def test_swizzle_matches_oracle(R, C):
    dev = _cuda()
    rng = np.random.Generator(np.random.PCG64(R * 1000 + C))
    s = rng.integers(0, 256, size=(R, C), dtype=np.uint8)
    got = api.nvfp4_swizzle_scales(torch.from_numpy(s).to(dev)).cpu().numpy()
    assert np.array_equal(got, oracle.swizzle_scales(s))


def _scaled_mm_nvfp4(a_codes, a_scales, b_codes, b_scales):
    """cuBLASLt NVFP4 GEMM of two K-major operands [M, K/2] and [N, K/2] -> FP32 [M, N]
    (block scales only; the global scales are applied by the caller)."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no FP4 dtype")
    try:
        return torch._scaled_mm(a_codes.view(torch.float4_e2m1fn_x2),
                                b_codes.view(torch.float4_e2m1fn_x2).t(),
                                api.nvfp4_swizzle_scales(a_scales).view(torch.float8_e4m3fn),
                                api.nvfp4_swizzle_scales(b_scales).view(torch.float8_e4m3fn),
                                out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError) as e:
        pytest.skip("NVFP4 scaled_mm unavailable: %s" % str(e)[:120])


def _check(out, gs_a, gs_b, deq_a, deq_b):
    ref = deq_a.double() @ deq_b.double().t()
    got = out.double() * (float(gs_a[1]) * float(gs_b[1]))
    rel = ((got - ref).abs().max() / ref.abs().max()).item()
    assert rel < 1e-6, rel


def test_cublaslt_nvfp4_gemm_reads_rowwise_codes_and_tiled_scales():
    dev = _cuda()
    M, N, K = 256, 384, 1024
    a = workloads.normal_with_outliers(M, K, seed=81).to(dev)
    b = workloads.normal(N, K, 0.5, seed=82).to(dev)
    qa = api.nvfp4_quantize(a, rowwise=True)
    qb = api.nvfp4_quantize(b, rowwise=True)
    out = _scaled_mm_nvfp4(qa["row_codes"], qa["row_scales"], qb["row_codes"], qb["row_scales"])
    _check(out, qa["row_gscale"], qb["row_gscale"],
           api.nvfp4_dequantize(qa["row_codes"], qa["row_scales"], qa["row_gscale"]),
           api.nvfp4_dequantize(qb["row_codes"], qb["row_scales"], qb["row_gscale"]))


def test_cublaslt_nvfp4_gemm_reads_columnwise_outputs():
    """X^T W from the columnwise outputs of X [M, K] and W [M, N] (both K-major along M), the
    shape of a weight-gradient GEMM."""
    dev = _cuda()
    M, K, N = 512, 256, 128
    x = workloads.normal(M, K, 1.0, seed=83).to(dev)
    w = workloads.laplace(M, N, 0.1, seed=84).to(dev)
    qx = api.nvfp4_quantize(x, rowwise=False, columnwise=True)
    qw = api.nvfp4_quantize(w, rowwise=False, columnwise=True)
    out = _scaled_mm_nvfp4(qx["col_codes"], qx["col_scales"], qw["col_codes"], qw["col_scales"])
    _check(out, qx["col_gscale"], qw["col_gscale"],
           api.nvfp4_dequantize(qx["col_codes"], qx["col_scales"], qx["col_gscale"]),
           api.nvfp4_dequantize(qw["col_codes"], qw["col_scales"], qw["col_gscale"]))
