"""Parity of the MX kernels (nvfp4_mx_quantize / nvfp4_mx_dequantize, through the C ABI) with
the oracle, element by element and bit for bit: E8M0 scales and FP8/FP4 codes are integer
decisions both sides take from the same binary32 values (the block maximum's exponent and one
exact power-of-two product), and dequantized values are one rounding of an exact product.

Formats: MXFP8 E4M3 and E5M2, MXFP4 E2M1 (32-element blocks, E8M0 scales; readings M1-M4 of the
oracle). A cuBLASLt block-scaled GEMM on the library's MXFP8 outputs ties the layout and the
scale semantics to NVIDIA's own reading of the format.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import api, workloads

pytestmark = pytest.mark.gpu

FORMATS = ["e4m3", "e5m2", "e2m1"]


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def run_both(x_cpu, fmt, rowwise, columnwise):
    dev = _cuda()
    M, N = x_cpu.shape
    out = api.alloc_mx_outputs(M, N, dev, fmt, rowwise, columnwise)
    for v in out.values():
        v.fill_(0xA5)  # poison: every byte must be written
    api.nvfp4_mx_quantize(x_cpu.to(dev), fmt, rowwise, columnwise, out=out)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = {}
    if rowwise:
        ref["row_codes"], ref["row_scales"] = oracle.mx_quantize_rowwise(x_cpu, fmt)
    if columnwise:
        ref["col_codes"], ref["col_scales"] = oracle.mx_quantize_colwise(x_cpu, fmt)
    return got, ref


def assert_same(got, ref, what):
    for k, r in ref.items():
        g = got[k]
        assert g.shape == r.shape, (what, k, g.shape, r.shape)
        if not np.array_equal(g, r):
            bad = np.argwhere(g != r)
            i = tuple(bad[0])
            raise AssertionError("%s %s: %d mismatches, first at %s: gpu=%#x oracle=%#x"
                                 % (what, k, len(bad), i, g[i], r[i]))


ORIENT = {"row": (True, False), "col": (False, True), "rowcol": (True, True)}
# several 32 x 128 units, ragged right edges (a unit with one box, a unit with part of a box),
# rowwise-only row counts that are not multiples of 32
SHAPES = {
    "row": [(1, 32), (32, 128), (80, 288), (33, 4096), (257, 160), (64, 96)],
    "col": [(32, 8), (32, 136), (96, 200), (320, 1056), (64, 64)],
    "rowcol": [(32, 32), (64, 256), (96, 160), (320, 1056), (128, 2080)],
}
CASES = [(o, s) for o in ORIENT for s in SHAPES[o]]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%dx%d" % (c[0], c[1][0], c[1][1]))
def test_mx_matches_oracle(fmt, case):
    orient, (M, N) = case
    x = workloads.normal_with_outliers(M, N, seed=M * 7 + N, fraction=0.01, gain=50.0)
    got, ref = run_both(x, fmt, *ORIENT[orient])
    assert_same(got, ref, "%s %s %dx%d" % (fmt, orient, M, N))


@pytest.mark.parametrize("fmt", FORMATS)
def test_mx_every_exponent_and_special_values(fmt):
    """Random finite BF16 bit patterns of every exponent (huge, tiny, subnormal blocks: the
    exponent clamp and saturation), signed zeros and all-zero blocks."""
    M, N = 256, 512
    bits = workloads.random_bf16_bits((M, N), seed=91)
    bits[0:32, 0:32] = 0                       # an all-zero block in both orientations
    bits[32:64, 32:64] = 0x8000                # negative zeros
    bits[64:96, 0:64] &= 0x807F                # subnormals only
    bits[96:128, 64:128] |= 0x7F00             # the largest binades
    bits[96:128, 64:128] &= 0xFF7F
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    got, ref = run_both(x, fmt, True, True)
    assert_same(got, ref, "%s special" % fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_mx_dequantize_matches_oracle(fmt):
    dev = _cuda()
    x = workloads.normal_with_outliers(96, 640, seed=17, fraction=0.01, gain=50.0)
    q = api.nvfp4_mx_quantize(x.to(dev), fmt, True, True)
    for side in ("row", "col"):
        codes, scales = q[side + "_codes"], q[side + "_scales"]
        got = api.nvfp4_mx_dequantize(codes, scales, fmt).cpu().numpy()
        ref = oracle.mx_dequantize(codes.cpu().numpy(), scales.cpu().numpy(), fmt)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (fmt, side)


@pytest.mark.parametrize("fmt", FORMATS)
def test_mx_full_size_activation(fmt):
    """8192 x 4096, rowwise + columnwise: the launch configuration of the benchmark."""
    x = workloads.normal_with_outliers(8192, 4096, seed=3, fraction=0.001, gain=100.0)
    got, ref = run_both(x, fmt, True, True)
    assert_same(got, ref, "%s 8192x4096" % fmt)


def test_mx_rejects_bad_arguments():
    dev = _cuda()
    x = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    from nvfp4_block_scaled_quantize_gb300 import _lib
    with pytest.raises(_lib.NVFP4Error):
        api.nvfp4_mx_quantize(x[:, :48].contiguous(), "e4m3", True, False)  # N % 32
    with pytest.raises(_lib.NVFP4Error):
        api.nvfp4_mx_quantize(x[:48].contiguous(), "e4m3", False, True)     # M % 32
    with pytest.raises(ValueError):
        api.nvfp4_mx_quantize(x, "fp6", True, False)


def _swizzled_e8m0(scales):
    return api.nvfp4_swizzle_scales(scales).view(torch.float8_e8m0fnu)


@pytest.mark.parametrize("side", ["row", "col"])
def test_cublaslt_mxfp8_gemm_reads_the_outputs(side):
    """cuBLASLt's MXFP8 GEMM (torch._scaled_mm with E8M0 scales in the 128 x 4 tiled layout)
    on this library's E4M3 codes must give the product of the dequantized operands."""
    dev = _cuda()
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no E8M0 dtype")
    if side == "row":   # A [M, K] and B [N, K], both K-major
        a = workloads.normal_with_outliers(256, 1024, seed=85).to(dev)
        b = workloads.normal(384, 1024, 0.5, seed=86).to(dev)
        qa = api.nvfp4_mx_quantize(a, "e4m3", True, False)
        qb = api.nvfp4_mx_quantize(b, "e4m3", True, False)
    else:               # X^T W from the columnwise outputs of X [K, M] and W [K, N]
        a = workloads.normal(512, 256, 1.0, seed=87).to(dev)
        b = workloads.laplace(512, 128, 0.1, seed=88).to(dev)
        qa = api.nvfp4_mx_quantize(a, "e4m3", False, True)
        qb = api.nvfp4_mx_quantize(b, "e4m3", False, True)
    ca, sa = qa[side + "_codes"], qa[side + "_scales"]
    cb, sb = qb[side + "_codes"], qb[side + "_scales"]
    try:
        out = torch._scaled_mm(ca.view(torch.float8_e4m3fn), cb.view(torch.float8_e4m3fn).t(),
                               _swizzled_e8m0(sa), _swizzled_e8m0(sb), out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError) as e:
        pytest.skip("MXFP8 scaled_mm unavailable: %s" % str(e)[:120])
    da = torch.from_numpy(oracle.mx_dequantize(ca.cpu().numpy(), sa.cpu().numpy(), "e4m3"))
    db = torch.from_numpy(oracle.mx_dequantize(cb.cpu().numpy(), sb.cpu().numpy(), "e4m3"))
    ref = da.double() @ db.double().t()
    rel = ((out.cpu().double() - ref).abs().max() / ref.abs().max()).item()
    assert rel < 1e-6, rel
