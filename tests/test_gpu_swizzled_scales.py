"""Scale outputs written by the quantize kernel itself in the 128 x 4 tiled layout of the
tensor-core block-scaled GEMMs (nvfp4_config.swizzle_scales; "[nvfp4_training] Optimize
CuteDSL kernels for NVFP4 training", "Config surface and AUTO": the reference's columnwise
scale store is hardwired to that layout).

Every output must equal the oracle's: codes and global scales as in row-major mode, and each
scale buffer byte for byte equal to oracle.swizzle_scales of the oracle's row-major scales,
the zero padding of partial 128 x 4 tiles included (the buffers are filled with a poison value
first). Modes cover both orientations, RHT + stochastic rounding, 2D tiles and the
single-launch amax; shapes cover whole tiles, several tiles with ragged row and column counts
(scale matrices that fill no whole tile), and the no-alloc entry point. cuBLASLt's NVFP4 GEMM
then reads the kernel's own tiled scales (no separate swizzle launch) and must give the
product of the dequantized tensors."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

MODES = {
    "rowcol": dict(rowwise=True, columnwise=True),
    "row_rtne_col_rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x4C3A,
                                round_col="sr", seed=21, offset=1),
    "row_sr": dict(rowwise=True, round_row="sr", seed=5),
    "col_rht": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0x0F0F),
    "2d_rowcol": dict(rowwise=True, columnwise=True, block2d=True),
    "2d_col": dict(rowwise=False, columnwise=True, block2d=True),
}
SHAPES = [(256, 512), (208, 272), (2048, 4096), (4160, 1296)]


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def _oracle(x_cpu, cfg):
    return oracle.quantize(x_cpu, oracle.Config(
        rowwise=cfg.get("rowwise", True), columnwise=cfg.get("columnwise", False),
        block2d=cfg.get("block2d", False), round_row_sr=cfg.get("round_row", "rn") == "sr",
        round_col_sr=cfg.get("round_col", "rn") == "sr", rht_col=cfg.get("rht_col", False),
        sign_mask=cfg.get("sign_mask", 0), seed=cfg.get("seed", 0), offset=cfg.get("offset", 0)))


def _poisoned(M, N, dev, cfg):
    out = api.alloc_outputs(M, N, dev, cfg.get("rowwise", True), cfg.get("columnwise", False),
                            swizzled=True)
    for v in out.values():
        v.fill_(0xA5 if v.dtype == torch.uint8 else float("nan"))
    return out


def _check(out, ref, what):
    for k, r in ref.items():
        g = out[k].cpu().numpy()
        if k.endswith("_scales"):
            r = oracle.swizzle_scales(r)
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), np.asarray(r).view(np.uint32)
        assert g.shape == r.shape, (what, k, g.shape, r.shape)
        bad = int((g != r).sum())
        assert bad == 0, "%s %s: %d bytes differ" % (what, k, bad)


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("fused", [False, True], ids=["two_pass", "fused"])
def test_tiled_scales_match_the_oracle(mode, shape, fused):
    dev = _cuda()
    M, N = shape
    cfg = dict(MODES[mode])
    x = workloads.normal_with_outliers(M, N, seed=M + 3 * N, fraction=0.003, gain=40.0)
    out = _poisoned(M, N, dev, cfg)
    api.nvfp4_quantize(x.to(dev), out=out, fused_amax=fused, swizzle_scales=True, **cfg)
    torch.cuda.synchronize()
    _check(out, _oracle(x, cfg), "%s %dx%d" % (mode, M, N))
    assert api.nvfp4_get_status(dev) == (0, 0)


def test_tiled_scales_through_the_noalloc_entry_point():
    dev = _cuda()
    L = _lib.load()
    for M, N in [(2048, 4096), (208, 272)]:
        cfg = dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1234,
                   round_col="sr", seed=3)
        x = workloads.normal_with_outliers(M, N, seed=M + N, fraction=0.003, gain=40.0)
        xd = x.to(dev)
        out = _poisoned(M, N, dev, cfg)
        c = api.make_config(swizzle_scales=True, **cfg)
        p = lambda k: ctypes.c_void_p(out[k].data_ptr())  # noqa: E731
        st = L.nvfp4_quantize_noalloc(ctypes.c_void_p(xd.data_ptr()), M, N, ctypes.byref(c),
                                      p("row_codes"), p("row_scales"), p("row_gscale"),
                                      p("col_codes"), p("col_scales"), p("col_gscale"),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        _check(out, _oracle(x, cfg), "noalloc %dx%d" % (M, N))


def test_tiled_scales_are_rejected_where_unsupported():
    dev = _cuda()
    x = workloads.normal(64, 64, 1.0, seed=1).to(dev)
    off = torch.tensor([32, 64], dtype=torch.int32, device=dev)
    L = _lib.load()
    c = api.make_config(rowwise=True, columnwise=True, swizzle_scales=True)
    o = api.alloc_outputs(64, 64, dev, True, True, col_ld=64, groups=2)
    p = lambda k: ctypes.c_void_p(o[k].data_ptr())  # noqa: E731
    st = L.nvfp4_quantize_grouped(ctypes.c_void_p(x.data_ptr()), 64, 64,
                                  ctypes.c_void_p(off.data_ptr()), 2, 64, ctypes.byref(c), None,
                                  None, p("row_codes"), p("row_scales"), p("row_gscale"),
                                  p("col_codes"), p("col_scales"), p("col_gscale"), None)
    assert _lib.STATUS_NAMES[st] == "NVFP4_ERR_UNSUPPORTED"
    c.swizzle_scales = 2
    st = L.nvfp4_quantize(ctypes.c_void_p(x.data_ptr()), 64, 64, ctypes.byref(c), None, None,
                          p("row_codes"), p("row_scales"), p("row_gscale"), None, None, None,
                          None)
    assert _lib.STATUS_NAMES[st] == "NVFP4_ERR_INVALID_ARG"


def _scaled_mm(a_codes, a_tiled, b_codes, b_tiled):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no FP4 dtype")
    try:
        return torch._scaled_mm(a_codes.view(torch.float4_e2m1fn_x2),
                                b_codes.view(torch.float4_e2m1fn_x2).t(),
                                a_tiled.view(torch.float8_e4m3fn),
                                b_tiled.view(torch.float8_e4m3fn), out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError) as e:
        pytest.skip("NVFP4 scaled_mm unavailable: %s" % str(e)[:120])


def test_cublaslt_nvfp4_gemm_reads_the_kernels_tiled_scales():
    """X^T W of a weight-gradient GEMM straight from the columnwise outputs (RHT + SR, whose
    transform cancels in the product) and A B^T from the rowwise outputs, the scales as the
    kernel wrote them."""
    dev = _cuda()
    M, K, N = 512, 256, 384
    a = workloads.normal_with_outliers(K, M, seed=91).to(dev)
    b = workloads.normal(N, M, 0.5, seed=92).to(dev)
    qa = api.nvfp4_quantize(a, rowwise=True, swizzle_scales=True)
    qb = api.nvfp4_quantize(b, rowwise=True, swizzle_scales=True)
    ref_a = api.nvfp4_quantize(a, rowwise=True)
    ref_b = api.nvfp4_quantize(b, rowwise=True)
    out = _scaled_mm(qa["row_codes"], qa["row_scales"], qb["row_codes"], qb["row_scales"])
    deq_a = api.nvfp4_dequantize(ref_a["row_codes"], ref_a["row_scales"], ref_a["row_gscale"])
    deq_b = api.nvfp4_dequantize(ref_b["row_codes"], ref_b["row_scales"], ref_b["row_gscale"])
    ref = deq_a.double() @ deq_b.double().t()
    got = out.double() * (float(qa["row_gscale"][1]) * float(qb["row_gscale"][1]))
    assert ((got - ref).abs().max() / ref.abs().max()).item() < 1e-6

    x = workloads.normal(M, K, 1.0, seed=93).to(dev)
    w = workloads.laplace(M, N, 0.1, seed=94).to(dev)
    kw = dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0x5AA5, round_col="sr",
              seed=8)
    qx = api.nvfp4_quantize(x, swizzle_scales=True, **kw)
    qw = api.nvfp4_quantize(w, swizzle_scales=True, **kw)
    rx = api.nvfp4_quantize(x, **kw)
    rw = api.nvfp4_quantize(w, **kw)
    out = _scaled_mm(qx["col_codes"], qx["col_scales"], qw["col_codes"], qw["col_scales"])
    deq_x = api.nvfp4_dequantize(rx["col_codes"], rx["col_scales"], rx["col_gscale"])
    deq_w = api.nvfp4_dequantize(rw["col_codes"], rw["col_scales"], rw["col_gscale"])
    ref = deq_x.double() @ deq_w.double().t()
    got = out.double() * (float(qx["col_gscale"][1]) * float(qw["col_gscale"][1]))
    assert ((got - ref).abs().max() / ref.abs().max()).item() < 1e-6
