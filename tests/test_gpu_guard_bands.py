"""Guard bands: every output buffer of every entry point sits between two 4 KiB bands of canary
bytes, and the bands must read back unchanged after the call. This catches writes past either
end of an output (a wrong leading dimension, a ragged tile or expert that overruns, a scale row
written once too often) without a memory checker. Shapes are ragged in both directions (tiles
and 16-row slabs cut short) and the grouped tensors have empty experts and a tail past the last
one. Each guarded call is also compared byte for byte with the same call on plain buffers
filled with the same body pattern, so a write that lands inside the wrong buffer, or a byte
left unwritten, shows up too (the parity tests check those outputs against the oracle)."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quantize_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

BAND = 4096    # bytes of canary on each side (keeps every view 4 KiB aligned)
CANARY = 0xA5
BODY = 0x5A    # what the output bytes hold before the call


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def _nbytes(shape, dtype):
    return int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()


class Guarded:
    """Output tensors carved out of larger byte buffers with canary bands on both sides."""

    def __init__(self, dev):
        self.dev, self.bufs = dev, []

    def empty(self, shape, dtype):
        n = _nbytes(shape, dtype)
        base = torch.full((BAND + n + BAND,), CANARY, dtype=torch.uint8, device=self.dev)
        base[BAND:BAND + n].fill_(BODY)
        self.bufs.append((base, n, tuple(shape), dtype))
        return base[BAND:BAND + n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        for base, n, shape, dtype in self.bufs:
            lo, hi = base[:BAND], base[BAND + n:]
            bad_lo = int((lo != CANARY).sum())
            bad_hi = int((hi != CANARY).sum())
            assert bad_lo == 0 and bad_hi == 0, \
                "%s: output %s %s: %d bytes before and %d after it overwritten" % (
                    what, shape, dtype, bad_lo, bad_hi)


def _plain(dev, shape, dtype):
    return torch.full((_nbytes(shape, dtype),), BODY, dtype=torch.uint8, device=dev).view(
        dtype).view(shape)


def _same_bytes(a, b, what):
    a = a.contiguous().view(torch.uint8).cpu().numpy()
    b = b.contiguous().view(torch.uint8).cpu().numpy()
    assert np.array_equal(a, b), (what, int((a != b).sum()))


def _outputs(make, M, N, rowwise, columnwise, col_ld=None, groups=None):
    g = () if groups is None else (groups,)
    ld = M if col_ld is None else col_ld
    out = {}
    if rowwise:
        out["row_codes"] = make((M, N // 2), torch.uint8)
        out["row_scales"] = make((M, N // 16), torch.uint8)
        out["row_gscale"] = make(g + (2,), torch.float32)
    if columnwise:
        out["col_codes"] = make((N, ld // 2), torch.uint8)
        out["col_scales"] = make((N, ld // 16), torch.uint8)
        out["col_gscale"] = make(g + (2,), torch.float32)
    return out


def _compare(got, ref, what):
    for k in ref:
        _same_bytes(got[k], ref[k], "%s %s" % (what, k))


SHAPES = [(80, 272), (304, 1040), (1040, 4112)]
MODES = {
    "rowcol_rn": dict(rowwise=True, columnwise=True),
    "row_sr": dict(rowwise=True, round_row="sr", seed=5),
    "col_rht_sr": dict(columnwise=True, rowwise=False, rht_col=True, sign_mask=0x9C31,
                       round_col="sr", seed=11, offset=4),
    "2d": dict(rowwise=True, columnwise=True, block2d=True),
    "fused_rowcol_rht": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x0FF0,
                             fused_amax=True),
    "fast_rht": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1234,
                     fast_math=True),
}


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
def test_quantize_writes_nothing_outside_its_outputs(mode, shape):
    dev = _cuda()
    M, N = shape
    cfg = MODES[mode]
    x = workloads.normal_with_outliers(M, N, seed=M + N, fraction=0.01, gain=40.0).to(dev)
    g = Guarded(dev)
    out = _outputs(g.empty, M, N, cfg.get("rowwise", True), cfg.get("columnwise", False))
    api.nvfp4_quantize(x, out=out, **cfg)
    g.check(mode)
    ref = _outputs(lambda s, d: _plain(dev, s, d), M, N, cfg.get("rowwise", True),
                   cfg.get("columnwise", False))
    api.nvfp4_quantize(x, out=ref, **cfg)
    _compare(out, ref, mode)


@pytest.mark.parametrize("block2d", [False, True], ids=["1d_rht_sr", "2d"])
def test_grouped_quantize_writes_nothing_outside_its_outputs(block2d):
    dev = _cuda()
    H = 272
    offs = np.array([0, 37, 37, 150, 391], dtype=np.int32)  # an empty first and third expert
    T = 420                                                 # a tail past the last expert
    cap = api.padded_capacity(np.diff(np.concatenate([[0], offs]))) + 16
    cfg = dict(block2d=True) if block2d else dict(rht_col=True, sign_mask=0x5A3C,
                                                  round_col="sr", seed=3)
    x = workloads.normal_with_outliers(T, H, seed=17, fraction=0.01, gain=40.0).to(dev)
    o = torch.from_numpy(offs).to(dev)
    E = len(offs)
    g = Guarded(dev)
    out = _outputs(g.empty, T, H, True, True, col_ld=cap, groups=E)
    api.nvfp4_quantize_grouped(x, o, col_capacity=cap, out=out, rowwise=True, columnwise=True,
                               **cfg)
    g.check("grouped")
    ref = _outputs(lambda s, d: _plain(dev, s, d), T, H, True, True, col_ld=cap, groups=E)
    api.nvfp4_quantize_grouped(x, o, col_capacity=cap, out=ref, rowwise=True, columnwise=True,
                               **cfg)
    _compare(out, ref, "grouped")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("shape", [(96, 320), (1056, 2080)], ids=lambda s: "%dx%d" % s)
def test_mx_quantize_writes_nothing_outside_its_outputs(fmt, shape):
    dev = _cuda()
    M, N = shape
    fp4 = fmt == "e2m1"
    x = workloads.normal_with_outliers(M, N, seed=M ^ N, fraction=0.01, gain=60.0).to(dev)

    def outs(make):
        return dict(row_codes=make((M, N // 2 if fp4 else N), torch.uint8),
                    row_scales=make((M, N // 32), torch.uint8),
                    col_codes=make((N, M // 2 if fp4 else M), torch.uint8),
                    col_scales=make((N, M // 32), torch.uint8))
    g = Guarded(dev)
    out = outs(g.empty)
    api.nvfp4_mx_quantize(x, fmt, True, True, out=out)
    g.check("mx " + fmt)
    ref = outs(lambda s, d: _plain(dev, s, d))
    api.nvfp4_mx_quantize(x, fmt, True, True, out=ref)
    _compare(out, ref, "mx " + fmt)


def test_other_entry_points_write_nothing_outside_their_outputs():
    dev = _cuda()
    L = _lib.load()
    vp = ctypes.c_void_p
    ptr = lambda t: vp(t.data_ptr())
    stream = vp(torch.cuda.current_stream().cuda_stream)
    M, N = 304, 1040
    x = workloads.normal_with_outliers(M, N, seed=23, fraction=0.01, gain=40.0).to(dev)
    q = api.nvfp4_quantize(x, rowwise=True, columnwise=True, rht_col=True, sign_mask=0x77)
    g = Guarded(dev)

    # amax
    cfg = api.make_config(rht_col=True, sign_mask=0x77)
    a_row, a_col = g.empty((1,), torch.float32), g.empty((1,), torch.float32)
    assert L.nvfp4_amax(ptr(x), M, N, ctypes.byref(cfg), ptr(a_row), ptr(a_col), stream) == 0
    # grouped amax
    offs = torch.tensor([0, 100, 100, 290], dtype=torch.int32, device=dev)
    ga_row, ga_col = g.empty((4,), torch.float32), g.empty((4,), torch.float32)
    assert L.nvfp4_amax_grouped(ptr(x), M, N, ptr(offs), 4, ctypes.byref(cfg), ptr(ga_row),
                                ptr(ga_col), stream) == 0
    # dequantize (FP32) and dequantize_ex (inverse RHT, BF16) of the columnwise outputs
    d32 = g.empty((N, M), torch.float32)
    assert L.nvfp4_dequantize(ptr(q["col_codes"]), ptr(q["col_scales"]), ptr(q["col_gscale"]),
                              N, M, ptr(d32), stream) == 0
    d16 = g.empty((N, M), torch.bfloat16)
    assert L.nvfp4_dequantize_ex(ptr(q["col_codes"]), ptr(q["col_scales"]),
                                 ptr(q["col_gscale"]), N, M, 1, 0x77, 1, ptr(d16), stream) == 0
    # scale swizzle (a ragged 304 x 65 scale matrix: partial 128-row and 4-column tiles)
    rs = q["row_scales"]
    sw = g.empty((((M + 127) // 128) * ((N // 16 + 3) // 4) * 512,), torch.uint8)
    assert L.nvfp4_swizzle_scales(ptr(rs), M, N // 16, ptr(sw), stream) == 0
    # MX dequantize
    mx = api.nvfp4_mx_quantize(x[:, :1024].contiguous(), "e2m1", True, False)
    mxd = g.empty((M, 1024), torch.float32)
    assert L.nvfp4_mx_dequantize(ptr(mx["row_codes"]), ptr(mx["row_scales"]), 2, M, 1024,
                                 ptr(mxd), stream) == 0
    # RMSNorm producer, and norm + quantize
    w = torch.linspace(0.5, 1.5, N, device=dev).to(torch.bfloat16)
    y, am = g.empty((M, N), torch.bfloat16), g.empty((1,), torch.float32)
    assert L.nvfp4_rmsnorm_amax(ptr(x), ptr(w), M, N, 1e-6, 0.0, ptr(y), ptr(am), stream) == 0
    qc = api.make_config(rowwise=True, columnwise=True)
    y2, am2 = g.empty((M, N), torch.bfloat16), g.empty((1,), torch.float32)
    nq = _outputs(g.empty, M, N, True, True)
    assert L.nvfp4_rmsnorm_quantize(ptr(x), ptr(w), M, N, 1e-6, 0.0, ctypes.byref(qc), ptr(y2),
                                    ptr(am2), ptr(nq["row_codes"]), ptr(nq["row_scales"]),
                                    ptr(nq["row_gscale"]), ptr(nq["col_codes"]),
                                    ptr(nq["col_scales"]), ptr(nq["col_gscale"]), stream) == 0
    # the allocation-free entry point
    na = _outputs(g.empty, M, N, True, True)
    assert L.nvfp4_quantize_noalloc(ptr(x), M, N, ctypes.byref(qc), ptr(na["row_codes"]),
                                    ptr(na["row_scales"]), ptr(na["row_gscale"]),
                                    ptr(na["col_codes"]), ptr(na["col_scales"]),
                                    ptr(na["col_gscale"]), stream) == 0
    g.check("other entry points")
    # and the guarded results are the plain calls' results
    ref_a = api.nvfp4_amax(x, rht_col=True, sign_mask=0x77)
    _same_bytes(a_row, ref_a[0], "amax row")
    _same_bytes(a_col, ref_a[1], "amax col")
    ref_ga = api.nvfp4_amax_grouped(x, offs, rht_col=True, sign_mask=0x77)
    _same_bytes(ga_row, ref_ga[0], "grouped amax row")
    _same_bytes(ga_col, ref_ga[1], "grouped amax col")
    _same_bytes(d32, api.nvfp4_dequantize(q["col_codes"], q["col_scales"], q["col_gscale"]),
                "dequantize")
    _same_bytes(d16, api.nvfp4_dequantize_ex(q["col_codes"], q["col_scales"], q["col_gscale"],
                                             inverse_rht=True, sign_mask=0x77, bf16=True),
                "dequantize_ex")
    _same_bytes(sw, api.nvfp4_swizzle_scales(rs), "swizzle")
    _same_bytes(mxd, api.nvfp4_mx_dequantize(mx["row_codes"], mx["row_scales"], "e2m1"),
                "mx dequantize")
    ref_y, ref_am = api.nvfp4_rmsnorm_amax(x, w)
    _same_bytes(y, ref_y, "rmsnorm y")
    _same_bytes(am, ref_am, "rmsnorm amax")
    _same_bytes(y2, ref_y, "rmsnorm_quantize y")
    ref_nq = api.nvfp4_rmsnorm_quantize(x, w, rowwise=True, columnwise=True)
    _compare(nq, {k: ref_nq[k] for k in nq}, "rmsnorm_quantize")
    ref_q = api.nvfp4_quantize(x, rowwise=True, columnwise=True)
    _compare(na, ref_q, "noalloc")
