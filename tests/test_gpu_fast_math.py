"""The fast-math variant (nvfp4_config.fast_math = 1), bounded against the exact path.

The fast variant ("NVFP4 quantization kernels: CuteDSL and Triton", section "Fast math") has
two parts: element multipliers from the hardware's approximate reciprocal (rcp.approx.ftz)
instead of a correctly rounded 1 / (s * S_dec), and, with the RHT, columnwise block scales and
codes taken from the FP32 transform without its BF16 round-through. Neither can be reproduced
on the CPU bit for bit, so this variant has no oracle of its own; the pages tie it to the exact
path by a signal-to-noise floor of 25 dB (fast against exact), and that is what is tested here,
next to the properties that hold exactly:
  - the amax and the global scales are exact in both modes (bit-identical);
  - rowwise and plain columnwise block scales do not depend on the reciprocal (bit-identical);
  - a code can only move to a neighbouring E2M1 magnitude, with the same sign;
  - with round-to-nearest and no RHT, a code moves only where the exact scaled value x * r
    (the oracle's) lies at an E2M1 midpoint to within the reciprocal's error;
  - with the RHT, a columnwise block scale moves by at most one E4M3 step;
  - 2D (weight) quantization has no fast variant: its output is bit-identical;
  - the fused-amax launch and the two-pass pipeline agree bit for bit in fast mode.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import api, workloads

pytestmark = pytest.mark.gpu

KEYS = ("row_codes", "row_scales", "row_gscale", "col_codes", "col_scales", "col_gscale")
SQNR_FLOOR_DB = 25.0
MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float64)


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def _np(out):
    return {k: v.cpu().numpy() for k, v in out.items()}


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _nibbles(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return np.stack([c & 0xF, c >> 4], axis=-1).reshape(c.shape[0], -1)


def sqnr_db(ref, test):
    noise = float(np.sum((ref.astype(np.float64) - test.astype(np.float64)) ** 2))
    sig = float(np.sum(ref.astype(np.float64) ** 2))
    return float("inf") if noise == 0.0 else 10.0 * np.log10(sig / noise)


def dequant(o, side, s_dec_row=1):
    return oracle.dequantize(o[side + "_codes"], o[side + "_scales"],
                             o[side + "_gscale"].reshape(-1)[s_dec_row])


def assert_codes_adjacent(exact, fast, what):
    e, f = _nibbles(exact), _nibbles(fast)
    assert np.array_equal(e & 8, f & 8), "%s: a code changed sign" % what
    step = np.abs((e & 7).astype(int) - (f & 7).astype(int))
    assert step.max(initial=0) <= 1, "%s: a code moved by %d E2M1 steps" % (what, step.max())


def exact_scaled_rowwise(x_cpu, o):
    """The oracle's x * r per element (rowwise, exact mode) from its scales and global scale."""
    s_dec = o["row_gscale"][1]
    table = np.array([oracle.element_multiplier(s, s_dec) for s in range(256)], dtype=np.float32)
    r = np.repeat(table[o["row_scales"]], 16, axis=1)
    xf = x_cpu.float().numpy()
    return (xf * r).astype(np.float32)


def run(x, **cfg):
    out = api.nvfp4_quantize(x, **cfg)
    torch.cuda.synchronize()
    return _np(out)


PLAIN = {
    "row_rn": dict(rowwise=True),
    "col_rn": dict(rowwise=False, columnwise=True),
    "rowcol_rn": dict(rowwise=True, columnwise=True),
    "rowcol_sr": dict(rowwise=True, columnwise=True, round_row="sr", round_col="sr", seed=21),
}

RHT = {
    "col_rht": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0xB3C5),
    "col_rht_sr": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0x0F0F,
                       round_col="sr", seed=33, offset=4),
    "rowcol_rht": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1234),
    "rowcol_rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x5A3C,
                          round_col="sr", seed=4),
    "rowcol_rht_sr_both": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x7777,
                               round_row="sr", round_col="sr", seed=6),
}


@pytest.mark.parametrize("mode", sorted(PLAIN))
def test_fast_plain_modes_bounded_by_exact(mode):
    dev = _cuda()
    cfg = PLAIN[mode]
    x_cpu = workloads.normal_with_outliers(1024, 2048, seed=17, fraction=0.002, gain=40.0)
    x = x_cpu.to(dev)
    ex, fa = run(x, **cfg), run(x, fast_math=True, **cfg)
    for side in ("row", "col"):
        if side + "_codes" not in ex:
            continue
        for k in ("_gscale", "_scales"):
            assert np.array_equal(_bits(ex[side + k]), _bits(fa[side + k])), (mode, side + k)
        assert_codes_adjacent(ex[side + "_codes"], fa[side + "_codes"], mode + "/" + side)
        diff = np.mean(ex[side + "_codes"] != fa[side + "_codes"])
        assert diff < 0.05, (mode, side, diff)
        db = sqnr_db(dequant(ex, side), dequant(fa, side))
        assert db >= SQNR_FLOOR_DB, (mode, side, db)


def test_fast_rowwise_rn_flips_only_at_midpoints():
    """Round-to-nearest without the RHT: only the multiplier differs, by the reciprocal's
    error, so an element's code can move only where the exact x * r sits on a midpoint."""
    dev = _cuda()
    x_cpu = workloads.normal_with_outliers(2048, 4096, seed=224, fraction=0.002, gain=40.0)
    x = x_cpu.to(dev)
    fa = run(x, rowwise=True, fast_math=True)
    rc, rs, rg = oracle.quantize_rowwise(x_cpu)
    ref = dict(row_codes=rc, row_scales=rs, row_gscale=rg)
    assert np.array_equal(fa["row_scales"], rs)
    ef, ff = _nibbles(rc), _nibbles(fa["row_codes"])
    moved = ef != ff
    if not moved.any():
        return  # no product disagreed: the output is the exact one
    scaled = np.abs(exact_scaled_rowwise(x_cpu, ref)[moved]).astype(np.float64)
    rel = np.min(np.abs(scaled[:, None] - MIDPOINTS[None, :]) / MIDPOINTS[None, :], axis=1)
    assert rel.max() <= 2.0 ** -16, "a code moved %.3g away from every midpoint" % rel.max()


@pytest.mark.parametrize("mode", sorted(RHT))
def test_fast_rht_modes_bounded_by_exact(mode):
    dev = _cuda()
    cfg = RHT[mode]
    x_cpu = workloads.normal_with_outliers(1024, 2048, seed=29, fraction=0.002, gain=40.0)
    x = x_cpu.to(dev)
    ex, fa = run(x, **cfg), run(x, fast_math=True, **cfg)
    if "row_codes" in ex:
        for k in ("row_gscale", "row_scales"):
            assert np.array_equal(_bits(ex[k]), _bits(fa[k])), (mode, k)
        assert_codes_adjacent(ex["row_codes"], fa["row_codes"], mode + "/row")
    assert np.array_equal(_bits(ex["col_gscale"]), _bits(fa["col_gscale"])), mode
    ds = np.abs(ex["col_scales"].astype(int) - fa["col_scales"].astype(int))
    assert ds.max(initial=0) <= 1, (mode, "block scale moved", ds.max())
    if "sr" not in cfg.get("round_col", "rn"):
        assert_codes_adjacent(ex["col_codes"], fa["col_codes"], mode + "/col")
    diff = np.mean(ex["col_codes"] != fa["col_codes"])
    assert 0.0 < diff < 0.05, (mode, diff)  # the FP32 transform must change something
    db = sqnr_db(dequant(ex, "col"), dequant(fa, "col"))
    assert db >= SQNR_FLOOR_DB, (mode, db)


def test_fast_rht_activation_size_sqnr():
    """At the activation shape the pages measure (8192 x 4096, RHT + SR columnwise)."""
    dev = _cuda()
    cfg = RHT["rowcol_rht_sr"]
    x_cpu = workloads.normal_with_outliers(8192, 4096, seed=5, fraction=0.001, gain=100.0)
    x = x_cpu.to(dev)
    ex, fa = run(x, **cfg), run(x, fast_math=True, **cfg)
    db = sqnr_db(dequant(ex, "col"), dequant(fa, "col"))
    diff = np.mean(ex["col_codes"] != fa["col_codes"])
    assert db >= SQNR_FLOOR_DB and diff < 0.05, (db, diff)


@pytest.mark.parametrize("mode", ["2d_rowcol", "2d_row"])
def test_fast_math_leaves_2d_untouched(mode):
    dev = _cuda()
    cfg = dict(rowwise=True, columnwise=mode == "2d_rowcol", block2d=True)
    x = workloads.normal_with_outliers(512, 1792, seed=3, fraction=0.002, gain=40.0).to(dev)
    ex, fa = run(x, **cfg), run(x, fast_math=True, **cfg)
    for k in KEYS:
        if k in ex:
            assert np.array_equal(_bits(ex[k]), _bits(fa[k])), (mode, k)


@pytest.mark.parametrize("mode", ["rowcol_rn", "rowcol_rht_sr"])
def test_fast_fused_amax_matches_two_pass(mode):
    dev = _cuda()
    cfg = dict(PLAIN, **RHT)[mode]
    x = workloads.normal_with_outliers(640, 1040, seed=8, fraction=0.002, gain=40.0).to(dev)
    a = run(x, fast_math=True, **cfg)
    b = run(x, fast_math=True, fused_amax=True, **cfg)
    for k in KEYS:
        if k in a:
            assert np.array_equal(_bits(a[k]), _bits(b[k])), (mode, k)


@pytest.mark.parametrize("mode", ["rn", "rht_sr"])
def test_fast_grouped_bounded_by_exact(mode):
    dev = _cuda()
    cfg = {"rn": dict(rowwise=True, columnwise=True),
           "rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x6A5C,
                          round_col="sr", seed=5, offset=2)}[mode]
    T, H = 1500, 512
    offs_np = np.cumsum([16, 200, 0, 333, 48, 700, 203]).astype(np.int32)
    x = workloads.normal_with_outliers(T, H, seed=12, fraction=0.002, gain=40.0).to(dev)
    off = torch.from_numpy(offs_np).to(dev)
    cap = oracle.padded_capacity(offs_np)
    res = []
    for fast in (False, True):
        out = api.alloc_outputs(T, H, dev, True, True, col_ld=cap, groups=len(offs_np))
        for v in out.values():
            v.zero_()
        api.nvfp4_quantize_grouped(x, off, col_capacity=cap, out=out, fast_math=fast, **cfg)
        torch.cuda.synchronize()
        res.append(_np(out))
    ex, fa = res
    for k in ("row_gscale", "col_gscale", "row_scales"):
        assert np.array_equal(_bits(ex[k]), _bits(fa[k])), (mode, k)
    assert_codes_adjacent(ex["row_codes"], fa["row_codes"], mode + "/row")
    row_db = sqnr_db(dequant_grouped_rows(ex, offs_np), dequant_grouped_rows(fa, offs_np))
    col_db = sqnr_db(dequant_grouped_cols(ex, offs_np), dequant_grouped_cols(fa, offs_np))
    assert row_db >= SQNR_FLOOR_DB and col_db >= SQNR_FLOOR_DB, (mode, row_db, col_db)


def dequant_grouped_rows(o, offs):
    parts, start = [], 0
    for e, end in enumerate(offs):
        if end > start:
            parts.append(oracle.dequantize(o["row_codes"][start:end], o["row_scales"][start:end],
                                           o["row_gscale"][e, 1]))
        start = end
    return np.concatenate(parts, axis=0)


def dequant_grouped_cols(o, offs):
    """Each expert's columnwise block starts at a 16-aligned column of the padded output."""
    parts, start, col0 = [], 0, 0
    for e, end in enumerate(offs):
        n = int(end) - start
        pad = (n + 15) // 16 * 16
        if n > 0:
            parts.append(oracle.dequantize(o["col_codes"][:, col0 // 2:(col0 + pad) // 2],
                                           o["col_scales"][:, col0 // 16:(col0 + pad) // 16],
                                           o["col_gscale"][e, 1]))
        start, col0 = int(end), col0 + pad
    return np.concatenate(parts, axis=1)
