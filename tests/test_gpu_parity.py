"""Parity of the CUDA library (through its C ABI) with the oracle, element by element.

Codes, E4M3 scales and global scales must be bit-identical (the method is an encoding:
every float step is one IEEE binary32 operation on both sides, and the E2M1/E4M3 decisions are
taken in the same precision). Stochastic rounding is compared bit for bit too: both sides draw
the same Philox4x32-10 words for the same block positions.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import api, workloads

pytestmark = pytest.mark.gpu

KEYS = ("row_codes", "row_scales", "row_gscale", "col_codes", "col_scales", "col_gscale")


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def assert_same(gpu: dict, ref: dict, what=""):
    for k in KEYS:
        if k not in ref:
            continue
        g = gpu[k].cpu().numpy()
        r = ref[k]
        assert g.shape == r.shape, (what, k, g.shape, r.shape)
        gb, rb = _bits(g), _bits(r)
        if not np.array_equal(gb, rb):
            bad = np.argwhere(gb != rb)
            i = tuple(bad[0])
            raise AssertionError("%s %s: %d mismatches, first at %s: gpu=%s oracle=%s"
                                 % (what, k, len(bad), i, gb[i], rb[i]))


def run_both(x_cpu, **cfg):
    dev = _cuda()
    x = x_cpu.to(dev)
    out = api.nvfp4_quantize(x, **cfg)
    torch.cuda.synchronize()
    oc = oracle.Config(rowwise=cfg.get("rowwise", True), columnwise=cfg.get("columnwise", False),
                       block2d=cfg.get("block2d", False),
                       round_row_sr=cfg.get("round_row", "rn") == "sr",
                       round_col_sr=cfg.get("round_col", "rn") == "sr",
                       rht_col=cfg.get("rht_col", False), sign_mask=cfg.get("sign_mask", 0),
                       seed=cfg.get("seed", 0), offset=cfg.get("offset", 0))
    ref = oracle.quantize(x_cpu, oc)
    return out, ref


MODES = {
    "row_rn": dict(rowwise=True),
    "row_sr": dict(rowwise=True, round_row="sr", seed=11, offset=3),
    "col_rn": dict(rowwise=False, columnwise=True),
    "col_sr": dict(rowwise=False, columnwise=True, round_col="sr", seed=12),
    "col_rht": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0xB3C5),
    "col_rht_sr": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0x0F0F,
                       round_col="sr", seed=2**40 + 5, offset=9),
    "rowcol_rn": dict(rowwise=True, columnwise=True),
    "rowcol_sr": dict(rowwise=True, columnwise=True, round_row="sr", round_col="sr", seed=77),
    "rowcol_rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1234,
                          round_col="sr", seed=4),
    "2d_rowcol": dict(rowwise=True, columnwise=True, block2d=True),
    "2d_row": dict(rowwise=True, block2d=True),
    "2d_col": dict(rowwise=False, columnwise=True, block2d=True),
}

# several tiles (64 x 256) and ragged tails in both directions
SHAPES = [(16, 16), (16, 32), (64, 256), (80, 272), (144, 528), (320, 1040), (256, 512)]


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
def test_modes_and_shapes_match_oracle(mode, shape):
    M, N = shape
    x = workloads.normal(M, N, 1.0, seed=M * 7919 + N)
    out, ref = run_both(x, **MODES[mode])
    assert_same(out, ref, "%s %s" % (mode, shape))


def test_rowwise_any_row_count():
    x = workloads.normal(77, 64, 1.0, seed=5)  # M not a multiple of 16 is fine rowwise
    out, ref = run_both(x, rowwise=True, round_row="sr", seed=1)
    assert_same(out, ref)


@pytest.mark.parametrize("mode", ["rowcol_rn", "rowcol_rht_sr", "2d_rowcol"])
def test_special_values(mode):
    M, N = 64, 256
    rng = np.random.Generator(np.random.PCG64(99))
    cases = {
        "zeros": np.zeros((M, N), np.float32),
        "signed_zeros": np.where(rng.random((M, N)) < 0.5, -0.0, 0.0).astype(np.float32),
        "subnormal_only": (rng.integers(1, 128, (M, N)) * 2.0 ** -133 *
                           rng.choice([-1, 1], (M, N))).astype(np.float32),
        "saturating_outliers": np.where(rng.random((M, N)) < 0.01, 3.0e38,
                                        rng.standard_normal((M, N))).astype(np.float32),
        "tiny_and_huge": np.where(rng.random((M, N)) < 0.5, 1e-30, 1e30).astype(np.float32),
        "grid_exact": (rng.choice([0, 0.5, 1, 1.5, 2, 3, 4, 6], (M, N)) *
                       rng.choice([-1, 1], (M, N))).astype(np.float32),
    }
    for name, v in cases.items():
        x = workloads.to_bf16(v)
        out, ref = run_both(x, **MODES[mode])
        assert_same(out, ref, "%s/%s" % (mode, name))


def test_random_bit_patterns_every_exponent():
    bits = workloads.random_bf16_bits((128, 512), seed=3)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    for mode in ("rowcol_rn", "rowcol_rht_sr", "2d_rowcol"):
        out, ref = run_both(x, **MODES[mode])
        assert_same(out, ref, mode)


def test_every_bf16_block_maximum_with_supplied_amax():
    """All finite BF16 magnitudes as the maxima of 1x16 blocks, quantized under a sweep of
    supplied global amax values: covers the block-scale arithmetic (x/6, E4M3, reciprocal)
    for every possible block maximum."""
    dev = _cuda()
    mags = np.arange(1, 0x7F80, dtype=np.uint32)
    f = (mags << 16).view(np.float32)
    rng = np.random.Generator(np.random.PCG64(8))
    blocks = f[:, None] * rng.uniform(-1, 1, (f.size, 16)).astype(np.float32)
    blocks[:, 5] = f
    rows = (f.size // 16) * 16
    x_cpu = workloads.to_bf16(blocks[:rows])
    xb = oracle.as_bf16_bits(x_cpu)
    x = x_cpu.to(dev)
    for k in range(-136, 127, 6):
        amax = np.float32(2.0 ** k * 1.37)
        a = torch.tensor([amax], dtype=torch.float32, device=dev)
        out = api.nvfp4_quantize(x, rowwise=True, amax_row=a)
        rc, rs, gs = oracle.quantize_rowwise(xb, amax_value=amax)
        assert_same(out, {"row_codes": rc, "row_scales": rs, "row_gscale": gs}, "amax 2^%d" % k)


def test_supplied_amax_columnwise_and_rht():
    dev = _cuda()
    x_cpu = workloads.laplace(128, 512, 1e-3, seed=21)
    xb = oracle.as_bf16_bits(x_cpu)
    x = x_cpu.to(dev)
    a_row = np.float32(0.01)
    a_col = np.float32(0.02)
    out = api.nvfp4_quantize(x, rowwise=True, columnwise=True, rht_col=True, sign_mask=0x5555,
                             round_col="sr", seed=3,
                             amax_row=torch.tensor([a_row], device=dev),
                             amax_col=torch.tensor([a_col], device=dev))
    rc, rs, rg = oracle.quantize_rowwise(xb, amax_value=a_row)
    cc, cs, cg = oracle.quantize_colwise(xb, amax_value=a_col, rht=True, sign_mask=0x5555, sr=True,
                                         seed=3)
    assert_same(out, dict(row_codes=rc, row_scales=rs, row_gscale=rg, col_codes=cc,
                          col_scales=cs, col_gscale=cg))


def test_amax_entry_point():
    dev = _cuda()
    x_cpu = workloads.normal_with_outliers(256, 1024, seed=31)
    xb = oracle.as_bf16_bits(x_cpu)
    a_row, a_col = api.nvfp4_amax(x_cpu.to(dev), rht_col=True, sign_mask=0x8001)
    assert a_row.item() == oracle.amax(xb)
    assert a_col.item() == oracle.amax_rht(xb, 0x8001)
    a_row, a_col = api.nvfp4_amax(x_cpu.to(dev))
    assert a_row.item() == a_col.item() == oracle.amax(xb)


def test_empty_tensors():
    dev = _cuda()
    for M, N in [(0, 32), (32, 0), (0, 0)]:
        x = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        out = api.nvfp4_quantize(x, rowwise=True, columnwise=True)
        torch.cuda.synchronize()
        assert out["row_gscale"].tolist() == [0.0, 1.0]
        assert out["col_gscale"].tolist() == [0.0, 1.0]


def test_dequantize_matches_oracle():
    dev = _cuda()
    x_cpu = workloads.normal(192, 320, 2.0, seed=41)
    out = api.nvfp4_quantize(x_cpu.to(dev), rowwise=True, columnwise=True, rht_col=True,
                             sign_mask=7)
    for side in ("row", "col"):
        d = api.nvfp4_dequantize(out[side + "_codes"], out[side + "_scales"],
                                 out[side + "_gscale"]).cpu().numpy()
        r = oracle.dequantize(out[side + "_codes"].cpu().numpy(),
                              out[side + "_scales"].cpu().numpy(),
                              out[side + "_gscale"].cpu().numpy()[1])
        np.testing.assert_array_equal(d.view(np.uint32), r.view(np.uint32))


# ------------------------------------------------------------------------------------------
# Stochastic rounding properties on the GPU ([PR4798] "Correctness")
# ------------------------------------------------------------------------------------------

def test_sr_seed_offset_reproducibility_and_step_bound():
    dev = _cuda()
    x = workloads.normal(128, 512, 1.0, seed=51).to(dev)
    kw = dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1111, round_row="sr",
              round_col="sr")
    a = api.nvfp4_quantize(x, seed=9, offset=0, **kw)
    b = api.nvfp4_quantize(x, seed=9, offset=0, **kw)
    c = api.nvfp4_quantize(x, seed=9, offset=1, **kw)
    n = api.nvfp4_quantize(x, rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1111)
    for k in ("row_codes", "col_codes"):
        assert torch.equal(a[k], b[k])
        assert (a[k] != c[k]).sum().item() > 1000
        sr = a[k].cpu().numpy()
        rn = n[k].cpu().numpy()
        for sh in (0, 4):
            qs = (sr >> sh) & 0xF
            qr = (rn >> sh) & 0xF
            zero = (qs & 7) == 0
            same_sign = ((qs & 8) == (qr & 8)) | zero | ((qr & 7) == 0)
            assert same_sign.all()
            assert (np.abs((qs & 7).astype(int) - (qr & 7).astype(int)) <= 1).all()


# ------------------------------------------------------------------------------------------
# Grouped
# ------------------------------------------------------------------------------------------

def run_grouped_both(x_cpu, offsets_np, cap=None, **cfg):
    dev = _cuda()
    off = torch.from_numpy(np.asarray(offsets_np, dtype=np.int32)).to(dev)
    if cap is None:
        cap = oracle.padded_capacity(offsets_np)
    rowwise = cfg.get("rowwise", True)
    columnwise = cfg.get("columnwise", True)
    T, H = x_cpu.shape
    E = len(offsets_np)
    out = api.alloc_outputs(T, H, dev, rowwise, columnwise, col_ld=cap, groups=E)
    for k in ("row_codes", "row_scales", "col_codes", "col_scales"):
        if k in out:
            out[k].fill_(0xEE)  # poison: untouched regions must keep it
    api.nvfp4_quantize_grouped(x_cpu.to(dev), off, col_capacity=cap, out=out, **cfg)
    torch.cuda.synchronize()
    rc, rs, rg, cc, cs, cg = oracle.quantize_grouped(
        x_cpu, offsets_np, cap=cap, rowwise=rowwise, columnwise=columnwise,
        round_row_sr=cfg.get("round_row") == "sr", round_col_sr=cfg.get("round_col") == "sr",
        rht_col=cfg.get("rht_col", False), sign_mask=cfg.get("sign_mask", 0),
        seed=cfg.get("seed", 0), offset=cfg.get("offset", 0), fill=0xEE,
        block2d=cfg.get("block2d", False))
    ref = {}
    if rowwise:
        ref.update(row_codes=rc, row_scales=rs, row_gscale=rg)
    if columnwise:
        ref.update(col_codes=cc, col_scales=cs, col_gscale=cg)
    return out, ref


GROUPED_CASES = [
    ("one_expert", 100, 64, [100]),
    ("odd_counts", 203, 272, [5, 5, 37, 37, 70, 150, 203]),
    ("zero_experts_and_tail", 300, 64, [0, 0, 17, 17, 129, 250]),
    ("many_small", 260, 32, list(np.cumsum([1, 2, 3, 15, 16, 17, 31, 33, 0, 64, 65, 13]))),
    # column starts 16, 48, 96: segments that begin inside a 64-row tile of the columnwise
    # space (tiles shared by two or three segments), then experts long enough for whole tiles
    ("lead_slabs", 700, 512, list(np.cumsum([16, 200, 32, 150, 48, 200, 1, 53]))),
]


@pytest.mark.parametrize("case", GROUPED_CASES, ids=lambda c: c[0])
@pytest.mark.parametrize("mode", ["2d_rowcol", "2d_row", "2d_col"])
def test_grouped_2d_matches_oracle(case, mode):
    """Stacked expert weights with 16x16 tiles per expert (ragged experts zero-padded)."""
    name, T, H, offs = case
    cfg = {"2d_rowcol": dict(rowwise=True, columnwise=True),
           "2d_row": dict(rowwise=True, columnwise=False),
           "2d_col": dict(rowwise=False, columnwise=True)}[mode]
    x = workloads.normal_with_outliers(T, H, seed=T * 5 + H, fraction=0.01, gain=30.0)
    out, ref = run_grouped_both(x, offs, block2d=True, **cfg)
    assert_same(out, ref, "%s/%s" % (name, mode))


def test_grouped_2d_weights_of_the_pages_shape():
    """E = 4 experts' stacked weights (DeepSeek-V3 gate/up-like rows of 7168), 16x16 tiles."""
    E, rows, H = 4, 512, 7168
    offs = list(np.cumsum([rows] * E))
    x = workloads.normal(E * rows, H, 0.02, seed=71)
    out, ref = run_grouped_both(x, offs, block2d=True, rowwise=True, columnwise=True)
    assert_same(out, ref, "grouped 2D weights")


@pytest.mark.parametrize("case", GROUPED_CASES, ids=lambda c: c[0])
@pytest.mark.parametrize("mode", ["rn", "rht_sr", "row_only_sr", "col_only_rht"])
def test_grouped_matches_oracle(case, mode):
    name, T, H, offs = case
    cfg = {
        "rn": dict(rowwise=True, columnwise=True),
        "rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x6A5C,
                       round_col="sr", seed=5, offset=2),
        "row_only_sr": dict(rowwise=True, columnwise=False, round_row="sr", seed=8),
        "col_only_rht": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0xFFFF),
    }[mode]
    x = workloads.normal(T, H, 1.0, seed=T + H)
    out, ref = run_grouped_both(x, offs, **cfg)
    assert_same(out, ref, "%s/%s" % (name, mode))


@pytest.mark.parametrize("mode", ["rn", "rht_sr", "row_only_sr", "col_only_rht", "2d_rowcol"])
def test_grouped_many_tiles_per_cta_matches_oracle(mode):
    """Enough tiles that every CTA refills each stage of its ring several times (about ten
    tiles per CTA), with 40 experts of seeded random sizes (empty and tiny ones included), so
    that tiles shared by segments, the per-warp loads of the refills and the amax pass's
    refills all run; the per-expert maxima are computed inside the call."""
    rng = np.random.default_rng(0x5EED_0040)
    counts = rng.integers(0, 300, size=40)
    counts[[3, 17, 18]] = 0
    counts[[5, 9]] = [1, 15]
    offs = list(np.cumsum(counts))
    T, H = int(offs[-1]), 4096
    cfg = {
        "rn": dict(rowwise=True, columnwise=True),
        "rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x3A5C,
                       round_col="sr", seed=11, offset=3),
        "row_only_sr": dict(rowwise=True, columnwise=False, round_row="sr", seed=12),
        "col_only_rht": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0x8001),
        "2d_rowcol": dict(rowwise=True, columnwise=True, block2d=True),
    }[mode]
    x = workloads.normal_with_outliers(T, H, seed=T + 7, fraction=0.002, gain=40.0)
    out, ref = run_grouped_both(x, offs, **cfg)
    assert_same(out, ref, "many tiles/%s" % mode)


@pytest.mark.parametrize("mode", ["rht_sr", "row_only_sr", "2d_rowcol"])
def test_grouped_most_experts_matches_oracle(mode):
    """The largest expert count (256), most experts tiny or empty: tiles shared by up to four
    experts, deep segment searches, the per-warp tables of slabs in other experts."""
    rng = np.random.default_rng(0x5EED_0100)
    counts = rng.integers(0, 40, size=256)
    counts[rng.random(256) < 0.25] = 0
    counts[-1] = 0                      # trailing empty experts
    offs = list(np.cumsum(counts))
    T, H = int(offs[-1]) + 9, 512       # a tail past the last expert
    cfg = {
        "rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x9E37,
                       round_col="sr", seed=31, offset=5),
        "row_only_sr": dict(rowwise=True, columnwise=False, round_row="sr", seed=32),
        "2d_rowcol": dict(rowwise=True, columnwise=True, block2d=True),
    }[mode]
    x = workloads.normal_with_outliers(T, H, seed=T + 11, fraction=0.01, gain=30.0)
    out, ref = run_grouped_both(x, offs, **cfg)
    assert_same(out, ref, "256 experts/%s" % mode)


@pytest.mark.parametrize("case", GROUPED_CASES[1:3], ids=lambda c: c[0])
@pytest.mark.parametrize("mode", ["rn", "rht_sr", "col_only_rht", "2d_rowcol", "2d_col"])
def test_grouped_with_supplied_amax_matches_oracle(case, mode):
    """Per-expert maxima from nvfp4_amax_grouped passed in (no amax pass inside the call):
    every output equals the oracle's, as with the maxima computed inside."""
    name, T, H, offs = case
    cfg = {
        "rn": dict(rowwise=True, columnwise=True),
        "rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x6A5C,
                       round_col="sr", seed=5, offset=2),
        "col_only_rht": dict(rowwise=False, columnwise=True, rht_col=True, sign_mask=0xFFFF),
        "2d_rowcol": dict(rowwise=True, columnwise=True, block2d=True),
        "2d_col": dict(rowwise=False, columnwise=True, block2d=True),
    }[mode]
    dev = _cuda()
    x = workloads.normal_with_outliers(T, H, seed=T * 3 + H, fraction=0.01, gain=30.0)
    off = torch.from_numpy(np.asarray(offs, dtype=np.int32)).to(dev)
    xd = x.to(dev)
    a_row, a_col = api.nvfp4_amax_grouped(xd, off, rht_col=cfg.get("rht_col", False),
                                          sign_mask=cfg.get("sign_mask", 0))
    cap = oracle.padded_capacity(offs)
    _, ref = run_grouped_both(x, offs, **cfg)
    out = api.nvfp4_quantize_grouped(xd, off, col_capacity=cap, amax_row=a_row,
                                     amax_col=None if cfg.get("block2d") else a_col, **cfg)
    torch.cuda.synchronize()
    # regions the call does not write hold whatever the allocation held: compare written parts
    rows = int(offs[-1])
    for k in list(ref):
        if k.startswith("row_") and k != "row_gscale":
            ref[k] = ref[k][:rows]
            out[k] = out[k][:rows]
        if k.startswith("col_") and k != "col_gscale":
            w = cap // 2 if k == "col_codes" else cap // 16
            ref[k] = ref[k][:, :w]
            out[k] = out[k][:, :w]
    assert_same(out, ref, "%s/%s with supplied maxima" % (name, mode))


def test_grouped_extra_capacity_left_untouched():
    x = workloads.normal(100, 48, 1.0, seed=61)
    offs = [30, 30, 64, 99]
    cap = oracle.padded_capacity(offs) + 48
    out, ref = run_grouped_both(x, offs, cap=cap, rht_col=True, sign_mask=3)
    assert_same(out, ref)


def test_grouped_bad_offsets_set_device_status():
    dev = _cuda()
    x = workloads.normal(64, 32, 1.0, seed=62).to(dev)
    api.nvfp4_get_status()  # clear
    for bad in ([40, 20], [10, 65], [-1, 10]):
        off = torch.tensor(bad, dtype=torch.int32, device=dev)
        out = api.nvfp4_quantize_grouped(x, off, col_capacity=128, rht_col=True)
        status, bits = api.nvfp4_get_status()
        assert bits & 1, bad
        assert status == 6
    # capacity too small for the padded token total
    off = torch.tensor([20, 40], dtype=torch.int32, device=dev)
    api.nvfp4_quantize_grouped(x, off, col_capacity=32)
    status, bits = api.nvfp4_get_status()
    assert bits & 1
    status, bits = api.nvfp4_get_status()
    assert status == 0 and bits == 0


# ------------------------------------------------------------------------------------------
# The workloads at full size, in the launch configuration the benchmark times
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_full_size_workload_matches_oracle(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_input(w)
    x = inp["x"]
    if w.grouped:
        cfg = dict(rowwise=w.rowwise, columnwise=w.columnwise, rht_col=w.rht_col,
                   sign_mask=inp["sign_mask"], round_col="sr" if w.round_col_sr else "rn",
                   round_row="sr" if w.round_row_sr else "rn", seed=inp["seed"],
                   block2d=w.block2d)
        out, ref = run_grouped_both(x, inp["offsets"], **cfg)
    else:
        cfg = dict(rowwise=w.rowwise, columnwise=w.columnwise, block2d=w.block2d,
                   rht_col=w.rht_col, sign_mask=inp["sign_mask"],
                   round_col="sr" if w.round_col_sr else "rn",
                   round_row="sr" if w.round_row_sr else "rn", seed=inp["seed"])
        out, ref = run_both(x, **cfg)
    assert_same(out, ref, name)


# ------------------------------------------------------------------------------------------
# Single-launch amax (fused_amax): same outputs as the two-pass pipeline and the oracle
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("shape", [(16, 16), (80, 272), (320, 1040)], ids=lambda s: "%dx%d" % s)
def test_fused_amax_matches_oracle(mode, shape):
    M, N = shape
    x = workloads.normal_with_outliers(M, N, seed=M * 31 + N, fraction=0.01, gain=50.0)
    out, ref = run_both(x, fused_amax=True, **MODES[mode])
    assert_same(out, ref, "fused %s %s" % (mode, shape))


def test_fused_amax_repeated_calls_reuse_the_barrier():
    """The arrival count and the epoch-tagged maxima need no clearing: many fused launches in a
    row stay correct."""
    dev = _cuda()
    for k in range(6):
        x_cpu = workloads.laplace(64 * (k + 1), 512, 1e-2 * (k + 1), seed=70 + k)
        x = x_cpu.to(dev)
        out = api.nvfp4_quantize(x, rowwise=True, columnwise=True, rht_col=True, sign_mask=0x0FF0,
                                 round_col="sr", seed=k, fused_amax=True)
        ref = oracle.quantize(x_cpu, oracle.Config(rowwise=True, columnwise=True, rht_col=True,
                                                   sign_mask=0x0FF0, round_col_sr=True, seed=k))
        torch.cuda.synchronize()
        assert_same(out, ref, "repeat %d" % k)
    status, bits = api.nvfp4_get_status()
    assert status == 0 and bits == 0


# Single launch, rowwise + columnwise RTNE on shapes that mix whole 64 x 256 tiles with ragged
# row and column tiles, N a multiple of 64 or not.
FUSED_ROWCOL_SHAPES = [(64, 256), (128, 512), (304, 1088), (576, 2304), (1024, 4096), (320, 1040)]


@pytest.mark.parametrize("shape", FUSED_ROWCOL_SHAPES, ids=lambda s: "%dx%d" % s)
def test_fused_rowcol_whole_and_ragged_tiles_match_oracle(shape):
    M, N = shape
    # a second call on other data into reused memory
    for k, gain in enumerate((40.0, 3.0)):
        x = workloads.normal_with_outliers(M, N, seed=M + N + k, fraction=0.01, gain=gain)
        out, ref = run_both(x, rowwise=True, columnwise=True, fused_amax=True)
        assert_same(out, ref, "fused rowcol %s call %d" % (shape, k))


def test_fused_rowcol_special_tiles():
    # whole tiles that are all zero, all negative, or hold one large negative value
    M, N = 192, 768
    x = workloads.normal_with_outliers(M, N, seed=5, fraction=0.01, gain=20.0).float()
    x[0:64, 0:256] = 0.0
    x[64:128, 256:512] = -x[64:128, 256:512].abs() - 1e-3
    x[128:192, 512:768] = 0.0
    x[150, 600] = -3.0e4
    out, ref = run_both(x.to(torch.bfloat16), rowwise=True, columnwise=True, fused_amax=True)
    assert_same(out, ref, "fused rowcol special tiles")


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items() if not w.grouped])
def test_full_size_workload_fused_matches_oracle(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_input(w)
    cfg = dict(rowwise=w.rowwise, columnwise=w.columnwise, block2d=w.block2d, rht_col=w.rht_col,
               sign_mask=inp["sign_mask"], round_col="sr" if w.round_col_sr else "rn",
               round_row="sr" if w.round_row_sr else "rn", seed=inp["seed"], fused_amax=True)
    out, ref = run_both(inp["x"], **cfg)
    assert_same(out, ref, "fused " + name)


def test_caller_workspace_serves_the_fused_path_and_status():
    """nvfp4_set_workspace: the single-launch amax and the status word on caller memory, then
    back on the library's own; outputs equal the oracle's either way."""
    dev = _cuda()
    ws = torch.empty(api.WORKSPACE_BYTES // 4 + 64, dtype=torch.int32, device=dev)
    try:
        api.nvfp4_set_workspace(ws)
        for seed in (1, 2):
            x = workloads.normal_with_outliers(320, 1040, seed=seed, fraction=0.01, gain=30.0)
            out, ref = run_both(x, rowwise=True, columnwise=True, fused_amax=True)
            assert_same(out, ref, "caller workspace %d" % seed)
        assert api.nvfp4_get_status(dev) == (0, 0)
    finally:
        api.nvfp4_set_workspace(None)
        torch.cuda.synchronize()
    x = workloads.normal_with_outliers(320, 1040, seed=3, fraction=0.01, gain=30.0)
    out, ref = run_both(x, rowwise=True, columnwise=True, fused_amax=True)
    assert_same(out, ref, "own workspace again")


@pytest.mark.parametrize("case", GROUPED_CASES, ids=lambda c: c[0])
@pytest.mark.parametrize("rht", [False, True])
def test_amax_grouped_matches_oracle(case, rht):
    dev = _cuda()
    name, T, H, offs = case
    x = workloads.normal_with_outliers(T, H, seed=T + 3 * H, fraction=0.01, gain=30.0)
    mask = 0x3C5A
    a_row, a_col = api.nvfp4_amax_grouped(x.to(dev), torch.from_numpy(np.asarray(offs, np.int32)).to(dev),
                                          rht_col=rht, sign_mask=mask)
    torch.cuda.synchronize()
    _, _, rg, _, _, cg = oracle.quantize_grouped(x, offs, rht_col=rht, sign_mask=mask)
    assert np.array_equal(_bits(a_row.cpu().numpy()), _bits(rg[:, 0].copy())), name
    assert np.array_equal(_bits(a_col.cpu().numpy()), _bits(cg[:, 0].copy())), name
