"""Seeded random sweep of shapes, modes and options against the oracle, bit for bit: plain
tensors (every orientation, 2D, RHT, SR, single-launch amax), grouped tensors with random expert
counts (1D and 2D) and MX formats. Shapes are drawn to hit ragged tile edges in both directions;
the seed of each case is in its id, so a failure reproduces alone."""
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


def _same(got, ref, what):
    for k in KEYS:
        if k in ref:
            g, r = _bits(got[k].cpu().numpy()), _bits(ref[k])
            assert g.shape == r.shape, (what, k, g.shape, r.shape)
            assert np.array_equal(g, r), (what, k, int((g != r).sum()))


def _plain_case(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 40)) * 16
    N = int(rng.integers(1, 80)) * 16
    kind = rng.choice(["row", "col", "rowcol", "2d"])
    cfg = dict(rowwise=kind in ("row", "rowcol", "2d"),
               columnwise=kind in ("col", "rowcol") or (kind == "2d" and bool(rng.integers(2))))
    if kind == "2d":
        cfg["block2d"] = True
    else:
        if cfg["columnwise"] and rng.integers(2):
            cfg.update(rht_col=True, sign_mask=int(rng.integers(0, 1 << 16)))
        if cfg["rowwise"] and rng.integers(2):
            cfg["round_row"] = "sr"
        if cfg["columnwise"] and rng.integers(2):
            cfg["round_col"] = "sr"
        cfg.update(seed=int(rng.integers(0, 2 ** 62)), offset=int(rng.integers(0, 1000)))
    cfg["fused_amax"] = bool(rng.integers(2))
    return M, N, cfg


@pytest.mark.parametrize("seed", range(1000, 1040), ids=lambda s: "seed%d" % s)
def test_random_plain_cases(seed):
    dev = _cuda()
    M, N, cfg = _plain_case(seed)
    x = workloads.normal_with_outliers(M, N, seed=seed, fraction=0.01, gain=50.0)
    out = api.nvfp4_quantize(x.to(dev), **cfg)
    torch.cuda.synchronize()
    oc = oracle.Config(rowwise=cfg["rowwise"], columnwise=cfg["columnwise"],
                       block2d=cfg.get("block2d", False),
                       round_row_sr=cfg.get("round_row") == "sr",
                       round_col_sr=cfg.get("round_col") == "sr",
                       rht_col=cfg.get("rht_col", False), sign_mask=cfg.get("sign_mask", 0),
                       seed=cfg.get("seed", 0), offset=cfg.get("offset", 0))
    _same(out, oracle.quantize(x, oc), "seed %d %dx%d %s" % (seed, M, N, cfg))


@pytest.mark.parametrize("seed", range(2000, 2020), ids=lambda s: "seed%d" % s)
def test_random_grouped_cases(seed):
    dev = _cuda()
    rng = np.random.default_rng(seed)
    H = int(rng.integers(1, 40)) * 16
    E = int(rng.integers(1, 20))
    counts = rng.integers(0, 90, size=E)
    counts[rng.random(E) < 0.2] = 0                     # some empty experts
    offs = np.cumsum(counts).astype(np.int32)
    T = int(offs[-1]) + int(rng.integers(0, 40))        # a tail past the last expert
    if T == 0:
        T = 16
    two_d = bool(rng.integers(2))
    cfg = dict(rowwise=bool(rng.integers(2)) or two_d, columnwise=True)
    if two_d:
        cfg["block2d"] = True
    else:
        if rng.integers(2):
            cfg.update(rht_col=True, sign_mask=int(rng.integers(0, 1 << 16)))
        if rng.integers(2):
            cfg["round_col"] = "sr"
        if cfg["rowwise"] and rng.integers(2):
            cfg["round_row"] = "sr"
        cfg.update(seed=int(rng.integers(0, 2 ** 62)), offset=int(rng.integers(0, 1000)))
    x = workloads.normal_with_outliers(T, H, seed=seed, fraction=0.01, gain=50.0)
    cap = oracle.padded_capacity(offs) + 16 * int(rng.integers(0, 3))
    out = api.alloc_outputs(T, H, dev, cfg["rowwise"], True, col_ld=cap, groups=E)
    for k in ("row_codes", "row_scales", "col_codes", "col_scales"):
        if k in out:
            out[k].fill_(0xEE)
    api.nvfp4_quantize_grouped(x.to(dev), torch.from_numpy(offs).to(dev), col_capacity=cap,
                               out=out, **cfg)
    torch.cuda.synchronize()
    rc, rs, rg, cc, cs, cg = oracle.quantize_grouped(
        x, offs, cap=cap, rowwise=cfg["rowwise"], columnwise=True,
        round_row_sr=cfg.get("round_row") == "sr", round_col_sr=cfg.get("round_col") == "sr",
        rht_col=cfg.get("rht_col", False), sign_mask=cfg.get("sign_mask", 0),
        seed=cfg.get("seed", 0), offset=cfg.get("offset", 0), fill=0xEE,
        block2d=cfg.get("block2d", False))
    ref = dict(col_codes=cc, col_scales=cs, col_gscale=cg)
    if cfg["rowwise"]:
        ref.update(row_codes=rc, row_scales=rs, row_gscale=rg)
    _same(out, ref, "seed %d T=%d H=%d offs=%s %s" % (seed, T, H, offs.tolist(), cfg))


@pytest.mark.parametrize("seed", range(3000, 3024), ids=lambda s: "seed%d" % s)
def test_random_mx_cases(seed):
    dev = _cuda()
    rng = np.random.default_rng(seed)
    fmt = str(rng.choice(["e4m3", "e5m2", "e2m1"]))
    kind = rng.choice(["row", "col", "rowcol"])
    row, col = kind in ("row", "rowcol"), kind in ("col", "rowcol")
    M = int(rng.integers(1, 30)) * 32 if col else int(rng.integers(1, 700))
    N = int(rng.integers(1, 60)) * 32 if row else int(rng.integers(1, 240)) * 8
    x = workloads.normal_with_outliers(M, N, seed=seed, fraction=0.01, gain=80.0)
    out = api.nvfp4_mx_quantize(x.to(dev), fmt, row, col)
    torch.cuda.synchronize()
    if row:
        c, s = oracle.mx_quantize_rowwise(x, fmt)
        assert np.array_equal(out["row_codes"].cpu().numpy(), c), (seed, fmt, M, N)
        assert np.array_equal(out["row_scales"].cpu().numpy(), s), (seed, fmt, M, N)
    if col:
        c, s = oracle.mx_quantize_colwise(x, fmt)
        assert np.array_equal(out["col_codes"].cpu().numpy(), c), (seed, fmt, M, N)
        assert np.array_equal(out["col_scales"].cpu().numpy(), s), (seed, fmt, M, N)
