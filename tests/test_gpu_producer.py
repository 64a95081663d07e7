"""The RMSNorm producer with the amax in its epilogue (nvfp4_rmsnorm_amax) and the
norm-then-quantize call built on it (nvfp4_rmsnorm_quantize), against the oracle bit for bit:
y, its amax, and every quantize output (the oracle quantizes its own y with its own amax)."""
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


def _weight(N, seed):
    rng = np.random.default_rng(seed)
    return torch.tensor(rng.normal(1.0, 0.3, N).astype(np.float32)).to(torch.bfloat16)


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("shape", [(1, 8), (5, 264), (64, 4096), (300, 1040), (8192, 4096)],
                         ids=lambda s: "%dx%d" % s)
@pytest.mark.parametrize("eps,bias", [(1e-6, 0.0), (1e-5, 1.0), (0.0, -0.25)])
def test_rmsnorm_amax_matches_oracle(shape, eps, bias):
    dev = _cuda()
    M, N = shape
    x = workloads.normal_with_outliers(M, N, seed=M * 3 + N, fraction=0.01, gain=30.0)
    w = _weight(N, seed=N)
    y, amax = api.nvfp4_rmsnorm_amax(x.to(dev), w.to(dev), eps=eps, weight_bias=bias)
    torch.cuda.synchronize()
    y_ref, amax_ref = oracle.rmsnorm(x, w, eps=eps, bias=bias)
    got = y.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, y_ref), int((got != y_ref).sum())
    assert amax.item() == float(amax_ref)


MODES = {
    "rowcol_rn": dict(rowwise=True, columnwise=True),
    "rowcol_rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x1234,
                          round_col="sr", seed=4),
    "2d_rowcol": dict(rowwise=True, columnwise=True, block2d=True),
    "row_sr": dict(rowwise=True, round_row="sr", seed=9, offset=2),
}


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("shape", [(320, 1040), (8192, 4096)], ids=lambda s: "%dx%d" % s)
def test_rmsnorm_quantize_matches_oracle(mode, shape):
    dev = _cuda()
    M, N = shape
    cfg = MODES[mode]
    x = workloads.normal_with_outliers(M, N, seed=11 + M, fraction=0.01, gain=30.0)
    w = _weight(N, seed=5)
    out = api.nvfp4_rmsnorm_quantize(x.to(dev), w.to(dev), eps=1e-6, weight_bias=0.0, **cfg)
    torch.cuda.synchronize()
    y_ref, _ = oracle.rmsnorm(x, w, eps=1e-6, bias=0.0)
    oc = oracle.Config(rowwise=cfg.get("rowwise", True), columnwise=cfg.get("columnwise", False),
                       block2d=cfg.get("block2d", False),
                       round_row_sr=cfg.get("round_row", "rn") == "sr",
                       round_col_sr=cfg.get("round_col", "rn") == "sr",
                       rht_col=cfg.get("rht_col", False), sign_mask=cfg.get("sign_mask", 0),
                       seed=cfg.get("seed", 0), offset=cfg.get("offset", 0))
    ref = oracle.quantize(y_ref, oc)
    assert np.array_equal(out["y"].cpu().view(torch.int16).numpy().view(np.uint16), y_ref)
    for k in KEYS:
        if k in ref:
            g, r = _bits(out[k].cpu().numpy()), _bits(ref[k])
            assert g.shape == r.shape and np.array_equal(g, r), (mode, k, int((g != r).sum()))
