"""nvfp4_quantize_noalloc: the entry point for callers that cannot allocate device memory
(code inside an allocator's callbacks, latency-critical paths that must never reach cudaMalloc,
hosts with a fixed memory budget). Its scratch lives in a static device array instead of the
library's lazily allocated workspace.

Called directly through the C ABI (ctypes) and compared with the regular nvfp4_quantize on the
same input, bit for bit (the tolerance of every parity test here), twice in a row so that the
second call runs on the scratch the first one left behind. Kept in a file of its own that
pytest collects last; it passes alone in a fresh process and after the other tests.

A call whose bounded wait gives up (forced with the test hook that makes the wait expect one
share more than exists) must be visible through nvfp4_noalloc_get_status, which reads the
array's own status word without allocating; the next call must be correct again. A call whose
last CTAs are held back (another test hook) has their shares taken over and is still correct.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quantize_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

KEYS = ("row_codes", "row_scales", "row_gscale", "col_codes", "col_scales", "col_gscale")


def _noalloc(x, out, cfg):
    L = _lib.load()
    M, N = x.shape
    p = lambda k: ctypes.c_void_p(out[k].data_ptr()) if k in out else None
    stream = ctypes.c_void_p(torch.cuda.current_stream(x.device).cuda_stream)
    return L.nvfp4_quantize_noalloc(ctypes.c_void_p(x.data_ptr()), M, N, ctypes.byref(cfg),
                                    p("row_codes"), p("row_scales"), p("row_gscale"),
                                    p("col_codes"), p("col_scales"), p("col_gscale"), stream)


CASES = [
    ("row_col_rtne", (8192, 4096), dict(rowwise=True, columnwise=True)),
    ("row_rtne_col_rht_sr", (1024, 2048), dict(rowwise=True, columnwise=True, rht_col=True,
                                               sign_mask=0x5A3C, round_col="sr", seed=9)),
    ("weight_2d", (512, 1792), dict(rowwise=True, columnwise=True, block2d=True)),
    ("ragged_row_sr", (80, 272), dict(rowwise=True, round_row="sr", seed=3)),
    ("row_col_rht_fast_math", (1024, 2048), dict(rowwise=True, columnwise=True, rht_col=True,
                                                  sign_mask=0x3C5A, fast_math=True)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_noalloc_matches_regular_entry_point_twice(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    name, (M, N), kw = case
    dev = torch.device("cuda")
    cfg = api.make_config(**kw)
    for call in range(2):
        x = workloads.normal_with_outliers(M, N, seed=100 * call + M % 97, fraction=0.002,
                                           gain=40.0).to(dev)
        ref = api.nvfp4_quantize(x, **kw)
        out = api.alloc_outputs(M, N, dev, kw.get("rowwise", True), kw.get("columnwise", False))
        for v in out.values():
            v.fill_(0x5A if v.dtype == torch.uint8 else float("nan"))
        status = _noalloc(x, out, cfg)
        assert status == 0, _lib.load().nvfp4_status_string(status).decode()
        torch.cuda.synchronize()
        for k in KEYS:
            if k not in ref:
                continue
            a, b = out[k].cpu().numpy(), ref[k].cpu().numpy()
            if a.dtype == np.float32:
                a, b = a.view(np.uint32), b.view(np.uint32)
            assert np.array_equal(a, b), "%s call %d: %s differs" % (name, call, k)


def test_noalloc_rejects_bad_arguments_before_launching():
    L = _lib.load()
    cfg = api.make_config(rowwise=True)
    p = ctypes.c_void_p(0x10000)
    assert L.nvfp4_quantize_noalloc(p, 0, 32, ctypes.byref(cfg), p, p, p, None, None, None,
                                    None) == 2          # empty tensor
    assert L.nvfp4_quantize_noalloc(p, 32, 24, ctypes.byref(cfg), p, p, p, None, None, None,
                                    None) == 2          # N % 16
    assert L.nvfp4_quantize_noalloc(ctypes.c_void_p(0x10008), 32, 32, ctypes.byref(cfg), p, p,
                                    p, None, None, None, None) == 3  # misaligned input


def _noalloc_status():
    L = _lib.load()
    bits = ctypes.c_uint32(0)
    st = L.nvfp4_noalloc_get_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(bits))
    return st, bits.value


def _same_as_regular(x, kw, what):
    cfg = api.make_config(**kw)
    M, N = x.shape
    ref = api.nvfp4_quantize(x, **kw)
    out = api.alloc_outputs(M, N, x.device, kw.get("rowwise", True), kw.get("columnwise", False))
    status = _noalloc(x, out, cfg)
    assert status == 0, _lib.load().nvfp4_status_string(status).decode()
    torch.cuda.synchronize()
    for k in KEYS:
        if k in ref:
            a, b = out[k].cpu().numpy(), ref[k].cpu().numpy()
            if a.dtype == np.float32:
                a, b = a.view(np.uint32), b.view(np.uint32)
            assert np.array_equal(a, b), "%s: %s differs" % (what, k)


def test_noalloc_timeout_is_reported_by_its_status_query():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    kw = dict(rowwise=True, columnwise=True)
    x = workloads.normal_with_outliers(2048, 4096, seed=31, fraction=0.002, gain=40.0).to(dev)
    _same_as_regular(x, kw, "before")
    assert _noalloc_status() == (0, 0)
    api.nvfp4_debug_fused_extra_arrivals(1)  # the next single-launch call cannot complete
    out = api.alloc_outputs(2048, 4096, dev, True, True)
    assert _noalloc(x, out, api.make_config(**kw)) == 0  # the launch itself succeeds
    status, bits = _noalloc_status()  # waits for the call (about 2 s)
    assert _lib.STATUS_NAMES[status] == "NVFP4_ERR_TIMEOUT" and bits & _lib.DEVICE_TIMEOUT
    assert _noalloc_status() == (0, 0)  # read and cleared
    assert api.nvfp4_get_status(dev) == (0, 0)  # the regular workspace saw nothing
    _same_as_regular(x, kw, "after the timeout")
    assert _noalloc_status() == (0, 0)


def test_noalloc_held_back_ctas_are_taken_over():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    kw = dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x0FF0, round_col="sr",
              seed=5)
    x = workloads.normal_with_outliers(4096, 4096, seed=32, fraction=0.002, gain=40.0).to(dev)
    _same_as_regular(x, kw, "before")
    api.nvfp4_debug_fused_late_ctas(30)
    _same_as_regular(x, kw, "with 30 held-back CTAs")
    assert _noalloc_status() == (0, 0)


def test_noalloc_matches_the_oracle():
    """The entry point's outputs against the oracle itself (not only against the regular
    entry point), with RHT + stochastic rounding columnwise and a ragged shape."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    dev = torch.device("cuda")
    M, N = 1040, 784
    kw = dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x6C39, round_col="sr",
              seed=17, offset=4)
    x = workloads.normal_with_outliers(M, N, seed=61, fraction=0.003, gain=40.0)
    out = api.alloc_outputs(M, N, dev, True, True)
    for v in out.values():
        v.fill_(0x5A if v.dtype == torch.uint8 else float("nan"))
    assert _noalloc(x.to(dev), out, api.make_config(**kw)) == 0
    torch.cuda.synchronize()
    ref = oracle.quantize(x, oracle.Config(rowwise=True, columnwise=True, rht_col=True,
                                           sign_mask=0x6C39, round_col_sr=True, seed=17,
                                           offset=4))
    for k, r in ref.items():
        a, b = out[k].cpu().numpy(), np.asarray(r)
        if a.dtype == np.float32:
            a, b = a.view(np.uint32), b.astype(np.float32).view(np.uint32)
        assert a.shape == b.shape and np.array_equal(a, b), "noalloc vs oracle: %s differs" % k
