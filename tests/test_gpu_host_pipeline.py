"""nvfp4_host_pipeline_*: host tensors in, host outputs out, copies of consecutive submissions
overlapped. Every submission's host outputs must equal nvfp4_quantize's on the device copy of
the same input, bit for bit, whatever the depth and however the slots are reused."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quantize_gb300 import api, workloads

pytestmark = pytest.mark.gpu

CONFIGS = [
    ("rowcol_rtne", dict(rowwise=True, columnwise=True)),
    ("row_rtne_col_rht_sr", dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x3C5A,
                                 round_col="sr", seed=17)),
    ("col_only_two_pass", dict(rowwise=False, columnwise=True, fused_amax=False)),
]


def _same(a, b, what):
    a, b = a.cpu().numpy(), b.cpu().numpy()
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    assert np.array_equal(a, b), what


@pytest.mark.parametrize("depth", [1, 2, 3])
@pytest.mark.parametrize("name,kw", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_pipeline_outputs_match_device_quantize(depth, name, kw):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N = 320, 1040   # ragged against the 64 x 256 tiles
    xs = [workloads.normal_with_outliers(M, N, seed=s, fraction=0.003, gain=30.0).pin_memory()
          for s in (11, 12, 13)]
    pipe = api.HostPipeline(M, N, depth=depth, **kw)
    try:
        outs = []
        for i in range(5):   # more submissions than slots: every slot is reused
            o = pipe.alloc_host_outputs()
            for v in o.values():
                v.fill_(0x77 if v.dtype == torch.uint8 else float("nan"))
            pipe.submit(xs[i % 3], o)
            outs.append(o)
        pipe.join()
        torch.cuda.synchronize()
        dkw = dict(kw)
        dkw.pop("fused_amax", None)
        for i, o in enumerate(outs):
            ref = api.nvfp4_quantize(xs[i % 3].cuda(), **dkw)
            assert sorted(o) == sorted(ref)
            for k in ref:
                _same(o[k], ref[k], "%s depth %d submission %d %s" % (name, depth, i, k))
    finally:
        pipe.close()


def test_pipeline_reused_host_buffers_hold_the_last_submission():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N = 256, 512
    xs = [workloads.normal(M, N, 1.0, s).pin_memory() for s in (3, 4)]
    pipe = api.HostPipeline(M, N, depth=2, rowwise=True, columnwise=True)
    try:
        o = pipe.alloc_host_outputs()
        for i in range(7):
            pipe.submit(xs[i % 2], o)
        pipe.join()
        torch.cuda.synchronize()
        ref = api.nvfp4_quantize(xs[0].cuda(), rowwise=True, columnwise=True)
        for k in ref:
            _same(o[k], ref[k], k)
    finally:
        pipe.close()


def test_pipeline_rejects_wrong_host_tensor():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pipe = api.HostPipeline(64, 64, depth=1, rowwise=True)
    try:
        with pytest.raises(ValueError):
            pipe.submit(torch.zeros((64, 32), dtype=torch.bfloat16), pipe.alloc_host_outputs())
    finally:
        pipe.close()


GROUPED_CONFIGS = [
    ("rowcol_rtne", dict(rowwise=True, columnwise=True)),
    ("row_rtne_col_rht_sr", dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x5AC3,
                                 round_col="sr", seed=23)),
    ("2d_weights", dict(rowwise=True, columnwise=True, block2d=True)),
]


@pytest.mark.parametrize("depth", [1, 2])
@pytest.mark.parametrize("name,kw", GROUPED_CONFIGS, ids=[c[0] for c in GROUPED_CONFIGS])
def test_grouped_pipeline_outputs_match_device_quantize(depth, name, kw):
    """Grouped submissions with different inputs and expert offsets per submission (empty and
    ragged experts): each host output equals nvfp4_quantize_grouped's on the device copy."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    T, H, E = 400, 784, 5
    cap = T + 16 * E
    offs = [np.cumsum(c).astype(np.int32) for c in
            ([0, 100, 33, 200, 67], [17, 17, 0, 300, 66], [400, 0, 0, 0, 0])]
    xs = [workloads.normal_with_outliers(T, H, seed=s, fraction=0.003, gain=30.0).pin_memory()
          for s in (31, 32, 33)]
    pipe = api.GroupedHostPipeline(T, H, E, cap, depth=depth, **kw)
    try:
        outs = []
        for i in range(5):   # more submissions than slots: every slot is reused
            o = pipe.alloc_host_outputs()
            for v in o.values():
                v.fill_(0x77 if v.dtype == torch.uint8 else float("nan"))
            pipe.submit(xs[i % 3], torch.from_numpy(offs[i % 3]), o)
            outs.append(o)
        pipe.join()
        torch.cuda.synchronize()
        for i, o in enumerate(outs):
            ref = api.alloc_outputs(T, H, torch.device("cuda"), True, True, col_ld=cap, groups=E)
            for v in ref.values():
                v.fill_(0x77 if v.dtype == torch.uint8 else float("nan"))
            api.nvfp4_quantize_grouped(xs[i % 3].cuda(), torch.from_numpy(offs[i % 3]).cuda(),
                                       col_capacity=cap, out=ref, **kw)
            torch.cuda.synchronize()
            assert sorted(o) == sorted(ref)
            for k in ref:
                _same(o[k], ref[k], "%s depth %d submission %d %s" % (name, depth, i, k))
    finally:
        pipe.close()


def test_grouped_pipeline_refuses_bad_offsets_on_the_host():
    """Offsets that decrease, pass T, or need more columns than the capacity are refused before
    anything is enqueued; a later valid submission still runs."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ctypes
    from nvfp4_block_scaled_quantize_gb300 import _lib
    T, H, E = 128, 256, 3
    pipe = api.GroupedHostPipeline(T, H, E, 144, depth=1, rowwise=True, columnwise=True)
    try:
        x = workloads.normal(T, H, 1.0, seed=5).pin_memory()
        o = pipe.alloc_host_outputs()
        L = _lib.load()
        p = lambda k: ctypes.c_void_p(o[k].data_ptr())  # noqa: E731
        for bad in ([40, 30, 128], [40, 80, 129], [1, 2, 128]):   # the last needs 160 columns
            offs = torch.tensor(bad, dtype=torch.int32)
            st = L.nvfp4_host_pipeline_submit_grouped(
                pipe._h, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(offs.data_ptr()),
                p("row_codes"), p("row_scales"), p("row_gscale"), p("col_codes"),
                p("col_scales"), p("col_gscale"), None)
            assert _lib.STATUS_NAMES[st] == "NVFP4_ERR_INVALID_ARG", bad
        pipe.submit(x, torch.tensor([40, 80, 128], dtype=torch.int32), o)
        pipe.join()
        torch.cuda.synchronize()
        ref = api.nvfp4_quantize_grouped(x.cuda(), torch.tensor([40, 80, 128], dtype=torch.int32).cuda(),
                                         col_capacity=144)
        for k in ref:
            _same(o[k], ref[k], k)
    finally:
        pipe.close()
