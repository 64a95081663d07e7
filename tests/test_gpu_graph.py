"""CUDA-graph capture and the bounded wait of the single-launch amax.

A captured call is replayed on new data written into the same input buffer; every replay must
match the oracle on that data bit for bit. The data's amax falls from replay to replay, so a
barrier that kept its maxima from an earlier replay (or counted arrivals against a target fixed
at capture) would show up as a wrong global scale.

The timeout test asks the next single-launch call to wait for one share more than its grid
has: every CTA gives up after its bounded wait, records NVFP4_DEVICE_TIMEOUT and exits, and the
call after it runs normally on the same workspace. Nothing faults or hangs: the wait has a
limit. The take-over tests hold the last CTAs of a launch back (a test hook, bounded) until
every share has arrived: the other CTAs must take their shares over, the outputs must be the
oracle's, and a launch whose held-back CTAs start only after the others have given up must
leave the workspace ready for the next call.
The launch-failure test has the next call launch an empty grid, which the runtime rejects
before anything reaches the GPU: the call reports NVFP4_ERR_CUDA, leaves no error behind for
the next CUDA call, and the call after it is correct."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import _lib, api, workloads

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
            assert g.shape == r.shape, (what, k)
            assert np.array_equal(g, r), (what, k, int((g != r).sum()))


def _oracle_cfg(cfg):
    return oracle.Config(rowwise=cfg.get("rowwise", True), columnwise=cfg.get("columnwise", False),
                         block2d=cfg.get("block2d", False),
                         round_row_sr=cfg.get("round_row", "rn") == "sr",
                         round_col_sr=cfg.get("round_col", "rn") == "sr",
                         rht_col=cfg.get("rht_col", False), sign_mask=cfg.get("sign_mask", 0),
                         seed=cfg.get("seed", 0), offset=cfg.get("offset", 0))


# the data of replay k: the same shape, gains falling so that each amax is below the last
GAINS = (60.0, 20.0, 5.0, 40.0)

MODES = {
    "fused_rowcol": dict(rowwise=True, columnwise=True, fused_amax=True),
    "fused_rht_sr": dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x3C5A,
                         round_col="sr", seed=77, offset=3, fused_amax=True),
    "fused_2d": dict(rowwise=True, columnwise=True, block2d=True, fused_amax=True),
    "two_pass_rowcol": dict(rowwise=True, columnwise=True, fused_amax=False),
}


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("shape", [(304, 1040), (2048, 4096)], ids=lambda s: "%dx%d" % s)
def test_captured_call_replays_on_new_data(mode, shape):
    dev = _cuda()
    M, N = shape
    cfg = MODES[mode]
    xs = [workloads.normal_with_outliers(M, N, seed=50 + k, fraction=0.01, gain=g)
          for k, g in enumerate(GAINS)]
    static_x = xs[0].to(dev)
    out = api.alloc_outputs(M, N, dev, cfg["rowwise"], cfg["columnwise"])
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside capture (workspace, kernel setup)
        api.nvfp4_quantize(static_x, out=out, **cfg)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.nvfp4_quantize(static_x, out=out, **cfg)
    for k, x in enumerate(xs):
        static_x.copy_(x.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        _same(out, oracle.quantize(x, _oracle_cfg(cfg)), "%s replay %d" % (mode, k))
    status, bits = api.nvfp4_get_status(dev)
    assert (status, bits) == (0, 0)


def _noalloc(x, out, cfg):
    L = _lib.load()
    M, N = x.shape
    p = lambda k: ctypes.c_void_p(out[k].data_ptr()) if k in out else None
    stream = ctypes.c_void_p(torch.cuda.current_stream(x.device).cuda_stream)
    status = L.nvfp4_quantize_noalloc(ctypes.c_void_p(x.data_ptr()), M, N,
                                      ctypes.byref(api.make_config(**cfg)), p("row_codes"),
                                      p("row_scales"), p("row_gscale"), p("col_codes"),
                                      p("col_scales"), p("col_gscale"), stream)
    assert status == 0, L.nvfp4_status_string(status).decode()


def test_captured_noalloc_call_replays_on_new_data():
    dev = _cuda()
    M, N = 640, 2064
    xs = [workloads.normal_with_outliers(M, N, seed=90 + k, fraction=0.01, gain=g)
          for k, g in enumerate(GAINS)]
    static_x = xs[0].to(dev)
    out = api.alloc_outputs(M, N, dev, True, True)
    cfg = dict(rowwise=True, columnwise=True, rht_col=True, sign_mask=0x0F0F)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # the first call (set-up) outside capture
        _noalloc(static_x, out, cfg)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _noalloc(static_x, out, cfg)
    for k, x in enumerate(xs):
        static_x.copy_(x.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        _same(out, oracle.quantize(x, _oracle_cfg(cfg)), "noalloc replay %d" % k)


@pytest.mark.parametrize("shape", [(64, 256), (4096, 4096)], ids=lambda s: "%dx%d" % s)
def test_barrier_wait_runs_out_then_next_call_is_correct(shape):
    dev = _cuda()
    M, N = shape
    x = workloads.normal_with_outliers(M, N, seed=7, fraction=0.01, gain=30.0)
    cfg = dict(rowwise=True, columnwise=True, fused_amax=True)
    api.nvfp4_quantize(x.to(dev), **cfg)  # set-up outside the measured part
    assert api.nvfp4_get_status(dev) == (0, 0)
    api.nvfp4_debug_fused_extra_arrivals(1)  # one arrival more than the grid can make
    api.nvfp4_quantize(x.to(dev), **cfg)
    status, bits = api.nvfp4_get_status(dev)  # waits for the launch (about 2 s)
    assert _lib.STATUS_NAMES[status] == "NVFP4_ERR_TIMEOUT" and bits & _lib.DEVICE_TIMEOUT, \
        (status, bits)
    # the hook was consumed and the last CTA readied the counts: a normal call again
    out = api.nvfp4_quantize(x.to(dev), **cfg)
    torch.cuda.synchronize()
    _same(out, oracle.quantize(x, _oracle_cfg(cfg)), "after timeout")
    assert api.nvfp4_get_status(dev) == (0, 0)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_pass"])
def test_failed_launch_is_reported_and_leaves_no_error_behind(fused):
    dev = _cuda()
    M, N = 256, 512
    x = workloads.normal_with_outliers(M, N, seed=3, fraction=0.01, gain=30.0)
    cfg = dict(rowwise=True, columnwise=True, fused_amax=fused)
    xd = x.to(dev)
    api.nvfp4_quantize(xd, **cfg)
    torch.cuda.synchronize()
    api.nvfp4_debug_fail_next_launch()
    with pytest.raises(_lib.NVFP4Error) as e:
        api.nvfp4_quantize(xd, **cfg)
    assert "NVFP4_ERR_CUDA" in str(e.value)
    # torch's next launch and error check see no leftover error
    y = (xd.float() * 2).sum()
    torch.cuda.synchronize()
    assert torch.isfinite(y)
    out = api.nvfp4_quantize(xd, **cfg)
    torch.cuda.synchronize()
    _same(out, oracle.quantize(x, _oracle_cfg(cfg)), "after a failed launch")
    assert api.nvfp4_get_status(dev) == (0, 0)


GAINS6 = (50.0, 2.0, 30.0, 7.0, 90.0, 1.0)


@pytest.mark.parametrize("mode", ["fused_rowcol", "fused_rht_sr"])
def test_back_to_back_single_launch_calls(mode):
    """Single-launch calls queued with no synchronization in between: after the first one,
    each may start on SMs the previous one leaves (programmatic dependent launch) and waits for
    it at entry. A full grid (one CTA per SM); every call's outputs match the oracle, into
    separate buffers and into one buffer reused by all (the last call's outputs remain)."""
    dev = _cuda()
    M, N = 2048, 4096
    cfg = MODES[mode]
    xs_cpu = [workloads.normal_with_outliers(M, N, seed=300 + k, fraction=0.01, gain=g)
              for k, g in enumerate(GAINS6)]
    xs = [x.to(dev) for x in xs_cpu]
    torch.cuda.synchronize()
    outs = [api.nvfp4_quantize(x, **cfg) for x in xs]
    shared = api.alloc_outputs(M, N, dev, True, True)
    for x in xs:
        api.nvfp4_quantize(x, out=shared, **cfg)
    torch.cuda.synchronize()
    refs = [oracle.quantize(x, _oracle_cfg(cfg)) for x in xs_cpu]
    for k, (o, r) in enumerate(zip(outs, refs)):
        _same(o, r, "%s call %d" % (mode, k))
    _same(shared, refs[-1], "%s reused outputs" % mode)
    assert api.nvfp4_get_status(dev) == (0, 0)


TAKEOVER_MODES = ["fused_rowcol", "fused_rht_sr", "fused_2d"]


@pytest.mark.parametrize("mode", TAKEOVER_MODES)
@pytest.mark.parametrize("late", [1, 40, 120])
def test_held_back_ctas_have_their_shares_taken_over(mode, late):
    """The last `late` CTAs of a full grid (one per SM) start their shares only after every
    share has arrived, so the other CTAs take them over; the held-back CTAs then find their
    shares taken and quantize them again (the same bytes)."""
    dev = _cuda()
    M, N = 4096, 4096
    cfg = MODES[mode]
    x = workloads.normal_with_outliers(M, N, seed=500 + late, fraction=0.01, gain=25.0)
    xd = x.to(dev)
    api.nvfp4_quantize(xd, **cfg)
    torch.cuda.synchronize()
    api.nvfp4_debug_fused_takeovers(dev)  # clear the count
    api.nvfp4_debug_fused_late_ctas(late)
    out = api.nvfp4_quantize(xd, **cfg)
    torch.cuda.synchronize()
    assert api.nvfp4_get_status(dev) == (0, 0)
    taken = api.nvfp4_debug_fused_takeovers(dev)
    assert taken == late, (taken, late)
    ref = oracle.quantize(x, _oracle_cfg(cfg))
    _same(out, ref, "%s with %d held-back CTAs" % (mode, late))
    # and the next call, on the counts the last CTA readied
    out = api.nvfp4_quantize(xd, **cfg)
    torch.cuda.synchronize()
    _same(out, ref, "%s after the take-over" % mode)
    assert api.nvfp4_get_status(dev) == (0, 0)
    assert api.nvfp4_debug_fused_takeovers(dev) == 0


def test_ctas_starting_after_a_timeout_leave_the_next_call_correct():
    """A launch that times out (one share more awaited than exists) while its last CTAs are
    held back until that count is reached (which never happens: they give up their hold after
    the bounded wait, about 2 s, and only then claim their shares, long after the others gave
    up): it reports NVFP4_DEVICE_TIMEOUT, and the next call must match the oracle bit for bit
    and report nothing (no count or maximum of the timed-out launch survives)."""
    dev = _cuda()
    M, N = 4096, 4096
    cfg = MODES["fused_rowcol"]
    xs = [workloads.normal_with_outliers(M, N, seed=600 + k, fraction=0.01, gain=g)
          for k, g in enumerate((80.0, 3.0))]
    api.nvfp4_quantize(xs[0].to(dev), **cfg)
    torch.cuda.synchronize()
    api.nvfp4_debug_fused_extra_arrivals(1)
    api.nvfp4_debug_fused_late_ctas(20)
    api.nvfp4_quantize(xs[0].to(dev), **cfg)  # larger amax than the next call's data
    status, bits = api.nvfp4_get_status(dev)  # about 4 s: the hold, then the wait
    assert _lib.STATUS_NAMES[status] == "NVFP4_ERR_TIMEOUT" and bits & _lib.DEVICE_TIMEOUT
    api.nvfp4_debug_fused_takeovers(dev)
    out = api.nvfp4_quantize(xs[1].to(dev), **cfg)
    torch.cuda.synchronize()
    _same(out, oracle.quantize(xs[1], _oracle_cfg(cfg)), "after a timeout with late CTAs")
    assert api.nvfp4_get_status(dev) == (0, 0)
    assert api.nvfp4_debug_fused_takeovers(dev) == 0
