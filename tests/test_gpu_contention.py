"""The single-launch quantize while another stream's kernel holds part of the GPU.

A bounded busy kernel (tests/probes/gpu_probes.cu: one-warp CTAs with 48 KiB of shared memory
each, so that no quantize CTA fits beside one, spinning on the global timer for 2.5 s) is
started on a second stream and occupies about half of the SMs. The single-launch quantize is
then launched on a third stream: its CTAs on the free SMs do their own shares, wait 20 us,
take over the shares of the CTAs that cannot start, and quantize them; the CTAs left waiting
for an SM start when the busy kernel ends, find their shares taken and only quantize again.
The call must match the oracle bit for bit and report no timeout, although the busy kernel
holds its SMs for longer than the 2 s limit of the wait. Nothing hangs: every wait involved
is bounded (the busy kernel's 2.5 s, the quantize kernel's 2 s)."""
import time

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import api, workloads

pytestmark = pytest.mark.gpu

KEYS = ("row_codes", "row_scales", "row_gscale", "col_codes", "col_scales", "col_gscale")
BUSY_NS = 2_500_000_000


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("mode", ["rowcol", "rht_sr"])
def test_single_launch_completes_while_another_stream_holds_sms(probe_lib, mode):
    dev = torch.device("cuda")
    M, N = 4096, 4096
    cfg = dict(rowwise=True, columnwise=True, fused_amax=True)
    if mode == "rht_sr":
        cfg.update(rht_col=True, sign_mask=0x6A95, round_col="sr", seed=4242)
    x = workloads.normal_with_outliers(M, N, seed=71, fraction=0.01, gain=30.0)
    xd = x.to(dev)
    out = api.alloc_outputs(M, N, dev, True, True)
    api.nvfp4_quantize(xd, out=out, **cfg)  # set-up and a first run outside the contention
    torch.cuda.synchronize()
    api.nvfp4_debug_fused_takeovers(dev)
    for v in out.values():
        v.zero_()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    started = torch.zeros(1, dtype=torch.int32, device=dev)
    seen = torch.zeros(1, dtype=torch.int32).pin_memory()
    busy_stream, work_stream, poll_stream = (torch.cuda.Stream(dev) for _ in range(3))
    torch.cuda.synchronize()
    rc = probe_lib.probe_busy_launch(sms // 2, BUSY_NS, started.data_ptr(),
                                     busy_stream.cuda_stream)
    assert rc == 0, "CUDA error %d" % rc
    t0 = time.monotonic()
    while True:  # until every busy CTA runs (bounded)
        with torch.cuda.stream(poll_stream):
            seen.copy_(started, non_blocking=True)
        poll_stream.synchronize()
        if int(seen[0]) >= sms // 2:
            break
        assert time.monotonic() - t0 < 2.0, "busy kernel did not start"
        time.sleep(0.001)
    with torch.cuda.stream(work_stream):
        api.nvfp4_quantize(xd, out=out, **cfg)
        done = torch.cuda.Event(enable_timing=False)
        done.record(work_stream)
    # the quantize kernel's own CTAs on the free SMs finish long before the busy kernel ends;
    # the held-out ones complete the launch when it does
    assert not busy_stream.query(), "the busy kernel ended before the quantize launch"
    work_stream.synchronize()
    busy_stream.synchronize()
    assert api.nvfp4_get_status(dev) == (0, 0)
    taken = api.nvfp4_debug_fused_takeovers(dev)
    assert taken > 0, "no share was taken over: the busy kernel held no SM"
    ref = oracle.quantize(x, oracle.Config(rowwise=True, columnwise=True,
                                           rht_col=cfg.get("rht_col", False),
                                           sign_mask=cfg.get("sign_mask", 0),
                                           round_col_sr=cfg.get("round_col") == "sr",
                                           seed=cfg.get("seed", 0)))
    for k in KEYS:
        g, r = _bits(out[k].cpu().numpy()), _bits(ref[k])
        assert np.array_equal(g, r), (mode, k, int((g != r).sum()))
