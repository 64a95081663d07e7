"""Python binding of the C ABI in include/nvfp4.h, with the same entry-point names.

Argument marshalling only: torch supplies device memory and the current CUDA stream; every
step of the computation runs in libnvfp4's kernels. Outputs are allocated here with
torch.empty on the input's device and returned in a dict:

    row_codes  uint8 [M, N/2]    row_scales  uint8 (E4M3 bits) [M, N/16]   row_gscale  float32 [2]
    col_codes  uint8 [N, M/2]    col_scales  uint8 (E4M3 bits) [N, M/16]   col_gscale  float32 [2]

(gscale = [amax, S_dec]; grouped: [E, 2]).
"""
import ctypes

import torch

from . import _lib
from ._lib import Config, NVFP4Error, ROUND_RN, ROUND_SR


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_x(x):
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError("x must be a 2-D torch.bfloat16 tensor")
    if not x.is_cuda:
        raise TypeError("x must live on a CUDA device (see quantize_from_host for host input)")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous (row-major)")


def _round(v):
    if v in ("rn", ROUND_RN, None):
        return ROUND_RN
    if v in ("sr", ROUND_SR):
        return ROUND_SR
    raise ValueError("rounding must be 'rn' or 'sr'")


def make_config(rowwise=True, columnwise=False, block2d=False, round_row="rn", round_col="rn",
                rht_col=False, sign_mask=0, seed=0, offset=0, fused_amax=False,
                fast_math=False, swizzle_scales=False) -> Config:
    return Config(rowwise=int(bool(rowwise)), columnwise=int(bool(columnwise)),
                  block2d=int(bool(block2d)), round_row=_round(round_row),
                  round_col=_round(round_col), rht_col=int(bool(rht_col)),
                  rht_sign_mask=int(sign_mask), rng_offset=int(offset), rng_seed=int(seed),
                  fused_amax=int(bool(fused_amax)), fast_math=int(bool(fast_math)),
                  swizzle_scales=int(bool(swizzle_scales)))


def _raise_if(status, where):
    if status != _lib.NVFP4_OK:
        raise NVFP4Error(status, where)


def nvfp4_amax(x, rht_col=False, sign_mask=0):
    """Per-tensor amax: returns (max |x|, max |RHT(x)| if rht_col else max |x|) as float32[1]
    device tensors."""
    _check_x(x)
    L = _lib.load()
    M, N = x.shape
    cfg = make_config(rht_col=rht_col, sign_mask=sign_mask)
    a_row = torch.empty(1, dtype=torch.float32, device=x.device)
    a_col = torch.empty(1, dtype=torch.float32, device=x.device)
    _raise_if(L.nvfp4_amax(_ptr(x), M, N, ctypes.byref(cfg), _ptr(a_row), _ptr(a_col),
                           _stream(x.device)), "nvfp4_amax")
    return a_row, a_col


def swizzled_scale_bytes(R, C) -> int:
    """Bytes of an [R][C] scale matrix in the 128 x 4 tiled layout (zero-padded tiles)."""
    return ((R + 127) // 128) * ((C + 3) // 4) * 512


def alloc_outputs(M, N, device, rowwise=True, columnwise=False, col_ld=None, groups=None,
                  swizzled=False):
    """Output buffers of one quantization; swizzled: scale buffers in the 128 x 4 tiled layout
    (flat uint8 tensors, see nvfp4_config.swizzle_scales)."""
    out = {}
    g = () if groups is None else (groups,)
    if rowwise:
        out["row_codes"] = torch.empty((M, N // 2), dtype=torch.uint8, device=device)
        out["row_scales"] = (torch.empty(swizzled_scale_bytes(M, N // 16), dtype=torch.uint8,
                                         device=device) if swizzled else
                             torch.empty((M, N // 16), dtype=torch.uint8, device=device))
        out["row_gscale"] = torch.empty(g + (2,), dtype=torch.float32, device=device)
    if columnwise:
        ld = M if col_ld is None else col_ld
        out["col_codes"] = torch.empty((N, ld // 2), dtype=torch.uint8, device=device)
        out["col_scales"] = (torch.empty(swizzled_scale_bytes(N, ld // 16), dtype=torch.uint8,
                                         device=device) if swizzled else
                             torch.empty((N, ld // 16), dtype=torch.uint8, device=device))
        out["col_gscale"] = torch.empty(g + (2,), dtype=torch.float32, device=device)
    return out


def nvfp4_quantize(x, rowwise=True, columnwise=False, block2d=False, round_row="rn",
                   round_col="rn", rht_col=False, sign_mask=0, seed=0, offset=0,
                   fused_amax=False, amax_row=None, amax_col=None, out=None, fast_math=False,
                   swizzle_scales=False):
    """Quantize a BF16 [M, N] CUDA tensor. amax_row / amax_col (float32[1] device tensors)
    skip the amax pass; `out` reuses preallocated outputs (see alloc_outputs); fast_math
    selects the approximate variant (see nvfp4_config.fast_math); swizzle_scales writes both
    scale outputs in the GEMMs' 128 x 4 tiled layout (see nvfp4_config.swizzle_scales)."""
    _check_x(x)
    L = _lib.load()
    M, N = x.shape
    cfg = make_config(rowwise, columnwise, block2d, round_row, round_col, rht_col, sign_mask,
                      seed, offset, fused_amax, fast_math, swizzle_scales)
    if out is None:
        out = alloc_outputs(M, N, x.device, rowwise, columnwise, swizzled=swizzle_scales)
    g = out.get
    status = L.nvfp4_quantize(_ptr(x), M, N, ctypes.byref(cfg), _ptr(amax_row), _ptr(amax_col),
                              _ptr(g("row_codes")), _ptr(g("row_scales")), _ptr(g("row_gscale")),
                              _ptr(g("col_codes")), _ptr(g("col_scales")), _ptr(g("col_gscale")),
                              _stream(x.device))
    _raise_if(status, "nvfp4_quantize")
    return out


def padded_capacity(counts) -> int:
    return int(sum((int(c) + 15) // 16 * 16 for c in counts))


def nvfp4_quantize_grouped(x, offsets, col_capacity=None, rowwise=True, columnwise=True,
                           round_row="rn", round_col="rn", rht_col=False, sign_mask=0, seed=0,
                           offset=0, out=None, fast_math=False, block2d=False, amax_row=None,
                           amax_col=None):
    """Grouped quantization of a packed BF16 [T, H] tensor; `offsets` is an int32 [E] device
    tensor of cumulative expert ends. col_capacity defaults to T + 16 * E rounded up to a
    multiple of 32 (always enough; a multiple of 32 keeps the columnwise codes' rows 16-byte
    aligned, so that whole tiles leave by TMA store).
    block2d: 16x16 tiles per expert (stacked expert weights), no RHT or SR. amax_row /
    amax_col (float32 [E] device tensors, e.g. from nvfp4_amax_grouped) skip the amax pass."""
    _check_x(x)
    L = _lib.load()
    if offsets.dtype != torch.int32 or not offsets.is_cuda or offsets.dim() != 1:
        raise TypeError("offsets must be a 1-D int32 CUDA tensor")
    T, H = x.shape
    E = offsets.shape[0]
    if col_capacity is None:
        col_capacity = ((T + 15) // 16 * 16 + 16 * E + 31) // 32 * 32
    cfg = make_config(rowwise, columnwise, block2d, round_row, round_col, rht_col, sign_mask, seed,
                      offset, fast_math=fast_math)
    if out is None:
        out = alloc_outputs(T, H, x.device, rowwise, columnwise, col_ld=col_capacity, groups=E)
    g = out.get
    status = L.nvfp4_quantize_grouped(
        _ptr(x), T, H, _ptr(offsets), E, col_capacity, ctypes.byref(cfg), _ptr(amax_row),
        _ptr(amax_col), _ptr(g("row_codes")), _ptr(g("row_scales")), _ptr(g("row_gscale")),
        _ptr(g("col_codes")), _ptr(g("col_scales")), _ptr(g("col_gscale")), _stream(x.device))
    _raise_if(status, "nvfp4_quantize_grouped")
    return out


def nvfp4_amax_grouped(x, offsets, rht_col=False, sign_mask=0):
    """Per-expert amax of a packed grouped tensor: (max |x|, max |RHT(x)| if rht_col else
    max |x|) as float32 [E] device tensors."""
    _check_x(x)
    L = _lib.load()
    T, H = x.shape
    E = offsets.shape[0]
    cfg = make_config(rht_col=rht_col, sign_mask=sign_mask)
    a_row = torch.empty(E, dtype=torch.float32, device=x.device)
    a_col = torch.empty(E, dtype=torch.float32, device=x.device)
    _raise_if(L.nvfp4_amax_grouped(_ptr(x), T, H, _ptr(offsets), E, ctypes.byref(cfg),
                                   _ptr(a_row), _ptr(a_col), _stream(x.device)),
              "nvfp4_amax_grouped")
    return a_row, a_col


def nvfp4_dequantize(codes, scales, gscale):
    """FP32 [R, C] reconstruction of codes [R, C/2] with scales [R, C/16] and gscale [2]."""
    L = _lib.load()
    R, half = codes.shape
    C = 2 * half
    out = torch.empty((R, C), dtype=torch.float32, device=codes.device)
    _raise_if(L.nvfp4_dequantize(_ptr(codes), _ptr(scales), _ptr(gscale), R, C, _ptr(out),
                                 _stream(codes.device)), "nvfp4_dequantize")
    return out


def nvfp4_dequantize_ex(codes, scales, gscale, inverse_rht=False, sign_mask=0, bf16=False):
    """nvfp4_dequantize, then optionally the inverse RHT of every 16-element block of every row
    (columnwise RHT outputs) and BF16 rounding: FP32 or BF16 [R, C]."""
    L = _lib.load()
    R, half = codes.shape
    C = 2 * half
    out = torch.empty((R, C), dtype=torch.bfloat16 if bf16 else torch.float32,
                      device=codes.device)
    _raise_if(L.nvfp4_dequantize_ex(_ptr(codes), _ptr(scales), _ptr(gscale), R, C,
                                    int(bool(inverse_rht)), int(sign_mask), int(bool(bf16)),
                                    _ptr(out), _stream(codes.device)), "nvfp4_dequantize_ex")
    return out


def nvfp4_swizzle_scales(scales, out=None):
    """uint8 [R, C] E4M3 scales -> the flat 128 x 4 tiled layout of the block-scaled GEMMs
    (into `out` when given)."""
    L = _lib.load()
    src = scales.contiguous()
    R, C = src.shape
    if out is None:
        out = torch.empty(swizzled_scale_bytes(R, C), dtype=torch.uint8, device=src.device)
    _raise_if(L.nvfp4_swizzle_scales(_ptr(src), R, C, _ptr(out), _stream(src.device)),
              "nvfp4_swizzle_scales")
    return out


def nvfp4_rmsnorm_amax(x, weight, eps=1e-6, weight_bias=0.0, y=None, amax=None):
    """RMSNorm producer with the amax in its epilogue: returns (y BF16 [M, N], amax float32[1])
    device tensors."""
    _check_x(x)
    L = _lib.load()
    M, N = x.shape
    if y is None:
        y = torch.empty_like(x)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _raise_if(L.nvfp4_rmsnorm_amax(_ptr(x), _ptr(weight.contiguous()), M, N, float(eps),
                                   float(weight_bias), _ptr(y), _ptr(amax), _stream(x.device)),
              "nvfp4_rmsnorm_amax")
    return y, amax


def nvfp4_rmsnorm_quantize(x, weight, eps=1e-6, weight_bias=0.0, out=None, y=None, amax=None,
                           **cfg):
    """RMSNorm with the amax in its epilogue, then NVFP4 quantization of the normed tensor
    (options as nvfp4_quantize). Returns the quantize outputs plus "y" and "amax"."""
    _check_x(x)
    L = _lib.load()
    M, N = x.shape
    c = make_config(cfg.get("rowwise", True), cfg.get("columnwise", False),
                    cfg.get("block2d", False), cfg.get("round_row", "rn"), cfg.get("round_col", "rn"),
                    cfg.get("rht_col", False), cfg.get("sign_mask", 0), cfg.get("seed", 0),
                    cfg.get("offset", 0), cfg.get("fused_amax", False), cfg.get("fast_math", False))
    if out is None:
        out = alloc_outputs(M, N, x.device, bool(c.rowwise), bool(c.columnwise))
    if y is None:
        y = torch.empty_like(x)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    p = lambda k: _ptr(out.get(k))
    _raise_if(L.nvfp4_rmsnorm_quantize(_ptr(x), _ptr(weight.contiguous()), M, N, float(eps),
                                       float(weight_bias), ctypes.byref(c), _ptr(y), _ptr(amax),
                                       p("row_codes"), p("row_scales"), p("row_gscale"),
                                       p("col_codes"), p("col_scales"), p("col_gscale"),
                                       _stream(x.device)), "nvfp4_rmsnorm_quantize")
    return dict(out, y=y, amax=amax)


MX_FORMATS = {"e4m3": 0, "e5m2": 1, "e2m1": 2}


def _mx_format(fmt):
    if fmt in MX_FORMATS:
        return MX_FORMATS[fmt]
    raise ValueError("MX format must be one of %s" % sorted(MX_FORMATS))


def alloc_mx_outputs(M, N, device, fmt="e4m3", rowwise=True, columnwise=False):
    """Output buffers of nvfp4_mx_quantize (torch.empty on `device`)."""
    fp4 = _mx_format(fmt) == MX_FORMATS["e2m1"]
    out = {}
    if rowwise:
        out["row_codes"] = torch.empty((M, N // 2 if fp4 else N), dtype=torch.uint8, device=device)
        out["row_scales"] = torch.empty((M, N // 32), dtype=torch.uint8, device=device)
    if columnwise:
        out["col_codes"] = torch.empty((N, M // 2 if fp4 else M), dtype=torch.uint8, device=device)
        out["col_scales"] = torch.empty((N, M // 32), dtype=torch.uint8, device=device)
    return out


def nvfp4_mx_quantize(x, fmt="e4m3", rowwise=True, columnwise=False, out=None):
    """MX quantization (MXFP8 "e4m3" / "e5m2", MXFP4 "e2m1") of a BF16 [M, N] CUDA tensor:
    codes and E8M0 scales (uint8), rowwise and/or columnwise (transposed)."""
    _check_x(x)
    L = _lib.load()
    M, N = x.shape
    f = _mx_format(fmt)
    if out is None:
        out = alloc_mx_outputs(M, N, x.device, fmt, rowwise, columnwise)
    _raise_if(L.nvfp4_mx_quantize(_ptr(x), M, N, f, int(bool(rowwise)), int(bool(columnwise)),
                                  _ptr(out.get("row_codes")), _ptr(out.get("row_scales")),
                                  _ptr(out.get("col_codes")), _ptr(out.get("col_scales")),
                                  _stream(x.device)), "nvfp4_mx_quantize")
    return out


def nvfp4_mx_dequantize(codes, scales, fmt="e4m3"):
    """FP32 [R, C] values of MX codes [R, C] (FP8) or [R, C/2] (FP4) and scales [R, C/32]."""
    L = _lib.load()
    f = _mx_format(fmt)
    R = codes.shape[0]
    C = codes.shape[1] * (2 if f == MX_FORMATS["e2m1"] else 1)
    out = torch.empty((R, C), dtype=torch.float32, device=codes.device)
    _raise_if(L.nvfp4_mx_dequantize(_ptr(codes), _ptr(scales), f, R, C, _ptr(out),
                                    _stream(codes.device)), "nvfp4_mx_dequantize")
    return out


WORKSPACE_BYTES = 16384


def nvfp4_set_workspace(workspace=None):
    """Make a caller-owned CUDA tensor (at least WORKSPACE_BYTES, 256-byte aligned) the current
    device's workspace; None returns to the library's own. Keep the tensor alive meanwhile."""
    L = _lib.load()
    if workspace is None:
        _raise_if(L.nvfp4_set_workspace(None, 0), "nvfp4_set_workspace")
        return
    nbytes = workspace.numel() * workspace.element_size()
    _raise_if(L.nvfp4_set_workspace(_ptr(workspace), nbytes), "nvfp4_set_workspace")


def nvfp4_get_status(device=None):
    """Synchronize the current stream and return (status, device status bits); clears them."""
    L = _lib.load()
    dev = torch.device("cuda") if device is None else torch.device(device)
    bits = ctypes.c_uint32(0)
    status = L.nvfp4_get_status(_stream(dev), ctypes.byref(bits))
    return status, bits.value


def nvfp4_debug_fused_extra_arrivals(extra):
    """Test hook: the next single-launch amax call waits for `extra` arrivals more than its grid
    has shares, so its bounded wait runs out (about 2 s) and it reports NVFP4_DEVICE_TIMEOUT."""
    _raise_if(_lib.load().nvfp4_debug_fused_extra_arrivals(int(extra)),
              "nvfp4_debug_fused_extra_arrivals")


def nvfp4_debug_fused_late_ctas(count):
    """Test hook: in the next single-launch amax call the last `count` CTAs hold back until
    every share has arrived, so the other CTAs take their shares over."""
    _raise_if(_lib.load().nvfp4_debug_fused_late_ctas(int(count)), "nvfp4_debug_fused_late_ctas")


def nvfp4_debug_fused_takeovers(device=None):
    """Synchronize the current stream and return (and clear) the count of shares taken over by
    single-launch calls on the device's workspace."""
    L = _lib.load()
    dev = torch.device("cuda") if device is None else torch.device(device)
    n = ctypes.c_uint32(0)
    _raise_if(L.nvfp4_debug_fused_takeovers(_stream(dev), ctypes.byref(n)),
              "nvfp4_debug_fused_takeovers")
    return n.value


def nvfp4_noalloc_get_status(device=None):
    """Synchronize the current stream and return (status, device status bits) of the no-alloc
    entry point's own status word; clears it."""
    L = _lib.load()
    dev = torch.device("cuda") if device is None else torch.device(device)
    bits = ctypes.c_uint32(0)
    status = L.nvfp4_noalloc_get_status(_stream(dev), ctypes.byref(bits))
    return status, bits.value


def nvfp4_debug_fail_next_launch(on=True):
    """Test hook: the next quantize call launches an empty grid, which the runtime rejects, so
    the call raises NVFP4Error(NVFP4_ERR_CUDA); the call after it runs normally."""
    _raise_if(_lib.load().nvfp4_debug_fail_next_launch(int(bool(on))),
              "nvfp4_debug_fail_next_launch")


def quantize_from_host(x_host, pinned_out=None, **kw):
    """End-to-end call for host data: copy a pinned host BF16 tensor to the device, quantize,
    and copy every output back into pinned host tensors (all on the current stream)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    x = x_host.to(dev, non_blocking=True)
    out = nvfp4_quantize(x, **kw)
    if pinned_out is None:
        pinned_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                      for k, v in out.items()}
    for k, v in out.items():
        pinned_out[k].copy_(v, non_blocking=True)
    return pinned_out


class HostPipeline:
    """nvfp4_host_pipeline_*: quantization of host (pinned) BF16 [M, N] tensors with the copies
    of consecutive submissions overlapped. The device staging is allocated once, here."""

    def __init__(self, M, N, depth=2, **kw):
        L = _lib.load()
        self.M, self.N = M, N
        self.cfg = make_config(fused_amax=kw.pop("fused_amax", True), **kw)
        self.rowwise = bool(self.cfg.rowwise)
        self.columnwise = bool(self.cfg.columnwise)
        self.device = torch.device("cuda", torch.cuda.current_device())
        handle = ctypes.c_void_p()
        _raise_if(L.nvfp4_host_pipeline_create(M, N, ctypes.byref(self.cfg), depth,
                                               ctypes.byref(handle)), "nvfp4_host_pipeline_create")
        self._h = handle

    def alloc_host_outputs(self):
        """Pinned host tensors for one submission's outputs."""
        out = {}
        M, N = self.M, self.N
        if self.rowwise:
            out["row_codes"] = torch.empty((M, N // 2), dtype=torch.uint8, pin_memory=True)
            out["row_scales"] = torch.empty((M, N // 16), dtype=torch.uint8, pin_memory=True)
            out["row_gscale"] = torch.empty(2, dtype=torch.float32, pin_memory=True)
        if self.columnwise:
            out["col_codes"] = torch.empty((N, M // 2), dtype=torch.uint8, pin_memory=True)
            out["col_scales"] = torch.empty((N, M // 16), dtype=torch.uint8, pin_memory=True)
            out["col_gscale"] = torch.empty(2, dtype=torch.float32, pin_memory=True)
        return out

    def submit(self, x_host, out_host):
        """Enqueue x_host (pinned BF16 [M, N]); outputs land in out_host (alloc_host_outputs)."""
        if x_host.device.type != "cpu" or x_host.dtype != torch.bfloat16 or \
                tuple(x_host.shape) != (self.M, self.N) or not x_host.is_contiguous():
            raise ValueError("x_host must be a contiguous CPU bfloat16 [%d, %d] tensor"
                             % (self.M, self.N))
        L = _lib.load()
        p = lambda k: ctypes.c_void_p(out_host[k].data_ptr()) if k in out_host else None
        _raise_if(L.nvfp4_host_pipeline_submit(
            self._h, ctypes.c_void_p(x_host.data_ptr()), p("row_codes"), p("row_scales"),
            p("row_gscale"), p("col_codes"), p("col_scales"), p("col_gscale"),
            _stream(self.device)), "nvfp4_host_pipeline_submit")

    def join(self):
        """Make the current stream wait until every submission's outputs are in host memory."""
        _raise_if(_lib.load().nvfp4_host_pipeline_join(self._h, _stream(self.device)),
                  "nvfp4_host_pipeline_join")

    def close(self):
        if self._h:
            _lib.load().nvfp4_host_pipeline_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class GroupedHostPipeline(HostPipeline):
    """nvfp4_host_pipeline_create_grouped / _submit_grouped: grouped BF16 [T, H] host tensors
    with E experts (offsets given per submission as a host int32 [E] array of expert ends),
    quantized by nvfp4_quantize_grouped with col_capacity columns of columnwise outputs."""

    def __init__(self, T, H, E, col_capacity, depth=2, **kw):
        L = _lib.load()
        self.M, self.N, self.E, self.cap = T, H, E, col_capacity
        kw.pop("fused_amax", None)
        self.cfg = make_config(fused_amax=False, **kw)
        self.rowwise = bool(self.cfg.rowwise)
        self.columnwise = bool(self.cfg.columnwise)
        self.device = torch.device("cuda", torch.cuda.current_device())
        handle = ctypes.c_void_p()
        _raise_if(L.nvfp4_host_pipeline_create_grouped(T, H, E, col_capacity,
                                                       ctypes.byref(self.cfg), depth,
                                                       ctypes.byref(handle)),
                  "nvfp4_host_pipeline_create_grouped")
        self._h = handle

    def alloc_host_outputs(self):
        out = {}
        T, H, E, cap = self.M, self.N, self.E, self.cap
        if self.rowwise:
            out["row_codes"] = torch.empty((T, H // 2), dtype=torch.uint8, pin_memory=True)
            out["row_scales"] = torch.empty((T, H // 16), dtype=torch.uint8, pin_memory=True)
            out["row_gscale"] = torch.empty((E, 2), dtype=torch.float32, pin_memory=True)
        if self.columnwise:
            out["col_codes"] = torch.empty((H, cap // 2), dtype=torch.uint8, pin_memory=True)
            out["col_scales"] = torch.empty((H, cap // 16), dtype=torch.uint8, pin_memory=True)
            out["col_gscale"] = torch.empty((E, 2), dtype=torch.float32, pin_memory=True)
        return out

    def submit(self, x_host, offsets_host, out_host):
        """Enqueue x_host (pinned BF16 [T, H]) with offsets_host (host int32 [E]); outputs land
        in out_host (alloc_host_outputs)."""
        if x_host.device.type != "cpu" or x_host.dtype != torch.bfloat16 or \
                tuple(x_host.shape) != (self.M, self.N) or not x_host.is_contiguous():
            raise ValueError("x_host must be a contiguous CPU bfloat16 [%d, %d] tensor"
                             % (self.M, self.N))
        if offsets_host.device.type != "cpu" or offsets_host.dtype != torch.int32 or \
                tuple(offsets_host.shape) != (self.E,) or not offsets_host.is_contiguous():
            raise ValueError("offsets_host must be a contiguous CPU int32 [%d] tensor" % self.E)
        L = _lib.load()
        p = lambda k: ctypes.c_void_p(out_host[k].data_ptr()) if k in out_host else None
        _raise_if(L.nvfp4_host_pipeline_submit_grouped(
            self._h, ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(offsets_host.data_ptr()),
            p("row_codes"), p("row_scales"), p("row_gscale"), p("col_codes"), p("col_scales"),
            p("col_gscale"), _stream(self.device)), "nvfp4_host_pipeline_submit_grouped")
