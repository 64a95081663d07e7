"""The C ABI without a GPU: the library builds, loads, exports every entry point the header
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from nvfp4_block_scaled_quantize_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "nvfp4.h")
FAKE = 0x10000  # a 16-byte-aligned address never dereferenced: argument checks come first


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z_]+)\s*\(", text)))


def test_header_and_library_agree(L):
    declared = declared_functions()
    assert declared == sorted(_lib.EXPORTED)
    for name in declared:
        assert hasattr(L, name), name


def test_config_struct_layout():
    # int32 x 6, uint32 x 2, uint64, int32 x 3 -> 52 bytes of fields, padded to 56 (the uint64's
    # alignment), rng_seed at offset 32, swizzle_scales at 48
    assert ctypes.sizeof(_lib.Config) == 56
    assert _lib.Config.rng_seed.offset == 32
    assert _lib.Config.swizzle_scales.offset == 48


def test_status_strings(L):
    for code in range(8):
        assert L.nvfp4_status_string(code)


def _cfg(**kw):
    c = _lib.Config(rowwise=1)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _quant(L, M, N, cfg, x=FAKE, outs=FAKE):
    p = ctypes.c_void_p
    return L.nvfp4_quantize(p(x), M, N, ctypes.byref(cfg), None, None, p(outs), p(outs), p(outs),
                            p(outs), p(outs), p(outs), None)


def test_argument_checks_return_before_any_launch(L):
    assert _quant(L, 32, 24, _cfg()) == 2                       # N % 16
    assert _quant(L, 24, 32, _cfg(columnwise=1)) == 2           # M % 16 with columnwise
    assert _quant(L, 24, 32, _cfg(rowwise=1, block2d=1)) == 2   # 2D needs both
    assert _quant(L, 32, 32, _cfg(rowwise=0)) == 4              # nothing selected
    assert _quant(L, 32, 32, _cfg(block2d=1, rht_col=1, columnwise=1)) == 4
    assert _quant(L, 32, 32, _cfg(block2d=1, round_row=1)) == 4
    assert _quant(L, 32, 32, _cfg(round_row=2)) == 1
    assert _quant(L, 32, 32, _cfg(fast_math=2)) == 1
    assert _quant(L, 32, 32, _cfg(rht_sign_mask=1 << 16)) == 1
    assert _quant(L, -1, 32, _cfg()) == 1
    assert _quant(L, 32, 32, _cfg(), x=FAKE + 8) == 3           # misaligned input
    assert _quant(L, 32, 32, _cfg(), outs=FAKE + 4) == 3        # misaligned outputs
    p = ctypes.c_void_p
    assert L.nvfp4_quantize(p(FAKE), 32, 32, ctypes.byref(_cfg()), None, None, None, None, None,
                            None, None, None, None) == 1       # missing rowwise outputs
    assert L.nvfp4_quantize(p(FAKE), 32, 32, None, None, None, p(FAKE), p(FAKE), p(FAKE), None,
                            None, None, None) == 1             # missing config


def test_grouped_and_dequant_argument_checks(L):
    p = ctypes.c_void_p
    cfg = _cfg(columnwise=1)

    def grouped(T, H, offs, E, cap, c=cfg):
        return L.nvfp4_quantize_grouped(p(FAKE), T, H, offs, E, cap, ctypes.byref(c), None, None,
                                        p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), None)
    assert grouped(64, 32, p(FAKE), 0, 64) == 1     # no experts
    assert grouped(64, 32, p(FAKE), 257, 64) == 1   # too many experts
    assert grouped(64, 32, None, 2, 64) == 1        # no offsets
    assert grouped(64, 24, p(FAKE), 2, 64) == 2     # H % 16
    assert grouped(64, 32, p(FAKE), 2, 40) == 2     # capacity % 16
    assert grouped(64, 32, p(FAKE + 2), 2, 64) == 3
    assert L.nvfp4_quantize_grouped(p(FAKE), 64, 32, p(FAKE), 2, 64, ctypes.byref(cfg), None,
                                    p(FAKE + 2), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                                    p(FAKE), None) == 3   # misaligned supplied amax
    # grouped 2D has no RHT or SR, and no grouped call takes the single-launch amax
    assert grouped(64, 32, p(FAKE), 2, 64, _cfg(columnwise=1, block2d=1, rht_col=1)) == 4
    assert grouped(64, 32, p(FAKE), 2, 64, _cfg(columnwise=1, block2d=1, round_col=1)) == 4
    assert grouped(64, 32, p(FAKE), 2, 64, _cfg(columnwise=1, fused_amax=1)) == 4
    assert L.nvfp4_dequantize(p(FAKE), p(FAKE), p(FAKE), 4, 24, p(FAKE), None) == 2
    assert L.nvfp4_dequantize(p(FAKE), p(FAKE), p(FAKE), 4, 32, p(FAKE + 4), None) == 3
    assert L.nvfp4_amax(p(FAKE), 16, 32, ctypes.byref(cfg), None, None, None) == 1
    assert L.nvfp4_get_status(None, None) == 1


def test_host_pipeline_argument_checks_return_before_any_cuda_call(L):
    h = ctypes.c_void_p()
    create = lambda M, N, c, depth: L.nvfp4_host_pipeline_create(M, N, ctypes.byref(c), depth,
                                                                 ctypes.byref(h))
    assert create(64, 64, _cfg(), 0) == 1                       # depth below 1
    assert create(64, 64, _cfg(), 5) == 1                       # depth above 4
    assert create(64, 64, _cfg(fast_math=-1), 2) == 1
    assert create(64, 64, _cfg(rowwise=0), 2) == 4              # nothing selected
    assert create(0, 64, _cfg(), 2) == 2                        # empty
    assert create(64, 24, _cfg(), 2) == 2                       # N % 16
    assert create(24, 64, _cfg(columnwise=1), 2) == 2           # M % 16 with columnwise
    assert L.nvfp4_host_pipeline_create(64, 64, None, 2, ctypes.byref(h)) == 1
    assert L.nvfp4_host_pipeline_submit(None, ctypes.c_void_p(FAKE), *([None] * 7)) == 1
    grouped = lambda T, H, E, cap, c, depth: L.nvfp4_host_pipeline_create_grouped(
        T, H, E, cap, ctypes.byref(c), depth, ctypes.byref(h))
    assert grouped(64, 64, 0, 64, _cfg(), 2) == 1                 # no experts
    assert grouped(64, 64, 257, 64, _cfg(), 2) == 1               # more than 256
    assert grouped(64, 64, 2, 64, _cfg(fused_amax=1), 2) == 4     # no single launch here
    assert grouped(64, 64, 2, 64, _cfg(swizzle_scales=1), 2) == 4
    assert grouped(64, 24, 2, 64, _cfg(), 2) == 2                 # H % 16
    assert grouped(64, 64, 2, 72, _cfg(columnwise=1), 2) == 2     # capacity % 16
    assert grouped(64, 64, 2, 64, _cfg(), 9) == 1                 # depth
    assert L.nvfp4_host_pipeline_submit_grouped(None, ctypes.c_void_p(FAKE),
                                                ctypes.c_void_p(FAKE), *([None] * 7)) == 1
    assert L.nvfp4_host_pipeline_join(None, None) == 1
    assert L.nvfp4_host_pipeline_destroy(None) == 0


def test_swizzle_argument_checks_return_before_any_cuda_call(L):
    p = ctypes.c_void_p
    assert L.nvfp4_swizzle_scales(p(FAKE), -1, 4, p(FAKE), None) == 1
    assert L.nvfp4_swizzle_scales(None, 0, 4, None, None) == 0           # empty: nothing to do
    assert L.nvfp4_swizzle_scales(None, 4, 4, p(FAKE), None) == 1
    assert L.nvfp4_swizzle_scales(p(FAKE), 4, 4, p(FAKE + 8), None) == 3  # misaligned output


def test_mx_argument_checks_return_before_any_cuda_call(L):
    p = ctypes.c_void_p
    q = lambda M, N, fmt=0, row=1, col=0, x=FAKE, out=FAKE: L.nvfp4_mx_quantize(
        p(x), M, N, fmt, row, col, p(out), p(out), p(out), p(out), None)
    assert q(32, 32, fmt=3) == 1 and q(32, 32, fmt=-1) == 1     # no such format
    assert q(-1, 32) == 1
    assert q(32, 32, row=0, col=0) == 4                          # neither orientation
    assert q(32, 48) == 2                                        # rowwise: N % 32
    assert q(48, 32, row=0, col=1) == 2                          # columnwise: M % 32
    assert q(32, 36, row=0, col=1) == 2                          # columnwise: N % 8 (TMA pitch)
    assert q(0, 32) == 0                                         # empty: nothing to do
    assert q(32, 32, x=0) == 1                                   # NULL input
    assert q(32, 32, x=FAKE + 8) == 3                            # input not 16-byte aligned
    assert q(32, 32, out=FAKE + 16) == 3                         # FP8 codes need 32 bytes
    assert L.nvfp4_mx_dequantize(p(FAKE), p(FAKE), 0, 4, 48, p(FAKE), None) == 2   # C % 32
    assert L.nvfp4_mx_dequantize(p(FAKE), p(FAKE), 5, 4, 32, p(FAKE), None) == 1
    assert L.nvfp4_mx_dequantize(None, None, 0, 0, 32, None, None) == 0           # empty
    assert L.nvfp4_mx_dequantize(p(FAKE + 8), p(FAKE), 0, 4, 32, p(FAKE), None) == 3


def test_dequantize_ex_argument_checks_return_before_any_cuda_call(L):
    p = ctypes.c_void_p
    d = lambda R, C, rht=0, mask=0, bf=0, out=FAKE: L.nvfp4_dequantize_ex(
        p(FAKE), p(FAKE), p(FAKE), R, C, rht, mask, bf, p(out), None)
    assert d(4, 24) == 2                                    # C % 16
    assert d(4, 32, rht=2) == 1 and d(4, 32, bf=-1) == 1    # flags are 0 or 1
    assert d(4, 32, mask=0x10000) == 1
    assert d(0, 32) == 0                                    # empty
    assert d(4, 32, out=FAKE + 8) == 3                      # output not 16-byte aligned


def test_rmsnorm_argument_checks_return_before_any_cuda_call(L):
    p = ctypes.c_void_p
    n = lambda M, N, eps=1e-6, bias=0.0, x=FAKE, amax=FAKE: L.nvfp4_rmsnorm_amax(
        p(x), p(FAKE), M, N, eps, bias, p(FAKE), p(amax), None)
    assert n(4, 12) == 2                                     # N % 8
    assert n(-1, 16) == 1
    assert n(4, 16, eps=float("nan")) == 1 and n(4, 16, bias=float("inf")) == 1
    assert n(4, 16, amax=0) == 1                             # amax is required
    assert n(4, 16, x=FAKE + 8) == 3                         # input not 16-byte aligned
    cfg = _cfg()
    assert L.nvfp4_rmsnorm_quantize(p(FAKE), p(FAKE), 4, 24, 1e-6, 0.0, ctypes.byref(cfg),
                                    p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), None, None,
                                    None, None) == 2         # N % 16


def test_set_workspace_argument_checks_return_before_any_cuda_call(L):
    p = ctypes.c_void_p
    assert L.nvfp4_set_workspace(p(FAKE), 16383) == 1       # below NVFP4_WORKSPACE_BYTES
    assert L.nvfp4_set_workspace(p(FAKE + 16), 16384) == 3  # not 256-byte aligned


def test_amax_grouped_argument_checks_return_before_any_cuda_call(L):
    p = ctypes.c_void_p
    cfg = _cfg()
    a = lambda T, H, offs, E, ar=FAKE, ac=FAKE: L.nvfp4_amax_grouped(
        p(FAKE), T, H, offs, E, ctypes.byref(cfg), p(ar) if ar else None, p(ac) if ac else None,
        None)
    assert a(64, 32, p(FAKE), 0) == 1 and a(64, 32, p(FAKE), 257) == 1
    assert a(64, 32, None, 2) == 1
    assert a(64, 32, p(FAKE), 2, ar=0, ac=0) == 1           # nothing to write
    assert a(64, 24, p(FAKE), 2) == 2                        # H % 16
    assert a(64, 32, p(FAKE + 2), 2) == 3                    # offsets alignment


def test_debug_hook_argument_checks(L):
    assert L.nvfp4_debug_fused_extra_arrivals(-1) == 1
    assert L.nvfp4_debug_fused_extra_arrivals(1025) == 1
    assert L.nvfp4_debug_fused_extra_arrivals(0) == 0  # clears it: no call consumes it here
    assert L.nvfp4_debug_fail_next_launch(2) == 1 and L.nvfp4_debug_fail_next_launch(-1) == 1
    assert L.nvfp4_debug_fail_next_launch(0) == 0
