"""ctypes loader for libnvfp4.so (the C ABI of include/nvfp4.h).

The library is built in-tree by ``nvfp4_block_scaled_quantize_gb300.build``. Loading fails
loudly when it is missing: there is no other implementation to fall back to.
"""
import ctypes
import os

from . import build as _build

NVFP4_OK = 0
STATUS_NAMES = {
    0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
    4: "NVFP4_ERR_UNSUPPORTED", 5: "NVFP4_ERR_CUDA", 6: "NVFP4_ERR_DEVICE_STATUS",
    7: "NVFP4_ERR_TIMEOUT",
}
ROUND_RN = 0
ROUND_SR = 1
DEVICE_BAD_OFFSETS = 0x1
DEVICE_TIMEOUT = 0x2

EXPORTED = ["nvfp4_status_string", "nvfp4_amax", "nvfp4_quantize", "nvfp4_quantize_grouped",
            "nvfp4_dequantize", "nvfp4_get_status", "nvfp4_quantize_noalloc",
            "nvfp4_host_pipeline_create", "nvfp4_host_pipeline_submit",
            "nvfp4_host_pipeline_create_grouped", "nvfp4_host_pipeline_submit_grouped",
            "nvfp4_host_pipeline_join", "nvfp4_host_pipeline_destroy", "nvfp4_swizzle_scales",
            "nvfp4_mx_quantize", "nvfp4_mx_dequantize", "nvfp4_dequantize_ex",
            "nvfp4_rmsnorm_amax", "nvfp4_rmsnorm_quantize", "nvfp4_set_workspace",
            "nvfp4_amax_grouped", "nvfp4_debug_fused_extra_arrivals",
            "nvfp4_debug_fail_next_launch", "nvfp4_noalloc_get_status",
            "nvfp4_debug_fused_late_ctas", "nvfp4_debug_fused_takeovers"]


class Config(ctypes.Structure):
    """Mirror of ``struct nvfp4_config``."""
    _fields_ = [
        ("rowwise", ctypes.c_int32),
        ("columnwise", ctypes.c_int32),
        ("block2d", ctypes.c_int32),
        ("round_row", ctypes.c_int32),
        ("round_col", ctypes.c_int32),
        ("rht_col", ctypes.c_int32),
        ("rht_sign_mask", ctypes.c_uint32),
        ("rng_offset", ctypes.c_uint32),
        ("rng_seed", ctypes.c_uint64),
        ("fused_amax", ctypes.c_int32),
        ("fast_math", ctypes.c_int32),
        ("swizzle_scales", ctypes.c_int32),
    ]


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().nvfp4_status_string(status).decode()
        super().__init__("%s: %s (%s)" % (where, STATUS_NAMES.get(status, status), msg))


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libnvfp4.so; raises if it has not been built (build() compiles it)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError("libnvfp4.so is not built (%s); run "
                               "`python -m nvfp4_block_scaled_quantize_gb300.build`" % path)
        _build.build()
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    cfgp = ctypes.POINTER(Config)
    L.nvfp4_status_string.restype = ctypes.c_char_p
    L.nvfp4_status_string.argtypes = [ctypes.c_int]
    L.nvfp4_amax.restype = ctypes.c_int
    L.nvfp4_amax.argtypes = [vp, i64, i64, cfgp, vp, vp, vp]
    L.nvfp4_quantize.restype = ctypes.c_int
    L.nvfp4_quantize.argtypes = [vp, i64, i64, cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.nvfp4_quantize_grouped.restype = ctypes.c_int
    L.nvfp4_quantize_grouped.argtypes = [vp, i64, i64, vp, i32, i64, cfgp, vp, vp, vp, vp, vp,
                                         vp, vp, vp, vp]
    L.nvfp4_dequantize.restype = ctypes.c_int
    L.nvfp4_dequantize.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    L.nvfp4_quantize_noalloc.restype = ctypes.c_int
    L.nvfp4_quantize_noalloc.argtypes = [vp, i64, i64, cfgp, vp, vp, vp, vp, vp, vp, vp]
    L.nvfp4_host_pipeline_create.restype = ctypes.c_int
    L.nvfp4_host_pipeline_create.argtypes = [i64, i64, cfgp, i32, ctypes.POINTER(vp)]
    L.nvfp4_host_pipeline_submit.restype = ctypes.c_int
    L.nvfp4_host_pipeline_submit.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.nvfp4_host_pipeline_create_grouped.restype = ctypes.c_int
    L.nvfp4_host_pipeline_create_grouped.argtypes = [i64, i64, i32, i64, cfgp, i32,
                                                     ctypes.POINTER(vp)]
    L.nvfp4_host_pipeline_submit_grouped.restype = ctypes.c_int
    L.nvfp4_host_pipeline_submit_grouped.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.nvfp4_host_pipeline_join.restype = ctypes.c_int
    L.nvfp4_host_pipeline_join.argtypes = [vp, vp]
    L.nvfp4_host_pipeline_destroy.restype = ctypes.c_int
    L.nvfp4_host_pipeline_destroy.argtypes = [vp]
    L.nvfp4_swizzle_scales.restype = ctypes.c_int
    L.nvfp4_swizzle_scales.argtypes = [vp, i64, i64, vp, vp]
    L.nvfp4_mx_quantize.restype = ctypes.c_int
    L.nvfp4_mx_quantize.argtypes = [vp, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp]
    L.nvfp4_mx_dequantize.restype = ctypes.c_int
    L.nvfp4_mx_dequantize.argtypes = [vp, vp, i32, i64, i64, vp, vp]
    L.nvfp4_dequantize_ex.restype = ctypes.c_int
    L.nvfp4_dequantize_ex.argtypes = [vp, vp, vp, i64, i64, i32, ctypes.c_uint32, i32, vp, vp]
    f32 = ctypes.c_float
    L.nvfp4_rmsnorm_amax.restype = ctypes.c_int
    L.nvfp4_rmsnorm_amax.argtypes = [vp, vp, i64, i64, f32, f32, vp, vp, vp]
    L.nvfp4_rmsnorm_quantize.restype = ctypes.c_int
    L.nvfp4_rmsnorm_quantize.argtypes = [vp, vp, i64, i64, f32, f32, cfgp, vp, vp, vp, vp, vp,
                                         vp, vp, vp, vp]
    L.nvfp4_amax_grouped.restype = ctypes.c_int
    L.nvfp4_amax_grouped.argtypes = [vp, i64, i64, vp, i32, cfgp, vp, vp, vp]
    L.nvfp4_set_workspace.restype = ctypes.c_int
    L.nvfp4_set_workspace.argtypes = [vp, ctypes.c_size_t]
    L.nvfp4_get_status.restype = ctypes.c_int
    L.nvfp4_get_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.nvfp4_debug_fused_extra_arrivals.restype = ctypes.c_int
    L.nvfp4_debug_fused_extra_arrivals.argtypes = [i32]
    L.nvfp4_debug_fail_next_launch.restype = ctypes.c_int
    L.nvfp4_debug_fail_next_launch.argtypes = [i32]
    L.nvfp4_noalloc_get_status.restype = ctypes.c_int
    L.nvfp4_noalloc_get_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.nvfp4_debug_fused_late_ctas.restype = ctypes.c_int
    L.nvfp4_debug_fused_late_ctas.argtypes = [i32]
    L.nvfp4_debug_fused_takeovers.restype = ctypes.c_int
    L.nvfp4_debug_fused_takeovers.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    _lib = L
    return L
