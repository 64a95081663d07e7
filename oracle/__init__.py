"""The oracle: a plain CPU statement of NVFP4 block-scaled quantization (numpy in, numpy out).

TEST INFRASTRUCTURE ONLY. The parity tests, the smoke check and the benchmark's CPU-baseline
leg are the only callers. The CUDA library (the product) never imports this package and shares
no code with it; the arithmetic lives in ``nvfp4_oracle.c`` (plain scalar C, IEEE binary32,
each step cited there to the page "[nvfp4_training] Optimize CuteDSL kernels for NVFP4
training", pytorch/ao pull request #4798).

The MX formats (MXFP8 with E4M3 or E5M2 elements, MXFP4 with E2M1 elements; 32-element
blocks, E8M0 power-of-two scales, no tensor scale) follow the same pattern; their readings
(M1-M4 in ``nvfp4_oracle.c``) take the OCP Microscaling Formats v1.0 conversion, which the pages
name but do not spell out.

BF16 tensors are passed as their 16-bit patterns (``numpy.uint16``). Outputs follow the
layouts of the C library: rowwise codes [M, N/2] and scales [M, N/16]; columnwise (transposed)
codes [N, M/2] and scales [N, M/16]; global scales as ``[amax, S_dec]``.

Parity status: every function here is pinned by the ``-m "not gpu"`` oracle tests, except the
rounding rule of stochastic rounding (reading R8 in ``nvfp4_oracle.c``), which is pinned by
its statistical properties there and otherwise rests on the PTX description of ``cvt`` with
``.rs`` rounding.
"""
import ctypes
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_i64 = ctypes.c_int64


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        sig = {
            "oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "oracle_e4m3_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "oracle_e2m1_encode_rn": (ctypes.c_uint8, [ctypes.c_float]),
            "oracle_e2m1_encode_sr": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_uint32]),
            "oracle_e2m1_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "oracle_sr_random16": (ctypes.c_uint32, [ctypes.c_uint32, ctypes.c_int32]),
            "oracle_sr_convert4_n": (None, [_f32p, _u32p, _i64, _u8p]),
            "oracle_e2m1_encode_rn_n": (None, [_f32p, _i64, _u8p]),
            "oracle_philox4x32_10": (None, [_u32p, _u32p, _u32p]),
            "oracle_fwht16": (None, [_f32p]),
            "oracle_rht16": (None, [_f32p, ctypes.c_uint32, _f32p]),
            "oracle_global_scale": (None, [ctypes.c_float, _f32p]),
            "oracle_block_scale": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_float]),
            "oracle_element_multiplier": (ctypes.c_float, [ctypes.c_uint8, ctypes.c_float]),
            "oracle_quantize_block16": (None, [_f32p, ctypes.c_float, ctypes.c_float, _u32p,
                                               _u8p, _u8p]),
            "oracle_amax": (ctypes.c_float, [_u16p, _i64, _i64]),
            "oracle_amax_rht": (ctypes.c_float, [_u16p, _i64, _i64, ctypes.c_uint32]),
            "oracle_quantize_rowwise": (None, [_u16p, _i64, _i64, ctypes.c_float, ctypes.c_int,
                                               ctypes.c_uint64, ctypes.c_uint32, _u8p, _u8p,
                                               _f32p]),
            "oracle_quantize_colwise": (None, [_u16p, _i64, _i64, ctypes.c_float, ctypes.c_int,
                                               ctypes.c_uint32, ctypes.c_int, ctypes.c_uint64,
                                               ctypes.c_uint32, _u8p, _u8p, _f32p]),
            "oracle_quantize_2d": (None, [_u16p, _i64, _i64, ctypes.c_float, _u8p, _u8p, _u8p,
                                          _u8p, _f32p]),
            "oracle_quantize_grouped": (ctypes.c_int, [_u16p, _i64, _i64, _i32p, ctypes.c_int32,
                                                       _i64, ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_uint32,
                                                       ctypes.c_uint64, ctypes.c_uint32,
                                                       _u8p, _u8p, _f32p, _u8p, _u8p, _f32p]),
            "oracle_dequantize": (None, [_u8p, _u8p, ctypes.c_float, _i64, _i64, _f32p]),
            "oracle_quantize_grouped_2d": (ctypes.c_int, [_u16p, _i64, _i64, _i32p,
                                                          ctypes.c_int32, _i64, _u8p, _u8p,
                                                          _f32p, _u8p, _u8p, _f32p]),
            "oracle_inverse_rht16": (None, [_f32p, ctypes.c_uint32, _f32p]),
            "oracle_inverse_rht_rows": (None, [_f32p, _i64, _i64, ctypes.c_uint32]),
            "oracle_f32_to_bf16_n": (None, [_f32p, _i64, _u16p]),
            "oracle_rsqrt_rn": (ctypes.c_float, [ctypes.c_float]),
            "oracle_rmsnorm": (ctypes.c_float, [_u16p, _u16p, _i64, _i64, ctypes.c_float,
                                                ctypes.c_float, _u16p]),
            "oracle_e5m2_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "oracle_e5m2_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "oracle_e8m0_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_mx_scale": (ctypes.c_uint8, [ctypes.c_double, ctypes.c_int32]),
            "oracle_mx_encode": (ctypes.c_uint8, [ctypes.c_double, ctypes.c_int32]),
            "oracle_mx_decode": (ctypes.c_double, [ctypes.c_uint8, ctypes.c_int32]),
            "oracle_mx_quantize_rowwise": (None, [_u16p, _i64, _i64, ctypes.c_int32, _u8p,
                                                  _u8p]),
            "oracle_mx_quantize_colwise": (None, [_u16p, _i64, _i64, ctypes.c_int32, _u8p,
                                                  _u8p]),
            "oracle_mx_dequantize": (None, [_u8p, _u8p, ctypes.c_int32, _i64, _i64, _f32p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a, t):
    return a.ctypes.data_as(t) if a is not None else None


def as_bf16_bits(x) -> np.ndarray:
    """BF16 input as a C-contiguous uint16 array of bit patterns (torch bf16 tensors accepted)."""
    if hasattr(x, "dtype") and str(getattr(x, "dtype", "")) == "torch.bfloat16":
        import torch  # plumbing only: reinterpret the tensor's storage as 16-bit integers
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("expected uint16 BF16 bit patterns or a torch.bfloat16 tensor")
    return a


# ----------------------------------------------------------------------------------------
# Scalar primitives (vectorised over numpy arrays with plain Python loops: small inputs only)
# ----------------------------------------------------------------------------------------

def f32_to_bf16(values) -> np.ndarray:
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib().oracle_f32_to_bf16(float(f)) for f in v], dtype=np.uint16)


def e4m3_encode(values) -> np.ndarray:
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib().oracle_e4m3_encode(float(f)) for f in v], dtype=np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib().oracle_e4m3_decode(int(b)) for b in c], dtype=np.float32)


def e2m1_encode_rn(values) -> np.ndarray:
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib().oracle_e2m1_encode_rn(float(f)) for f in v], dtype=np.uint8)


def e2m1_encode_sr(values, rand16) -> np.ndarray:
    v = np.asarray(values, dtype=np.float32).ravel()
    r = np.broadcast_to(np.asarray(rand16, dtype=np.uint32), v.shape)
    return np.array([lib().oracle_e2m1_encode_sr(float(f), int(b)) for f, b in zip(v, r)],
                    dtype=np.uint8)


def sr_random16(word: int, i: int) -> int:
    return lib().oracle_sr_random16(word, i)


def sr_convert4(values, words) -> np.ndarray:
    """Codes (one per byte) of 4 * len(words) values, element 4k+i rounded stochastically with
    the 16-bit random value that word k gives lane i (reading R8: one
    cvt.rs.satfinite.e2m1x4.f32 per word)."""
    t = np.ascontiguousarray(values, dtype=np.float32).ravel()
    w = np.ascontiguousarray(words, dtype=np.uint32).ravel()
    if t.size != 4 * w.size:
        raise ValueError("need four values per random word")
    out = np.zeros(t.size, dtype=np.uint8)
    lib().oracle_sr_convert4_n(_ptr(t, _f32p), _ptr(w, _u32p), w.size, _ptr(out, _u8p))
    return out


def e2m1_encode_rn_n(values) -> np.ndarray:
    """Round-to-nearest-even codes (one per byte) of an array of binary32 values."""
    t = np.ascontiguousarray(values, dtype=np.float32).ravel()
    out = np.zeros(t.size, dtype=np.uint8)
    lib().oracle_e2m1_encode_rn_n(_ptr(t, _f32p), t.size, _ptr(out, _u8p))
    return out


def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib().oracle_e2m1_decode(int(b)) for b in c], dtype=np.float32)


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c, _u32p), _ptr(k, _u32p), _ptr(out, _u32p))
    return out


def fwht16(v) -> np.ndarray:
    w = np.array(v, dtype=np.float32).copy()
    assert w.shape == (16,)
    lib().oracle_fwht16(_ptr(w, _f32p))
    return w


def rht16(v, sign_mask: int) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.float32)
    y = np.zeros(16, dtype=np.float32)
    lib().oracle_rht16(_ptr(a, _f32p), sign_mask, _ptr(y, _f32p))
    return y


def global_scale(amax: float):
    out = np.zeros(2, dtype=np.float32)
    lib().oracle_global_scale(float(np.float32(amax)), _ptr(out, _f32p))
    return out[0], out[1]


def block_scale(bamax: float, s_enc: float) -> int:
    return lib().oracle_block_scale(float(np.float32(bamax)), float(np.float32(s_enc)))


def element_multiplier(s: int, s_dec: float) -> np.float32:
    return np.float32(lib().oracle_element_multiplier(s, float(np.float32(s_dec))))


def quantize_block16(v, s_enc, s_dec, rand=None):
    a = np.ascontiguousarray(v, dtype=np.float32)
    r = None if rand is None else np.ascontiguousarray(rand, dtype=np.uint32)
    codes = np.zeros(8, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.uint8)
    lib().oracle_quantize_block16(_ptr(a, _f32p), float(np.float32(s_enc)),
                                  float(np.float32(s_dec)), _ptr(r, _u32p),
                                  _ptr(codes, _u8p), _ptr(scale, _u8p))
    return codes, int(scale[0])


# ----------------------------------------------------------------------------------------
# Tensors
# ----------------------------------------------------------------------------------------

def amax(x) -> np.float32:
    xb = as_bf16_bits(x)
    M, N = xb.shape
    return np.float32(lib().oracle_amax(_ptr(xb, _u16p), M, N))


def amax_rht(x, sign_mask: int) -> np.float32:
    xb = as_bf16_bits(x)
    M, N = xb.shape
    assert M % 16 == 0
    return np.float32(lib().oracle_amax_rht(_ptr(xb, _u16p), M, N, sign_mask))


def quantize_rowwise(x, amax_value=None, sr=False, seed=0, offset=0):
    xb = as_bf16_bits(x)
    M, N = xb.shape
    assert N % 16 == 0
    if amax_value is None:
        amax_value = amax(xb)
    codes = np.zeros((M, N // 2), dtype=np.uint8)
    scales = np.zeros((M, N // 16), dtype=np.uint8)
    gs = np.zeros(2, dtype=np.float32)
    lib().oracle_quantize_rowwise(_ptr(xb, _u16p), M, N, float(amax_value), int(bool(sr)),
                                  seed, offset, _ptr(codes, _u8p), _ptr(scales, _u8p),
                                  _ptr(gs, _f32p))
    return codes, scales, gs


def quantize_colwise(x, amax_value=None, rht=False, sign_mask=0, sr=False, seed=0, offset=0):
    xb = as_bf16_bits(x)
    M, N = xb.shape
    assert M % 16 == 0
    if amax_value is None:
        amax_value = amax_rht(xb, sign_mask) if rht else amax(xb)
    codes = np.zeros((N, M // 2), dtype=np.uint8)
    scales = np.zeros((N, M // 16), dtype=np.uint8)
    gs = np.zeros(2, dtype=np.float32)
    lib().oracle_quantize_colwise(_ptr(xb, _u16p), M, N, float(amax_value), int(bool(rht)),
                                  sign_mask, int(bool(sr)), seed, offset, _ptr(codes, _u8p),
                                  _ptr(scales, _u8p), _ptr(gs, _f32p))
    return codes, scales, gs


def quantize_2d(x, amax_value=None):
    xb = as_bf16_bits(x)
    M, N = xb.shape
    assert M % 16 == 0 and N % 16 == 0
    if amax_value is None:
        amax_value = amax(xb)
    rc = np.zeros((M, N // 2), dtype=np.uint8)
    rs = np.zeros((M, N // 16), dtype=np.uint8)
    cc = np.zeros((N, M // 2), dtype=np.uint8)
    cs = np.zeros((N, M // 16), dtype=np.uint8)
    gs = np.zeros(2, dtype=np.float32)
    lib().oracle_quantize_2d(_ptr(xb, _u16p), M, N, float(amax_value), _ptr(rc, _u8p),
                             _ptr(rs, _u8p), _ptr(cc, _u8p), _ptr(cs, _u8p), _ptr(gs, _f32p))
    return rc, rs, cc, cs, gs


def padded_capacity(offsets) -> int:
    """Sum over experts of the token count rounded up to 16 (columnwise output columns)."""
    prev, total = 0, 0
    for o in np.asarray(offsets).tolist():
        total += (o - prev + 15) // 16 * 16
        prev = o
    return total


def quantize_grouped(x, offsets, cap=None, rowwise=True, columnwise=True, round_row_sr=False,
                     round_col_sr=False, rht_col=False, sign_mask=0, seed=0, offset=0,
                     fill=0, block2d=False):
    """Grouped quantization. Output buffers start filled with ``fill`` so that untouched
    regions (the tail past the last offset, columns past the padded total) stay visible."""
    xb = as_bf16_bits(x)
    T, H = xb.shape
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    E = off.shape[0]
    if cap is None:
        cap = padded_capacity(off)
    rc = np.full((T, H // 2), fill, dtype=np.uint8) if rowwise else None
    rs = np.full((T, H // 16), fill, dtype=np.uint8) if rowwise else None
    rg = np.zeros((E, 2), dtype=np.float32) if rowwise else None
    cc = np.full((H, cap // 2), fill, dtype=np.uint8) if columnwise else None
    cs = np.full((H, cap // 16), fill, dtype=np.uint8) if columnwise else None
    cg = np.zeros((E, 2), dtype=np.float32) if columnwise else None
    rc_ = rc if rowwise else None
    if block2d:
        assert not (round_row_sr or round_col_sr or rht_col), "2D has no SR or RHT"
        status = lib().oracle_quantize_grouped_2d(
            _ptr(xb, _u16p), T, H, _ptr(off, _i32p), E, cap, _ptr(rc_, _u8p), _ptr(rs, _u8p),
            _ptr(rg, _f32p), _ptr(cc, _u8p), _ptr(cs, _u8p), _ptr(cg, _f32p))
        if status != 0:
            raise ValueError("invalid offsets or capacity for grouped quantization")
        return rc, rs, rg, cc, cs, cg
    status = lib().oracle_quantize_grouped(
        _ptr(xb, _u16p), T, H, _ptr(off, _i32p), E, cap, int(bool(round_row_sr)),
        int(bool(round_col_sr)), int(bool(rht_col)), sign_mask, seed, offset,
        _ptr(rc_, _u8p), _ptr(rs, _u8p), _ptr(rg, _f32p), _ptr(cc, _u8p), _ptr(cs, _u8p),
        _ptr(cg, _f32p))
    if status != 0:
        raise ValueError("invalid offsets or capacity for grouped quantization")
    return rc, rs, rg, cc, cs, cg


def dequantize(codes, scales, s_dec) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, half = c.shape
    C = 2 * half
    assert s.shape == (R, C // 16)
    out = np.zeros((R, C), dtype=np.float32)
    lib().oracle_dequantize(_ptr(c, _u8p), _ptr(s, _u8p), float(np.float32(s_dec)), R, C,
                            _ptr(out, _f32p))
    return out


def inverse_rht16(y, sign_mask: int) -> np.ndarray:
    """v = d * (0.25 * FWHT16(y)) in binary32 (reading R13)."""
    a = np.ascontiguousarray(y, dtype=np.float32)
    v = np.zeros(16, dtype=np.float32)
    lib().oracle_inverse_rht16(_ptr(a, _f32p), sign_mask, _ptr(v, _f32p))
    return v


def f32_to_bf16_array(values) -> np.ndarray:
    """binary32 -> BF16 bit patterns (uint16), round to nearest-even, any shape."""
    a = np.ascontiguousarray(values, dtype=np.float32)
    out = np.zeros(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_n(_ptr(a, _f32p), a.size, _ptr(out, _u16p))
    return out


def dequantize_ex(codes, scales, s_dec, inverse_rht=False, sign_mask=0, bf16=False):
    """dequantize(), then optionally the inverse RHT of every 16-element block of every row
    (columnwise RHT outputs) and optionally BF16 rounding (bit patterns as uint16)."""
    out = dequantize(codes, scales, s_dec)
    if inverse_rht:
        R, C = out.shape
        lib().oracle_inverse_rht_rows(_ptr(out, _f32p), R, C, sign_mask)
    return f32_to_bf16_array(out) if bf16 else out


def rsqrt_rn(a: float) -> np.float32:
    """1/sqrt(a) correctly rounded to binary32."""
    return np.float32(lib().oracle_rsqrt_rn(float(np.float32(a))))


def rmsnorm(x, w, eps: float, bias: float = 0.0):
    """RMSNorm producer (reading R14): (y as BF16 bit patterns [M, N], amax of y)."""
    xb = as_bf16_bits(x)
    wb = as_bf16_bits(w).reshape(-1)
    M, N = xb.shape
    assert wb.shape == (N,) and N % 8 == 0
    y = np.zeros((M, N), dtype=np.uint16)
    amax = lib().oracle_rmsnorm(_ptr(xb, _u16p), _ptr(np.ascontiguousarray(wb), _u16p), M, N,
                                float(np.float32(eps)), float(np.float32(bias)), _ptr(y, _u16p))
    return y, np.float32(amax)


def swizzle_scales(scales) -> np.ndarray:
    """E4M3 scale bytes [R, C] (row-major, as the quantize calls write them) rearranged into the
    128 x 4 tiled layout that the tensor-core block-scaled GEMMs read ([PR4798] "Config surface
    and AUTO": its columnwise scale store is hardwired to this swizzled layout; the layout is
    the 1D block-scaling-factor layout of the cuBLAS documentation). The matrix is padded with
    zeros to a multiple of 128 rows and 4 columns and cut into 128 x 4 tiles, stored one after
    another in row-major tile order, 512 bytes each; inside a tile the scale of row r, column c
    sits at byte (r mod 32) * 16 + ((r mod 128) div 32) * 4 + (c mod 4). Returns the flat byte
    array."""
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = s.shape
    tiles_c = (C + 3) // 4
    out = np.zeros(((R + 127) // 128) * tiles_c * 512, dtype=np.uint8)
    for r in range(R):
        for c in range(C):
            tile = (r // 128) * tiles_c + c // 4
            out[tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4] = s[r, c]
    return out


@dataclass
class Config:
    """The quantizer's options, named as in the C library's configuration."""
    rowwise: bool = True
    columnwise: bool = False
    block2d: bool = False
    round_row_sr: bool = False
    round_col_sr: bool = False
    rht_col: bool = False
    sign_mask: int = 0
    seed: int = 0
    offset: int = 0


def quantize(x, cfg: Config):
    """All outputs one configuration produces, as a dict (the oracle's counterpart of one
    library call with the amax computed inside)."""
    xb = as_bf16_bits(x)
    out = {}
    if cfg.block2d:
        rc, rs, cc, cs, gs = quantize_2d(xb)
        out.update(row_codes=rc, row_scales=rs, row_gscale=gs)
        if cfg.columnwise:
            out.update(col_codes=cc, col_scales=cs, col_gscale=gs.copy())
        if not cfg.rowwise:
            for k in ("row_codes", "row_scales", "row_gscale"):
                del out[k]
        return out
    if cfg.rowwise:
        rc, rs, gs = quantize_rowwise(xb, sr=cfg.round_row_sr, seed=cfg.seed, offset=cfg.offset)
        out.update(row_codes=rc, row_scales=rs, row_gscale=gs)
    if cfg.columnwise:
        cc, cs, gs = quantize_colwise(xb, rht=cfg.rht_col, sign_mask=cfg.sign_mask,
                                      sr=cfg.round_col_sr, seed=cfg.seed, offset=cfg.offset)
        out.update(col_codes=cc, col_scales=cs, col_gscale=gs)
    return out



# ----------------------------------------------------------------------------------------
# MX formats (readings M1-M4 in nvfp4_oracle.c)
# ----------------------------------------------------------------------------------------

MX_FORMATS = {"e4m3": 0, "e5m2": 1, "e2m1": 2}


def mx_format(fmt) -> int:
    return MX_FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def e5m2_encode(values) -> np.ndarray:
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib().oracle_e5m2_encode(float(f)) for f in v], dtype=np.uint8)


def e5m2_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib().oracle_e5m2_decode(int(b)) for b in c], dtype=np.float32)


def e8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib().oracle_e8m0_decode(int(b)) for b in c], dtype=np.float64)


def mx_scale(amax: float, fmt) -> int:
    """E8M0 code of a 32-element block whose largest magnitude is amax (reading M1)."""
    return lib().oracle_mx_scale(float(amax), mx_format(fmt))


def mx_encode(values, fmt) -> np.ndarray:
    """Element codes of already scaled values t = v / X (reading M2)."""
    f = mx_format(fmt)
    v = np.asarray(values, dtype=np.float64).ravel()
    return np.array([lib().oracle_mx_encode(float(t), f) for t in v], dtype=np.uint8)


def mx_decode(codes, fmt) -> np.ndarray:
    f = mx_format(fmt)
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib().oracle_mx_decode(int(b), f) for b in c], dtype=np.float64)


def _mx_outputs(rows, cols, fmt):
    f = mx_format(fmt)
    codes = np.zeros((rows, cols // 2 if f == 2 else cols), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    return f, codes, scales


def mx_quantize_rowwise(x, fmt):
    """Rowwise MX codes [M, N] (FP8) or [M, N/2] (FP4) and E8M0 scales [M, N/32]."""
    xb = as_bf16_bits(x)
    M, N = xb.shape
    assert N % 32 == 0
    f, codes, scales = _mx_outputs(M, N, fmt)
    lib().oracle_mx_quantize_rowwise(_ptr(xb, _u16p), M, N, f, _ptr(codes, _u8p),
                                     _ptr(scales, _u8p))
    return codes, scales


def mx_quantize_colwise(x, fmt):
    """Columnwise MX codes [N, M] (FP8) or [N, M/2] (FP4) and E8M0 scales [N, M/32]."""
    xb = as_bf16_bits(x)
    M, N = xb.shape
    assert M % 32 == 0
    f, codes, scales = _mx_outputs(N, M, fmt)
    lib().oracle_mx_quantize_colwise(_ptr(xb, _u16p), M, N, f, _ptr(codes, _u8p),
                                     _ptr(scales, _u8p))
    return codes, scales


def mx_dequantize(codes, scales, fmt) -> np.ndarray:
    """FP32 [R, C] values of MX codes and E8M0 scales [R, C/32]."""
    f = mx_format(fmt)
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R = c.shape[0]
    C = c.shape[1] * (2 if f == 2 else 1)
    assert s.shape == (R, C // 32)
    out = np.zeros((R, C), dtype=np.float32)
    lib().oracle_mx_dequantize(_ptr(c, _u8p), _ptr(s, _u8p), f, R, C, _ptr(out, _f32p))
    return out
