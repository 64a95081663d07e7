"""Pins for the oracle: each test checks it against something other than itself -- a format
specification table, a library routine (torch casts, cuRAND, numpy), a closed form, an
invariant, or brute force on small inputs. CPU only.

Pages cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
request #4798), by section.
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def _bf16_to_f32(bits_u16):
    return (np.asarray(bits_u16, dtype=np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------------------------------
# E2M1
# ------------------------------------------------------------------------------------------

def test_e2m1_grid_table_round_trips():
    """Every code decodes to the specification's value and encodes back to itself."""
    for code, value in _rows("e2m1_grid.txt"):
        code, value = int(code), float(value)
        dec = oracle.e2m1_decode([code])[0]
        assert dec == value and np.signbit(dec) == np.signbit(value)
        assert oracle.e2m1_encode_rn([dec])[0] == code


def test_e2m1_grid_times_every_e4m3_scale_dequantizes_exactly():
    """grid value * any positive E4M3 scale is exact in binary32 (2 + 4 significant bits)."""
    scales = oracle.e4m3_decode(np.arange(1, 0x7F))
    for s in scales:
        for g in GRID:
            assert np.float32(g) * np.float32(s) == g * float(s)


def test_e2m1_rtne_tie_table():
    for value, code in _rows("e2m1_rtne_ties.txt"):
        assert oracle.e2m1_encode_rn([float(value)])[0] == int(code), value


def _e2m1_argmin(t):
    """Brute force: nearest grid magnitude, ties to the even code; saturate at 6."""
    a = np.abs(t.astype(np.float64))
    d = np.abs(a[:, None] - GRID[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    code = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    code = np.where(a >= 6.0, 7, code)
    return (code | np.where(np.signbit(t), 8, 0)).astype(np.uint8)


def test_e2m1_rn_matches_brute_force_on_dense_values():
    rng = np.random.Generator(np.random.PCG64(11))
    t = np.concatenate([
        np.linspace(-7, 7, 20001, dtype=np.float32),
        rng.uniform(-8, 8, 5000).astype(np.float32),
        # one ulp either side of every midpoint
        np.nextafter(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), np.float32(0)),
        np.nextafter(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), np.float32(9)),
        np.float32([1e-30, -1e-30, 0.0, -0.0, 6.0, 6.5, 1e38, -1e38]),
    ])
    got = oracle.e2m1_encode_rn(t)
    np.testing.assert_array_equal(got, _e2m1_argmin(t))


# ------------------------------------------------------------------------------------------
# E4M3 against torch.float8_e4m3fn (a library routine) after clamping to the finite range
# ------------------------------------------------------------------------------------------

def _torch_e4m3(values):
    v = torch.tensor(np.clip(values, -448.0, 448.0), dtype=torch.float32)
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.e4m3_decode(codes), ref)


def test_e4m3_encode_matches_torch_on_midpoints_and_random_values():
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)  # exact in binary32
    rng = np.random.Generator(np.random.PCG64(12))
    rand = np.exp2(rng.uniform(-14, 10, 20000)).astype(np.float32)
    vals = np.concatenate([
        mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
        pos.astype(np.float32), rand, np.float32([448.0, 449.0, 464.0, 480.0, 1e30, 0.0]),
    ])
    vals = np.concatenate([vals, -vals])
    got = oracle.e4m3_encode(vals)
    np.testing.assert_array_equal(got, _torch_e4m3(vals))


# ------------------------------------------------------------------------------------------
# BF16 round-to-nearest-even against torch's cast
# ------------------------------------------------------------------------------------------

def test_bf16_rne_matches_torch_including_ties():
    rng = np.random.Generator(np.random.PCG64(13))
    bits = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]
    ties = (bits & 0xFFFF0000) | 0x8000
    vals = _f32(np.concatenate([bits, ties]))
    got = oracle.f32_to_bf16(vals)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------------------------------
# Philox4x32-10
# ------------------------------------------------------------------------------------------

def test_philox_known_answer_vectors():
    for row in _rows("philox4x32_10_kat.txt"):
        w = [int(h, 16) for h in row]
        np.testing.assert_array_equal(oracle.philox4x32_10(w[0:4], w[4:6]),
                                      np.array(w[6:10], dtype=np.uint32))


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if path:
            try:
                return ctypes.CDLL(path)
            except OSError:
                pass
    return None


def test_philox_matches_curand_host_generator():
    """cuRAND's host Philox4_32_10 generator with seed s and stream offset o emits, for output
    block i, Philox(key=(lo32 s, hi32 s), counter=(0, 0, j, 0)) with j = o/4 + i (checked for
    j < 2^16; the known-answer vectors cover the other counter words)."""
    cr = _curand()
    if cr is None:
        pytest.skip("libcurand not available")
    for seed, offset in [(0, 0), (0x0123456789ABCDEF, 0), (7, 4 * 1000), (99, 4 * 65000)]:
        gen = ctypes.c_void_p()
        assert cr.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0
        try:
            assert cr.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert cr.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
            n = 64
            buf = np.zeros(n, dtype=np.uint32)
            assert cr.curandGenerate(gen, buf.ctypes.data_as(ctypes.c_void_p),
                                     ctypes.c_size_t(n)) == 0
        finally:
            cr.curandDestroyGenerator(gen)
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i in range(n // 4):
            j = offset // 4 + i
            ctr = [0, 0, j, 0]
            np.testing.assert_array_equal(oracle.philox4x32_10(ctr, key), buf[4 * i:4 * i + 4])


def test_philox_words_look_uniform():
    """Chi-square over the 256 byte values of 4096 blocks' words."""
    words = np.concatenate([oracle.philox4x32_10([b, 0, 1, 0], [5, 0]) for b in range(4096)])
    by = words.view(np.uint8)
    counts = np.bincount(by, minlength=256)
    expected = by.size / 256
    chi2 = ((counts - expected) ** 2 / expected).sum()
    assert chi2 < 350  # 255 dof: p ~ 1e-4 at 350


# ------------------------------------------------------------------------------------------
# Hadamard transform
# ------------------------------------------------------------------------------------------

def _sylvester16():
    H = np.array([[1.0]])
    for _ in range(4):
        H = np.block([[H, H], [H, -H]])
    return H


def test_fwht_matrix_is_sylvester_and_orthogonal():
    cols = [oracle.fwht16(np.eye(16, dtype=np.float32)[i]) for i in range(16)]
    Hf = np.stack(cols, axis=1).astype(np.float64)
    np.testing.assert_array_equal(Hf, _sylvester16())
    np.testing.assert_array_equal(Hf @ Hf.T, 16 * np.eye(16))


def test_fwht_equals_dense_product_on_exact_inputs():
    rng = np.random.Generator(np.random.PCG64(14))
    H = _sylvester16()
    for _ in range(200):
        v = rng.integers(-1000, 1000, 16).astype(np.float32)
        np.testing.assert_array_equal(oracle.fwht16(v).astype(np.float64), H @ v)


def test_rht_is_bf16_of_quarter_hadamard_of_signed_input():
    rng = np.random.Generator(np.random.PCG64(15))
    H = _sylvester16()
    for _ in range(200):
        v = (rng.integers(-2000, 2000, 16) / 64.0).astype(np.float32)  # exact sums in binary32
        mask = int(rng.integers(0, 1 << 16))
        d = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
        exact = (0.25 * (H @ (d * v))).astype(np.float32)
        ref = torch.from_numpy(exact).to(torch.bfloat16).to(torch.float32).numpy()
        np.testing.assert_array_equal(oracle.rht16(v, mask), ref)


def test_rht_applied_twice_is_identity_and_preserves_norm():
    rng = np.random.Generator(np.random.PCG64(16))
    H = _sylvester16() / 4.0
    for _ in range(50):
        v = rng.integers(-8, 8, 16).astype(np.float32)
        y = oracle.rht16(v, 0).astype(np.float64)
        np.testing.assert_array_equal(y, H @ v)  # small integers: no rounding anywhere
        np.testing.assert_array_equal(H @ y, v)
        assert np.isclose(np.linalg.norm(y), np.linalg.norm(v))


# ------------------------------------------------------------------------------------------
# Global and block scales
# ------------------------------------------------------------------------------------------

def test_global_scale_closed_forms():
    assert oracle.global_scale(0.0) == (1.0, 1.0)
    for k in range(-20, 20):
        amax = np.float32(2688.0 * 2.0 ** -k)
        s_enc, s_dec = oracle.global_scale(amax)
        assert s_enc == np.float32(2.0 ** k) and s_dec == np.float32(2.0 ** -k)
    rng = np.random.Generator(np.random.PCG64(17))
    for amax in np.exp2(rng.uniform(-60, 60, 2000)).astype(np.float32):
        s_enc, s_dec = oracle.global_scale(amax)
        assert s_enc == np.float32(np.float32(2688.0) / amax)
        # S_dec * 2688 recovers amax within two rounding errors
        rel = abs(float(s_dec) * 2688.0 - float(amax)) / float(amax)
        assert rel < 2 ** -22
    tiny = _bf16_to_f32([1])[0]  # smallest BF16 subnormal: 2688/amax overflows
    assert oracle.global_scale(tiny)[0] == np.finfo(np.float32).max


def test_block_scale_bounds_and_block_max_maps_to_six():
    """In the normal E4M3 range, the block maximum encodes to +-6 (the E4M3 relative rounding
    error <= 2^-4 keeps bamax * r within [5.65, 6.4]); s <= 448 always."""
    rng = np.random.Generator(np.random.PCG64(18))
    for _ in range(500):
        amax = np.float32(np.exp2(rng.uniform(-10, 10)))
        s_enc, s_dec = oracle.global_scale(amax)
        bamax = np.float32(amax * rng.uniform(2 ** -8, 1.0))
        s = oracle.block_scale(bamax, s_enc)
        assert s <= 0x7E
        r = oracle.element_multiplier(s, s_dec)
        t = np.float32(bamax * r)
        assert 5.6 <= t <= 6.45
        assert oracle.e2m1_encode_rn([t])[0] == 7


def test_element_multiplier_zero_scale_and_reciprocal():
    assert oracle.element_multiplier(0, 1.0) == 0.0
    for s in range(1, 0x7F):
        for s_dec in (1.0, 2.0 ** -8, 1.0 / 3.0):
            p = np.float32(oracle.e4m3_decode([s])[0] * np.float32(s_dec))
            assert oracle.element_multiplier(s, s_dec) == np.float32(np.float32(1.0) / p)


# ------------------------------------------------------------------------------------------
# Blocks and tensors
# ------------------------------------------------------------------------------------------

def test_grid_valued_blocks_round_trip_exactly():
    """amax = 10.5 gives S_enc = 256, S_dec = 2^-8 (exact); a block whose maximum is 6 * 2^e
    and whose values are grid * 2^e quantizes and dequantizes without error."""
    rng = np.random.Generator(np.random.PCG64(19))
    for e in range(-3, 1):
        blocks = []
        for _ in range(32):
            g = rng.choice(GRID, 16) * rng.choice([-1.0, 1.0], 16)
            g[rng.integers(16)] = 6.0
            blocks.append(g * 2.0 ** e)
        x = np.array(blocks, dtype=np.float32).reshape(16, 32)  # [16 rows, 2 blocks/row]
        xb = workloads.to_bf16(x).view(torch.int16).numpy().view(np.uint16)
        codes, scales, gs = oracle.quantize_rowwise(xb, amax_value=10.5)
        assert gs[1] == np.float32(2 ** -8)
        np.testing.assert_array_equal(oracle.dequantize(codes, scales, gs[1]), x)


def test_rowwise_codes_on_every_bf16_pattern_match_brute_force():
    """All finite BF16 patterns laid out as a [2040, 16] tensor: each code is the brute-force
    nearest grid point of t = v * r, and each element is within half a grid step."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]
    bits = bits[: (bits.size // 16) * 16].reshape(-1, 16)
    codes, scales, gs = oracle.quantize_rowwise(bits)
    v = _bf16_to_f32(bits)
    s_enc, s_dec = oracle.global_scale(gs[0])
    assert gs[0] == np.abs(v).max()
    r = np.array([oracle.element_multiplier(int(s), s_dec) for s in scales[:, 0]],
                 dtype=np.float32)
    t = (v * r[:, None]).astype(np.float32)
    expect = _e2m1_argmin(t.ravel()).reshape(t.shape)
    got = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(t.shape)
    np.testing.assert_array_equal(got, expect)


def _sqnr_db(x, xh):
    return 10 * np.log10(np.sum(x.astype(np.float64) ** 2) / np.sum((x - xh).astype(np.float64) ** 2))


def test_rowwise_error_bound_and_sqnr_on_gaussian():
    """RTNE: every element within half a grid step of its dequantized value (plus binary32
    rounding slack); SQNR near NVFP4's ~20 dB ([PR4798] "Fast math")."""
    x = workloads.normal(256, 512, 1.0, 1)
    xb = oracle.as_bf16_bits(x)
    v = _bf16_to_f32(xb)
    codes, scales, gs = oracle.quantize_rowwise(xb)
    xh = oracle.dequantize(codes, scales, gs[1])
    s = oracle.e4m3_decode(scales.ravel()).reshape(scales.shape).repeat(16, axis=1)
    unit = s * gs[1]                        # value of one E2M1 unit in this block
    a = np.abs(v) / unit
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0)) * unit
    sat = np.abs(v) / unit >= 6.0
    err = np.abs(v - xh)
    assert np.all(err[~sat] <= half_step[~sat] * (1 + 2 ** -20) + 1e-30)
    assert 18.5 < _sqnr_db(v, xh) < 21.5


def test_colwise_equals_rowwise_of_transpose():
    x = oracle.as_bf16_bits(workloads.normal(64, 48, 1.0, 21))
    cc, cs, cg = oracle.quantize_colwise(x)
    rc, rs, rg = oracle.quantize_rowwise(np.ascontiguousarray(x.T))
    np.testing.assert_array_equal(cc, rc)
    np.testing.assert_array_equal(cs, rs)
    np.testing.assert_array_equal(cg, rg)


def test_colwise_rht_equals_rowwise_of_transformed_transpose():
    """RHT columnwise == rowwise quantization of the explicitly transformed tensor (built with a
    dense numpy Hadamard and torch's BF16 cast) under the same amax."""
    rng = np.random.Generator(np.random.PCG64(22))
    M, N = 64, 32
    x = (rng.integers(-256, 256, (M, N)) / 64.0).astype(np.float32)  # exact in BF16 and FP32 sums
    xb = oracle.as_bf16_bits(workloads.to_bf16(x))
    mask = 0xA5C3
    d = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    H = _sylvester16()
    y = np.zeros((N, M), dtype=np.float32)
    for rb in range(M // 16):
        blk = x[16 * rb:16 * rb + 16, :].astype(np.float64)          # [16, N]
        y[:, 16 * rb:16 * rb + 16] = (0.25 * (H @ (d[:, None] * blk))).T
    yb = oracle.as_bf16_bits(workloads.to_bf16(y))
    amax_c = oracle.amax_rht(xb, mask)
    assert amax_c == np.abs(_bf16_to_f32(yb)).max()
    cc, cs, cg = oracle.quantize_colwise(xb, rht=True, sign_mask=mask)
    rc, rs, rg = oracle.quantize_rowwise(yb, amax_value=amax_c)

    def nibbles_unsigned_zero(c):
        n = np.stack([c & 0xF, c >> 4], -1)
        return np.where((n & 7) == 0, 0, n)  # a dense matmul and the butterflies may give
                                             # opposite signs to an exact zero
    np.testing.assert_array_equal(nibbles_unsigned_zero(cc), nibbles_unsigned_zero(rc))
    np.testing.assert_array_equal(cs, rs)


def test_2d_codes_transpose_and_tile_scale():
    x = oracle.as_bf16_bits(workloads.normal(64, 96, 0.02, 23))
    rc, rs, cc, cs, gs = oracle.quantize_2d(x)
    v = _bf16_to_f32(x)
    s_enc, _ = oracle.global_scale(gs[0])
    # columnwise codes are the rowwise codes transposed (same tile scale, no transform)
    rn = np.stack([rc & 0xF, rc >> 4], -1).reshape(64, 96)
    cn = np.stack([cc & 0xF, cc >> 4], -1).reshape(96, 64)
    np.testing.assert_array_equal(rn.T, cn)
    for tr in range(4):
        for tc in range(6):
            tile = v[16 * tr:16 * tr + 16, 16 * tc:16 * tc + 16]
            s = oracle.block_scale(np.abs(tile).max(), s_enc)
            assert np.all(rs[16 * tr:16 * tr + 16, tc] == s)
            assert np.all(cs[16 * tc:16 * tc + 16, tr] == s)


# ------------------------------------------------------------------------------------------
# Stochastic rounding (reading R8) -- properties from [PR4798] "Correctness"
# ------------------------------------------------------------------------------------------

def test_sr_grid_values_are_fixed_points():
    rng = np.random.Generator(np.random.PCG64(30))
    u = np.concatenate([[0, 1, 0x8000, 0xFFFF], rng.integers(0, 1 << 16, 252)])
    for g in GRID:
        for sgn in (1.0, -1.0):
            codes = oracle.e2m1_encode_sr(np.full(u.size, sgn * g, np.float32), u)
            assert np.all(codes == oracle.e2m1_encode_rn([sgn * g])[0])


def test_sr_mean_over_all_random_values_is_the_truncated_value():
    """Averaging over all 2^16 random values: E[q] = lo + step * floor(2^16 f) / 2^16, so the
    bias is below step / 2^16 and exactly zero at halfway values (a 50/50 split)."""
    rng = np.random.Generator(np.random.PCG64(24))
    vals = np.concatenate([rng.uniform(0, 6, 6), [0.25, 1.75, 5.0, 4.00390625]]).astype(np.float32)
    u = np.arange(1 << 16)
    for t in vals:
        codes = oracle.e2m1_encode_sr(np.full(u.size, t, np.float32), u)
        mean = oracle.e2m1_decode(codes).astype(np.float64).mean()
        step = 0.5 if t < 2 else (1.0 if t < 4 else 2.0)
        lo = np.floor(t / step) * step
        expect = lo + step * np.floor((t - lo) / step * 65536) / 65536
        assert mean == pytest.approx(expect, abs=1e-12)
        assert abs(mean - t) < step / 65536 + 1e-12


def test_sr_random_values_of_a_word_are_uniform_per_element():
    """Each element's 16-bit value is a bijection of 16 bits of the word: over words covering
    those bits it takes every value once."""
    rng = np.random.Generator(np.random.PCG64(31))
    for i in range(4):
        base = int(rng.integers(0, 1 << 32))
        keep = 0xFF00FF00 if i >= 2 else 0x00FF00FF
        seen = set()
        for v in range(1 << 16):
            spread = (v & 0xFF) << (8 if i >= 2 else 0) | (v >> 8) << (24 if i >= 2 else 16)
            w = (base & ~keep & 0xFFFFFFFF) | spread
            seen.add(oracle.sr_random16(w, i))
        assert len(seen) == 1 << 16


def test_sr_at_most_one_step_from_rtne_with_same_sign():
    rng = np.random.Generator(np.random.PCG64(25))
    t = rng.uniform(-7, 7, 4000).astype(np.float32)
    r16 = rng.integers(0, 1 << 16, t.size)
    sr = oracle.e2m1_encode_sr(t, r16)
    rn = oracle.e2m1_encode_rn(t)
    assert np.all((sr & 8) == (rn & 8))
    assert np.all(np.abs((sr & 7).astype(int) - (rn & 7).astype(int)) <= 1)


def test_sr_unbiased_over_seeds_and_reconstructs():
    """Halfway values averaged over many Philox seeds converge with a ~50/50 split; SR
    reconstruction SQNR is above the pages' 15 dB bar."""
    row = np.array([1.25, 1.75, 2.5, 3.5, 5.0, 0.75, 0.25, 6.0] * 2, dtype=np.float32)
    x = np.tile(row, (16, 1))
    x[:, 7] = 6.0
    xb = oracle.as_bf16_bits(workloads.to_bf16(x))
    acc = np.zeros(x.shape)
    ups = 0
    n_seeds = 300
    for seed in range(n_seeds):
        codes, scales, gs = oracle.quantize_rowwise(xb, amax_value=10.5, sr=True, seed=seed)
        acc += oracle.dequantize(codes, scales, gs[1])
        ups += np.count_nonzero(np.abs(oracle.dequantize(codes, scales, gs[1]))[:, 0] > 1.25)
    mean = acc.mean(axis=0) / n_seeds          # 16 rows x 300 seeds per column
    assert np.allclose(mean, x[0], atol=0.06)   # 4 sigma for the widest step (2)
    assert 0.42 < ups / (16 * n_seeds) < 0.58
    g = oracle.as_bf16_bits(workloads.normal(128, 256, 1.0, 26))
    codes, scales, gs = oracle.quantize_rowwise(g, sr=True, seed=3)
    v = _bf16_to_f32(g)
    assert _sqnr_db(v, oracle.dequantize(codes, scales, gs[1])) > 15.0


def test_sr_seed_and_offset_control_the_stream():
    x = oracle.as_bf16_bits(workloads.normal(32, 64, 1.0, 27))
    a = oracle.quantize_rowwise(x, sr=True, seed=5, offset=0)[0]
    b = oracle.quantize_rowwise(x, sr=True, seed=5, offset=0)[0]
    c = oracle.quantize_rowwise(x, sr=True, seed=5, offset=1)[0]
    d = oracle.quantize_rowwise(x, sr=True, seed=6, offset=0)[0]
    np.testing.assert_array_equal(a, b)
    assert np.count_nonzero(a != c) > 100 and np.count_nonzero(a != d) > 100


# ------------------------------------------------------------------------------------------
# Grouped
# ------------------------------------------------------------------------------------------

def test_grouped_equals_per_expert_calls_and_leaves_tail_untouched():
    T, H = 100, 48
    x = oracle.as_bf16_bits(workloads.normal(T, H, 1.0, 28))
    offsets = np.array([5, 5, 37, 37, 70, 90], dtype=np.int32)  # zero experts; tail 90..99
    mask = 0x3C5A
    cap = oracle.padded_capacity(offsets) + 32
    rc, rs, rg, cc, cs, cg = oracle.quantize_grouped(x, offsets, cap=cap, rht_col=True,
                                                     sign_mask=mask, fill=0xEE)
    assert np.all(rc[90:] == 0xEE) and np.all(rs[90:] == 0xEE)
    col = 0
    prev = 0
    for e, end in enumerate(offsets.tolist()):
        n = end - prev
        sl = x[prev:end]
        amax_e = oracle.amax(sl) if n else np.float32(0)
        assert rg[e, 0] == amax_e
        if n:
            r_codes, r_scales, r_gs = oracle.quantize_rowwise(sl, amax_value=amax_e)
            np.testing.assert_array_equal(rc[prev:end], r_codes)
            np.testing.assert_array_equal(rs[prev:end], r_scales)
            P = (n + 15) // 16 * 16
            padded = np.zeros((P, H), dtype=np.uint16)
            padded[:n] = sl
            c_codes, c_scales, c_gs = oracle.quantize_colwise(padded, rht=True, sign_mask=mask)
            np.testing.assert_array_equal(cc[:, col // 2:(col + P) // 2], c_codes)
            np.testing.assert_array_equal(cs[:, col // 16:(col + P) // 16], c_scales)
            np.testing.assert_array_equal(cg[e], c_gs)
            col += P
        else:
            np.testing.assert_array_equal(rg[e], [0.0, 1.0])
            np.testing.assert_array_equal(cg[e], [0.0, 1.0])
        prev = end
    assert np.all(cc[:, col // 2:] == 0xEE) and np.all(cs[:, col // 16:] == 0xEE)


def test_grouped_rejects_bad_offsets():
    x = oracle.as_bf16_bits(workloads.normal(32, 16, 1.0, 29))
    with pytest.raises(ValueError):
        oracle.quantize_grouped(x, np.array([10, 5], dtype=np.int32))
    with pytest.raises(ValueError):
        oracle.quantize_grouped(x, np.array([10, 40], dtype=np.int32))
    with pytest.raises(ValueError):
        oracle.quantize_grouped(x, np.array([10, 30], dtype=np.int32), cap=32)


def test_swizzled_scales_are_a_permutation_padded_with_zeros():
    """The 128 x 4 tiled layout moves every scale byte exactly once and fills the padding with
    zeros: with all scales distinct and nonzero, each appears once in the output and every
    other byte is zero. (Whether it is the layout the block-scaled GEMM reads is pinned on the
    GPU by running cuBLASLt's NVFP4 GEMM on it.)"""
    rng = np.random.Generator(np.random.PCG64(71))
    for R, C in ((128, 1), (33, 3), (60, 4), (130, 1), (16, 15), (1, 5)):
        s = rng.permutation(np.arange(1, R * C + 1)).astype(np.uint8).reshape(R, C)
        out = oracle.swizzle_scales(s)
        Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
        assert out.shape == (Rp * Cp,)
        nz = out[out != 0]
        assert len(nz) == R * C
        assert np.array_equal(np.sort(nz), np.arange(1, R * C + 1, dtype=np.uint8))


# ------------------------------------------------------------------------------------------
# Verification at the GEMM boundary: inverse RHT and BF16 dequantization (reading R13)
# ------------------------------------------------------------------------------------------

def _sylvester16():
    h = np.array([[1.0]])
    for _ in range(4):
        h = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), h)
    return h


def test_inverse_rht_equals_dense_product_on_exact_inputs():
    H = _sylvester16()
    rng = np.random.default_rng(41)
    for mask in (0x0000, 0xFFFF, 0x1234, 0xB3C5):
        d = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
        y = rng.integers(-64, 65, size=16).astype(np.float64)
        want = d * (0.25 * (H @ y))        # small integers: every binary32 step is exact
        assert np.array_equal(oracle.inverse_rht16(y, mask).astype(np.float64), want), mask


def test_inverse_rht_undoes_the_rht_when_its_bf16_rounding_is_exact():
    rng = np.random.default_rng(42)
    for mask in (0x0F0F, 0x5A3C, 0xFFFF):
        v = rng.integers(-7, 8, size=16).astype(np.float32)  # 0.25 H (d v): <= 8 significant bits
        assert np.array_equal(oracle.inverse_rht16(oracle.rht16(v, mask), mask), v), mask


def test_f32_to_bf16_array_matches_torch_including_ties():
    rng = np.random.default_rng(43)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits[:2000] = (bits[:2000] & 0xFFFF0000) | 0x8000      # exact ties
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16_array(x), ref)


def test_inverse_rht_dequantization_keeps_the_transformed_domain_error():
    """0.25 H16 d is orthogonal, so the columnwise reconstruction error of an RHT-quantized
    tensor is the quantization error of the transformed values (up to their BF16 rounding)."""
    x = workloads.normal_with_outliers(256, 96, seed=44, fraction=0.01, gain=20.0)
    mask = 0x6A5C
    cc, cs, gs = oracle.quantize_colwise(x, rht=True, sign_mask=mask)
    xt = x.float().numpy().T.astype(np.float64)            # [N][M]: the columns of x
    rec = oracle.dequantize_ex(cc, cs, gs[1], inverse_rht=True, sign_mask=mask).astype(np.float64)
    yq = oracle.dequantize(cc, cs, gs[1]).astype(np.float64)  # transformed domain
    y = np.stack([np.concatenate([oracle.rht16(xt[n, 16 * b:16 * b + 16].astype(np.float32), mask)
                                  for b in range(xt.shape[1] // 16)]) for n in range(xt.shape[0])])
    err_x = ((rec - xt) ** 2).sum()
    err_y = ((yq - y) ** 2).sum()
    assert abs(err_x / err_y - 1.0) < 0.02, (err_x, err_y)
    db = 10 * np.log10((xt ** 2).sum() / err_x)
    assert 15.0 < db < 22.0, db


# ------------------------------------------------------------------------------------------
# RMSNorm producer with the amax in its epilogue (reading R14)
# ------------------------------------------------------------------------------------------

def test_rsqrt_rn_is_correctly_rounded():
    """Against exact rational arithmetic: the result's two midpoints enclose 1/sqrt(a), i.e.
    lo^2 a <= 1 <= hi^2 a (Fractions, independent of the oracle's integer comparison)."""
    from fractions import Fraction
    rng = np.random.default_rng(51)
    a = np.concatenate([rng.uniform(0.5, 2.0, 3000), 2.0 ** rng.uniform(-140, 120, 3000),
                        np.array([1.0, 2.0, 4.0, 0.25, 3.0])]).astype(np.float32)
    # hard cases: a whose 1/sqrt(a) is close to a binary32 midpoint
    m = (np.float32(1.25) + np.nextafter(np.float32(1.25), np.float32(2))) / 2
    a = np.concatenate([a, np.array([1 / float(m) ** 2], dtype=np.float32),
                        np.nextafter(np.array([1 / float(m) ** 2], dtype=np.float32), 2)])
    for ai in a:
        y = oracle.rsqrt_rn(ai)
        up = np.nextafter(y, np.float32(np.inf))
        dn = np.nextafter(y, np.float32(0))
        fa = Fraction(float(ai))
        hi = (Fraction(float(y)) + Fraction(float(up))) / 2
        lo = (Fraction(float(y)) + Fraction(float(dn))) / 2
        assert lo * lo * fa <= 1 <= hi * hi * fa, (ai, y)


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(52)
    N = 512
    w = _bf16(rng.normal(0, 1, N))
    wf = w.float().numpy()
    for c in (1.0, 2.0 ** -5, 2.0 ** 7):       # constant rows: mean = c^2 exactly, rms = 1/c
        x = _bf16(np.full((3, N), c))
        y, amax = oracle.rmsnorm(x, w, eps=0.0)
        yf = (y.astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(yf, np.broadcast_to(wf, yf.shape)), c
        assert amax == np.abs(wf).max()
    x = _bf16(np.ones((2, N)))
    y, _ = oracle.rmsnorm(x, w, eps=0.0, bias=1.0)   # y = bf16(w + 1)
    want = oracle.f32_to_bf16_array((wf + np.float32(1.0)).astype(np.float32))
    assert np.array_equal(y[0], want) and np.array_equal(y[1], want)


def test_rmsnorm_within_one_bf16_step_of_float64_and_amax():
    rng = np.random.default_rng(53)
    M, N = 64, 4096
    x = workloads.normal_with_outliers(M, N, seed=54, fraction=0.01, gain=20.0)
    w = _bf16(rng.normal(1.0, 0.2, N))
    eps, bias = 1e-6, 0.5
    y, amax = oracle.rmsnorm(x, w, eps=eps, bias=bias)
    xf = x.double().numpy()
    wf = w.double().numpy()
    ref = (wf + np.float32(bias)) * xf / np.sqrt((xf ** 2).mean(axis=1, keepdims=True) + np.float32(eps))
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert (np.abs(yf - ref) <= ulp * 1.0001).all()
    assert amax == np.float32(np.abs(yf).max())


# ------------------------------------------------------------------------------------------
# Grouped 2D weights (reading R15)
# ------------------------------------------------------------------------------------------

def test_grouped_2d_tile_scales_transposes_padding_and_special_cases():
    T, H = 150, 64
    x = oracle.as_bf16_bits(workloads.normal_with_outliers(T, H, seed=61, fraction=0.02, gain=20.0))
    offsets = np.array([32, 32, 57, 100, 140], dtype=np.int32)  # whole, empty, ragged; tail 140..
    cap = oracle.padded_capacity(offsets) + 16
    rc, rs, rg, cc, cs, cg = oracle.quantize_grouped(x, offsets, cap=cap, block2d=True, fill=0xEE)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert np.all(rc[140:] == 0xEE) and np.all(rs[140:] == 0xEE)
    prev, col = 0, 0
    for e, end in enumerate(offsets.tolist()):
        n = end - prev
        if n == 0:
            assert list(rg[e]) == [0.0, 1.0] and list(cg[e]) == [0.0, 1.0]
            continue
        P = (n + 15) // 16 * 16
        amax = np.abs(xf[prev:end]).max()
        s_enc, s_dec = oracle.global_scale(amax)
        assert rg[e][0] == amax and rg[e][1] == s_dec and list(cg[e]) == list(rg[e])
        for t in range(P // 16):
            rows = slice(prev + 16 * t, min(prev + 16 * t + 16, end))
            for tc in range(H // 16):
                tile_max = np.abs(xf[rows, 16 * tc:16 * tc + 16]).max()
                s = oracle.block_scale(tile_max, s_enc)
                assert np.all(rs[rows, tc] == s)                      # every real row of the tile
                assert np.all(cs[16 * tc:16 * tc + 16, (col + 16 * t) // 16] == s)
        # column codes are the transposed row codes; the padding rows encode zeros
        rn = np.stack([rc[prev:end] & 0xF, rc[prev:end] >> 4], axis=-1).reshape(n, H)
        cn = np.stack([cc[:, col // 2:(col + P) // 2] & 0xF, cc[:, col // 2:(col + P) // 2] >> 4],
                      axis=-1).reshape(H, P)
        assert np.array_equal(cn[:, :n], rn.T) and not cn[:, n:].any()
        if n % 16 == 0:   # a whole-tile expert is a plain 2D call on its slice
            pc, ps, pcc, pcs, pg = oracle.quantize_2d(x[prev:end])
            assert np.array_equal(pc, rc[prev:end]) and np.array_equal(ps, rs[prev:end])
            assert np.array_equal(pcc, cc[:, col // 2:(col + P) // 2])
        prev, col = end, col + P
    assert np.all(cc[:, col // 2:] == 0xEE) and np.all(cs[:, col // 16:] == 0xEE)


def test_batch_conversion_helpers_equal_the_per_element_steps():
    """oracle.sr_convert4 and oracle.e2m1_encode_rn_n (used to check the conversion
    instructions on the GPU) are batch forms of the pinned per-element encoders."""
    rng = np.random.default_rng(77)
    t = rng.uniform(-7, 7, size=4 * 300).astype(np.float32)
    w = rng.integers(0, 2**32, size=300, dtype=np.uint64).astype(np.uint32)
    one = np.array([oracle.e2m1_encode_sr(t[k], oracle.sr_random16(int(w[k // 4]), k % 4))[0]
                    for k in range(t.size)], dtype=np.uint8)
    assert np.array_equal(oracle.sr_convert4(t, w), one)
    assert np.array_equal(oracle.e2m1_encode_rn_n(t), oracle.e2m1_encode_rn(t))
