"""Pins for the oracle's MX formats (MXFP8 E4M3 / E5M2, MXFP4 E2M1; 32-element blocks with an
E8M0 power-of-two scale). Each test checks the oracle against something other than itself:
torch's FP8 and E8M0 dtypes, brute force over every code of a format, closed forms of the
scale rule on exact powers of two, and invariants. CPU only.

The pages ("CuTeDSL at Perplexity", its Blackwell paragraph) name the formats and their
32-element block maxima; the scale and rounding rules are those of the OCP Microscaling
Formats v1.0 conversion (readings M1-M4 of the oracle).
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_quantize_gb300 import workloads

FORMATS = ["e4m3", "e5m2", "e2m1"]
EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}
MAXNORM = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0}
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _torch_fp8_values(dtype):
    """Value of every code 0..255 of a torch FP8 dtype (an independent decoder)."""
    c = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return c.view(dtype).float().numpy().astype(np.float64)


def _finite_table(fmt):
    """(codes, values) of every finite code of the element format, from an independent decoder:
    torch's FP8 dtypes for E4M3/E5M2, the OCP E2M1 magnitude list for FP4."""
    if fmt == "e2m1":
        codes = np.arange(16, dtype=np.uint8)
        vals = np.where(codes & 8, -1.0, 1.0) * GRID[codes & 7]
        return codes, vals
    vals = _torch_fp8_values(torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2)
    codes = np.arange(256, dtype=np.uint8)
    ok = np.isfinite(vals)
    return codes[ok], vals[ok]


# ------------------------------------------------------------------------------------------
# Element formats
# ------------------------------------------------------------------------------------------

def test_e5m2_decode_matches_torch_for_every_code():
    ref = _torch_fp8_values(torch.float8_e5m2)
    got = oracle.e5m2_decode(np.arange(256)).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e5m2_encode_matches_torch_in_range_and_saturates():
    vals = _torch_fp8_values(torch.float8_e5m2)
    pos = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pos[:-1] + pos[1:]) / 2                       # every tie
    rng = np.random.default_rng(1)
    rand = rng.uniform(-57000, 57000, 20000) * 10.0 ** rng.uniform(-9, 0, 20000)
    x = np.concatenate([pos, -pos, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        rand]).astype(np.float32)
    x = x[np.abs(x) <= 57344.0]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e5m2_encode(x), ref)
    # satfinite: anything at or beyond the largest finite magnitude clamps to it (0x7B)
    big = np.array([57344.0, 61439.0, 61440.0, 1e6, 3e38], dtype=np.float32)
    assert (oracle.e5m2_encode(big) == 0x7B).all()
    assert (oracle.e5m2_encode(-big) == 0xFB).all()


def test_e8m0_decode_matches_torch():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    c = torch.arange(255, dtype=torch.int32).to(torch.uint8)
    ref = c.view(torch.float8_e8m0fnu).float().numpy().astype(np.float64)
    assert np.array_equal(oracle.e8m0_decode(np.arange(255)), ref)


@pytest.mark.parametrize("fmt", FORMATS)
def test_element_encode_is_the_nearest_code_by_brute_force(fmt):
    """Reading M2 against a search over every finite code: nearest value, ties to the code
    with an even mantissa (even code), magnitudes beyond the largest normal saturate."""
    codes, values = _finite_table(fmt)
    pos = np.unique(values[values >= 0]).astype(np.float32)
    mids = (pos[:-1] + pos[1:]) / 2  # exact in binary32 (few significant bits)
    rng = np.random.default_rng(2)
    # scaled elements are BF16 values times a power of two, so binary32 inputs cover them
    t = np.concatenate([pos, mids, np.nextafter(mids, np.float32(0)),
                        np.nextafter(mids, np.float32(np.inf)),
                        rng.uniform(0, 1.3 * pos[-1], 3000).astype(np.float32),
                        pos[-1] * np.array([1.0, 1.01, 2.0, 1e3], dtype=np.float32)])
    t = np.concatenate([t, -t]).astype(np.float64)
    got = oracle.mx_encode(t, fmt)
    sign_bit = 8 if fmt == "e2m1" else 0x80
    for ti, g in zip(t, got):
        if abs(ti) >= pos[-1]:
            assert oracle.mx_decode([g], fmt)[0] == np.copysign(pos[-1], ti), (fmt, ti, g)
            continue
        d = np.abs(values - ti)
        cand = codes[d == d.min()]
        if len(cand) > 1:  # +0 / -0, or a tie between neighbours: the sign of t, then even
            want = sign_bit if np.signbit(ti) else 0
            cand = [c for c in cand if (c & sign_bit) == want]
            if len(cand) > 1:
                cand = [c for c in cand if (c & 1) == 0]
        assert g in cand, (fmt, ti, g, cand)


# ------------------------------------------------------------------------------------------
# Scale rule (reading M1)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FORMATS)
def test_scale_of_exact_powers_of_two(fmt):
    """amax = 2^k (every BF16 binade, subnormals included): floor(log2 amax) = k, so the
    exponent is k - emax, clamped to [-127, 127]."""
    for k in range(-133, 128):
        want = min(max(k - EMAX[fmt], -127), 127) + 127
        assert oracle.mx_scale(2.0 ** k, fmt) == want, (fmt, k)
        # the whole binade [2^k, 2^(k+1)) shares the scale
        assert oracle.mx_scale(np.nextafter(2.0 ** (k + 1), 0), fmt) == want, (fmt, k)
    assert oracle.mx_scale(0.0, fmt) == 0


@pytest.mark.parametrize("fmt", FORMATS)
def test_scaled_block_max_lands_in_the_top_binade(fmt):
    """Unless clamped, amax / X is in [2^emax, 2^(emax+1)): the block maximum uses the element
    format's largest exponent, and saturates only above its largest normal."""
    rng = np.random.default_rng(3)
    amax = 2.0 ** rng.uniform(-100, 100, 2000)
    for a in amax:
        X = oracle.e8m0_decode([oracle.mx_scale(a, fmt)])[0]
        r = a / X
        assert 2.0 ** EMAX[fmt] <= r < 2.0 ** (EMAX[fmt] + 1), (fmt, a, r)


# ------------------------------------------------------------------------------------------
# Blocks and tensors
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FORMATS)
def test_grid_valued_blocks_round_trip_exactly(fmt):
    """A block of representable values times 2^j whose maximum is the format's largest value
    dequantizes to itself."""
    codes, values = _finite_table(fmt)
    rng = np.random.default_rng(4)
    for j in (-40, -3, 0, 5, 60):
        v = rng.choice(values, size=(4, 32))
        v[:, 7] = MAXNORM[fmt]
        x = torch.from_numpy(v * 2.0 ** j).to(torch.bfloat16)
        assert np.array_equal(x.double().numpy(), v * 2.0 ** j)  # representable in BF16
        c, s = oracle.mx_quantize_rowwise(x, fmt)
        assert np.array_equal(oracle.mx_dequantize(c, s, fmt).astype(np.float64), v * 2.0 ** j)


@pytest.mark.parametrize("fmt", FORMATS)
def test_rowwise_matches_per_block_brute_force(fmt):
    """Every element of a tensor is the nearest code times the block's scale (dequantized
    error at most half a grid step of the scaled grid, or saturated)."""
    x = workloads.normal_with_outliers(8, 256, seed=5, fraction=0.02, gain=30.0)
    c, s = oracle.mx_quantize_rowwise(x, fmt)
    xf = x.double().numpy()
    deq = oracle.mx_dequantize(c, s, fmt).astype(np.float64)
    _, values = _finite_table(fmt)
    for r in range(8):
        for b in range(8):
            blk = xf[r, 32 * b:32 * b + 32]
            X = 2.0 ** (int(s[r, b]) - 127)
            assert s[r, b] == oracle.mx_scale(np.abs(blk).max(), fmt)
            grid = values * X
            for i in range(32):
                best = np.abs(grid - blk[i]).min()
                assert abs(deq[r, 32 * b + i] - blk[i]) == best, (fmt, r, b, i)


@pytest.mark.parametrize("fmt", FORMATS)
def test_colwise_equals_rowwise_of_transpose(fmt):
    x = workloads.normal(64, 96, 1.0, seed=6)
    cc, cs = oracle.mx_quantize_colwise(x, fmt)
    rc, rs = oracle.mx_quantize_rowwise(x.t().contiguous(), fmt)
    assert np.array_equal(cc, rc) and np.array_equal(cs, rs)


def test_fp4_packs_the_even_element_in_the_low_nibble():
    v = np.zeros(32)
    v[0], v[1] = 6.0, -0.5  # block max 6: X = 1
    c, s = oracle.mx_quantize_rowwise(torch.from_numpy(v[None]).to(torch.bfloat16), "e2m1")
    assert s[0, 0] == 127 and c[0, 0] == 0x97  # low nibble 7 (6.0), high nibble 0x9 (-0.5)


@pytest.mark.parametrize("fmt", FORMATS)
def test_zero_and_subnormal_blocks(fmt):
    z = torch.zeros(1, 32, dtype=torch.bfloat16)
    c, s = oracle.mx_quantize_rowwise(z, fmt)
    assert s[0, 0] == 0 and not c.any()
    # BF16 subnormals only: the exponent clamps at -127, elements are v * 2^127 (exact)
    bits = np.arange(1, 33, dtype=np.uint16).reshape(1, 32)
    c, s = oracle.mx_quantize_rowwise(bits, fmt)
    assert s[0, 0] == 0
    vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    deq = oracle.mx_dequantize(c, s, fmt).astype(np.float64)
    _, table = _finite_table(fmt)
    grid = table * 2.0 ** -127
    for i in range(32):
        assert abs(deq[0, i] - vals[0, i]) == np.abs(grid - vals[0, i]).min()


@pytest.mark.parametrize("fmt,lo,hi", [("e4m3", 29.0, 33.5), ("e5m2", 23.0, 27.5),
                                       ("e2m1", 16.5, 20.5)])
def test_sqnr_on_gaussian(fmt, lo, hi):
    """Mantissa bits set the noise floor: ~6 dB per bit (E4M3 3 bits, E5M2 2, E2M1 1 over a
    coarser grid); a wrong emax saturates or wastes a binade and leaves the band."""
    x = workloads.normal(256, 512, 1.0, seed=7)
    c, s = oracle.mx_quantize_rowwise(x, fmt)
    xf = x.double().numpy()
    d = oracle.mx_dequantize(c, s, fmt).astype(np.float64)
    db = 10 * np.log10((xf ** 2).sum() / ((xf - d) ** 2).sum())
    assert lo <= db <= hi, (fmt, db)
