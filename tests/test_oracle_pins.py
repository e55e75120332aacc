"""Pins for the CPU oracle.

Every check here compares the oracle with something other than itself: a value
the pages print, a hand-worked block (tests/golden), a library conversion
(torch / numpy), a closed form, or a brute-force search written with different
primitives (math.frexp, a sorted grid, exact rationals).  None of it needs a
GPU.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import mx_synth as syn
import oracle as orc
from conftest import read_golden

FP8 = ["e4m3fn", "e5m2"]
ALL_FMTS = FP8 + ["e2m1"]
EMAX = {"e2m1": 2, "e4m3fn": 8, "e5m2": 15}  # page 2, "The EMAX Table", NOTE
MAXV = {"e2m1": 6.0, "e4m3fn": 448.0, "e5m2": 57344.0}
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # page 2, "FP4 e2m1", Grid =
TORCH_FP8 = {"e4m3fn": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


# ------------------------------------------------------------- helpers

def torch_decode_fp8(fmt, codes):
    """FP8 codes -> float64 via torch's own float8 conversion."""
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(TORCH_FP8[fmt])
    return t.to(torch.float64).numpy()


def positive_grid(fmt):
    """(magnitudes, codes) of every finite non-negative code, sorted."""
    if fmt == "e2m1":
        return np.array(E2M1_GRID), np.arange(8)
    codes = np.arange(128, dtype=np.uint8)
    vals = torch_decode_fp8(fmt, codes)
    keep = np.isfinite(vals)
    order = np.argsort(vals[keep], kind="stable")
    return vals[keep][order], codes[keep][order].astype(np.int64)


def nearest_grid_codes(fmt, y):
    """Brute-force narrow: nearest finite grid point, ties to the even code,
    saturating at the largest finite value; the sign bit is kept."""
    mags, codes = positive_grid(fmt)
    y = np.asarray(y, np.float32)
    a = np.abs(y.astype(np.float64))
    hi = np.searchsorted(mags, a, side="left")
    hi_c = np.minimum(hi, len(mags) - 1)
    lo_c = np.maximum(hi - 1, 0)
    d_lo = a - mags[lo_c]
    d_hi = mags[hi_c] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi_c] % 2 == 0))
    out = np.where(pick_hi, codes[hi_c], codes[lo_c])
    out = np.where(a >= mags[-1], codes[-1], out)  # saturate (Inf included)
    sign = (y.view(np.uint32) >> 31).astype(np.int64)
    return (out | (sign << (3 if fmt == "e2m1" else 7))).astype(np.uint8)


def frexp_exponent_byte(v):
    """Biased binary32 exponent of |v| from math.frexp; 0 for zero and
    binary32 subnormals, 255 for Inf/NaN."""
    if math.isnan(v) or math.isinf(v):
        return 255
    if v == 0 or abs(v) < 2.0 ** -126:
        return 0
    _, e = math.frexp(abs(v))
    return e - 1 + 127


def finite_bits(in_dtype):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = syn.from_bits(h, in_dtype)
    return h[np.isfinite(x)]


# ------------------------------------------------------- printed constants

def test_emax_table_values():
    # page 2, "The EMAX Table", NOTE: e2m1 2, e4m3fn 8, e5m2 15
    for fmt, v in EMAX.items():
        assert orc.emax(fmt) == v


def test_emax_alternative_mode():
    # page 2, doQuantizeMx QUIRK: emax_fp8_e4m3 = alt ? 7 : 8, emax_fp8_e5m2 = alt ? 14 : 15
    assert orc.emax_bias("e4m3fn", True) == 7 and orc.emax_bias("e4m3fn") == 8
    assert orc.emax_bias("e5m2", True) == 14 and orc.emax_bias("e5m2") == 15


def test_format_maxima_and_saturation():
    # page 2, "Gaps and Caveats" G1: 448 = 0x7E, 57344 = 0x7B; FP4 saturates to sign|7
    assert orc.narrow("e4m3fn", 1e30) == 0x7E and orc.decode("e4m3fn", 0x7E) == 448.0
    assert orc.narrow("e5m2", 1e30) == 0x7B and orc.decode("e5m2", 0x7B) == 57344.0
    assert orc.narrow("e4m3fn", -math.inf) == 0xFE
    assert orc.narrow("e5m2", math.inf) == 0x7B
    for v in (8.0, 7.0, 6.5, 1e38, math.inf):  # encode_e2m1: |x| >= 8 and round-up past 6 saturate
        assert orc.narrow("e2m1", v) == 0x7
        assert orc.narrow("e2m1", -v) == 0xF


def test_fp4_nan_is_signed_zero():
    # page 2, encode_e2m1: a NaN input becomes a signed zero nibble
    assert orc.narrow("e2m1", math.nan) == 0x0
    assert orc.narrow("e2m1", -math.nan) == 0x8


def test_fp4_decoder_matches_printed_grid():
    # page 2, decode_e2m1 and "Grid = {0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6}"
    vals = [orc.decode_e2m1_bits(i) for i in range(16)]
    assert vals[:8] == E2M1_GRID
    assert vals[8:] == [-v for v in E2M1_GRID]
    assert math.copysign(1.0, vals[8]) == -1.0
    assert [orc.decode("e2m1", i) for i in range(16)] == vals


@pytest.mark.parametrize("fmt", FP8)
def test_fp8_decode_matches_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.decode_array(fmt, codes)
    ref = torch_decode_fp8(fmt, codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


# -------------------------------------------------------------- E8M0 scale

def test_e8m0_clamp_low_then_zero_floor():
    # page 2, generateMxScales: floor the signed difference at 0, then raise a
    # 0 byte to 1; the byte always lies in [1, 255]
    for bias in (1, 2, 7, 8, 14, 15):
        seen = [orc.e8m0_from_max_exponent(m, bias) for m in range(256)]
        assert all(1 <= e <= 255 for e in seen)
        assert seen[0] == 1 and seen[bias] == 1 and seen[bias + 1] == 1
        assert seen[bias + 2] == 2 and seen[255] == 255 - bias
        assert all(b - a in (0, 1) for a, b in zip(seen, seen[1:]))  # monotone, unit steps


def test_prescale_multiplier_is_power_of_two():
    # page 2, quantizeDataApplyingMxScales: bit_cast((254 - E) << 23) = 2^(127 - E);
    # E = 127 multiplies by 1
    for e in range(1, 254):
        assert orc.prescale(1.0, e) == math.ldexp(1.0, 127 - e)
        assert orc.prescale(-3.0, e) == -3.0 * math.ldexp(1.0, 127 - e) or 127 - e > 126
    rng = np.random.default_rng(5)
    x = syn.from_bits(rng.integers(0, 0x7F80, 1000).astype(np.uint16), "bf16")
    assert np.array_equal(orc.prescale_array(x, np.uint8(127)), x)


def test_prescale_matches_numpy_binary32_multiply():
    # one binary32 multiply with round-to-nearest and gradual underflow
    h = finite_bits("bf16")
    x = syn.from_bits(h, "bf16")
    for e in range(1, 254, 7):
        mul = np.float32(math.ldexp(1.0, 127 - e))
        ref = x * mul
        got = orc.prescale_array(x, np.uint8(e))
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), e


# ------------------------------------------------------------- exponent byte

@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_exponent_byte_against_frexp(in_dtype):
    # page 2, findMaxExponentPerInputBlock GOTCHA: sign-independent; a binary32
    # denormal reads 0 (not its true exponent)
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = orc.widen_array(in_dtype, h)
    got = orc.exponent_byte_array(x)
    want = np.array([frexp_exponent_byte(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(orc.exponent_byte_array(-x), got)


def test_exponent_byte_of_binary32_denormal_is_zero():
    tiny = np.array([2.0 ** -130, -(2.0 ** -149), 2.0 ** -126 * 0.75], np.float32)
    assert list(orc.exponent_byte_array(tiny)) == [0, 0, 0]


# --------------------------------------------------------------- widening

def test_widen_bf16_matches_torch():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.widen_array("bf16", h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_widen_f16_matches_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.widen_array("f16", h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# --------------------------------------------------------- narrow, brute force

@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_narrow_equals_nearest_grid_search(in_dtype, fmt):
    # every finite input value times every prescale 2^(127-E), E in [1, 253]
    x = syn.from_bits(finite_bits(in_dtype), in_dtype)
    for e in range(1, 254):
        y = x * np.float32(math.ldexp(1.0, 127 - e))
        got = orc.narrow_array(fmt, y)
        want = nearest_grid_codes(fmt, y)
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0][:5]
            pytest.fail(f"E={e}: y={y[bad]} got={got[bad]} want={want[bad]}")


@pytest.mark.parametrize("fmt", FP8)
def test_narrow_matches_torch_after_clamp(fmt):
    # torch's float8 conversion rounds to nearest-even but does not saturate:
    # clamp to +-max first, then compare
    rng = np.random.default_rng(11)
    y = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))).astype(np.float32)
    y = np.concatenate([y, np.float32([0.0, -0.0, 448.0, 464.0, 480.0, 57344.0, 61440.0, 2.0 ** -10])])
    got = orc.narrow_array(fmt, y)
    clamped = np.clip(y, -MAXV[fmt], MAXV[fmt])
    ref = torch.from_numpy(clamped).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_fp8_nan_reading():
    # reading (the pages fix no NaN code): NaN -> 0x7F | sign for both FP8 formats
    for fmt in FP8:
        assert orc.narrow(fmt, math.nan) == 0x7F
        assert orc.narrow(fmt, -math.nan) == 0xFF


@pytest.mark.parametrize("fmt", FP8)
def test_fp8_nan_code_is_a_nan_of_the_format(fmt):
    # What the format definitions do fix, independently of the reading above:
    # a NaN input must come out as a code that the format decodes as NaN
    # (torch's float8 decoder, a library routine), carrying the input's sign
    # bit; no finite input may produce such a code.
    for sign, x in ((0, math.nan), (1, -math.nan)):
        c = orc.narrow(fmt, x)
        v = torch.tensor([c], dtype=torch.uint8).view(TORCH_FP8[fmt]).float().item()
        assert math.isnan(v), (fmt, hex(c))
        assert c >> 7 == sign, (fmt, hex(c))
    # inside a block: the NaN element decodes as NaN, its finite neighbours
    # stay finite
    bits = np.array([[0x3F80, 0x7FC0, 0xFFC0, 0xC040] * 8], np.uint16)  # 1, NaN, -NaN, -3
    q, _ = orc.quantize(bits, "bf16", fmt, geometry="1x32", dim=-1)
    dec = torch.from_numpy(np.ascontiguousarray(q[0, :4])).view(TORCH_FP8[fmt]).float().numpy()
    assert np.isnan(dec[1]) and np.isnan(dec[2]) and np.isfinite(dec[0]) and np.isfinite(dec[3])
    assert int(q[0, 1]) >> 7 == 0 and int(q[0, 2]) >> 7 == 1


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_every_code_round_trips(fmt):
    n = 16 if fmt == "e2m1" else 256
    for c in range(n):
        v = orc.decode(fmt, c)
        if math.isnan(v) or math.isinf(v):
            continue
        assert orc.narrow(fmt, v) == c, (fmt, hex(c), v)


# ------------------------------------------------------ hand-worked blocks

def _nibbles(packed, n):
    return [(int(packed[j // 2]) >> (4 * (j % 2))) & 0xF for j in range(n)]


@pytest.mark.parametrize("case", read_golden("hand_worked_blocks.txt"), ids=lambda c: c[0])
@pytest.mark.parametrize("geometry", ["1x32", "8x4"])
def test_hand_worked_block(case, geometry):
    name, in_dtype, fmt, inputs, e_hex, codes_hex = case
    vals = [int(t, 16) for t in inputs.split()]
    flat = np.zeros(32, np.uint16)
    flat[:len(vals)] = vals
    want_codes = [int(t, 16) for t in codes_hex.split()]
    shape, dim = ((1, 32), -1) if geometry == "1x32" else ((8, 4), -2)
    x = flat.reshape(shape)
    # stride 0 / parity 1 packs element 2k in the low nibble of byte k
    data, scale = orc.quantize(x, in_dtype, fmt, geometry=geometry, dim=dim,
                               lane_stride=0, nibble_parity=1)
    assert scale.shape == (1, 1) and scale[0, 0] == int(e_hex, 16)
    codes = _nibbles(data.reshape(-1), 32) if fmt == "e2m1" else list(data.reshape(-1))
    assert codes[:len(want_codes)] == want_codes
    zero = 0
    assert all(c == zero for c in codes[len(want_codes):])


@pytest.mark.parametrize("case", read_golden("fp4_packing.txt"), ids=lambda c: c[0])
def test_fp4_packing(case):
    name, stride, parity, nibs, packed = case
    nib = [int(t, 16) for t in nibs.split()]
    want = [int(t, 16) for t in packed.split()]
    assert list(orc.pack_nibbles(nib, int(stride), int(parity))) == want


def test_lane_remap_is_a_permutation_of_each_window():
    # page 2, lane_remap: reverse within each window of 2*stride
    for stride in range(1, 9):
        w = 2 * stride
        for q in range(4):
            window = list(range(q * w, (q + 1) * w))
            assert sorted(orc.lane_remap(i, stride) for i in window) == window
    assert [orc.lane_remap(i, 1) for i in range(8)] == list(range(8))


def test_fp4_quantize_packs_with_default_stride():
    # the whole quantizer with the default packing (stride 2, parity 0) puts
    # element 0 in the most significant nibble of each 16-bit container
    x = np.zeros((1, 32), np.uint16)
    x[0, :6] = [0x40C0, 0x40E0, 0x3E80, 0x3F40, 0xC0A0, 0x3FA0]
    data, _ = orc.quantize(x, "bf16", "e2m1", geometry="1x32", dim=-1)
    assert list(data[0, :4]) == [0x02, 0x77, 0x00, 0xE2]


# ------------------------------------------------------------ scale layout

def test_interleave_slots_injective_and_symmetric():
    # page 2, copy2DScaleVectorToArray: row i -> slot (i & 3) + 32 * (i >> 2);
    # groups of 4 stay contiguous; the read-back uses the same index
    slots = [orc.scale_row_slot(i, "interleave") for i in range(4096)]
    assert len(set(slots)) == len(slots)
    for i, s in enumerate(slots):
        assert s % 32 == i % 4 and s // 32 == i // 4
    assert [orc.scale_row_slot(i, "plain") for i in range(9)] == list(range(9))


@pytest.mark.parametrize("geometry,dim", [("8x4", -2), ("8x4", -1), ("1x32", -1), ("1x32", -2)])
def test_interleaved_scales_hold_plain_rows(geometry, dim):
    x = syn.random_bits(64, 64, "bf16", seed=3, block_exp=(-20, 20))
    _, plain = orc.quantize(x, "bf16", "e4m3fn", geometry=geometry, dim=dim)
    _, inter = orc.quantize(x, "bf16", "e4m3fn", geometry=geometry, dim=dim,
                            scale_layout="interleave", scale_fill=0xAB)
    n = plain.shape[0]
    assert inter.shape[0] == 32 * ((n + 3) // 4)
    live = np.zeros(inter.shape[0], bool)
    for i in range(n):
        slot = (i & 3) + 32 * (i >> 2)
        assert np.array_equal(inter[slot], plain[i])
        live[slot] = True
    assert np.all(inter[~live] == 0xAB)  # rows never addressed stay untouched


# ----------------------------------------- whole quantizer vs brute force

def _blocks(rows, cols, geometry, dim):
    br, bc = {("8x4", -2): (8, 4), ("8x4", -1): (4, 8),
              ("1x32", -1): (1, 32), ("1x32", -2): (32, 1)}[(geometry, dim)]
    return br, bc


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", ALL_FMTS)
@pytest.mark.parametrize("geometry,dim", [("8x4", -2), ("8x4", -1), ("1x32", -1), ("1x32", -2)])
def test_quantize_against_brute_force(in_dtype, fmt, geometry, dim):
    rows, cols = 64, 96
    br, bc = _blocks(rows, cols, geometry, dim)
    x = syn.random_bits(rows, cols, in_dtype, seed=7, special_fraction=0.03,
                        block_exp=(-40, 40) if in_dtype == "bf16" else (-12, 8), block=(br, bc))
    data, scale = orc.quantize(x, in_dtype, fmt, geometry=geometry, dim=dim,
                               lane_stride=0, nibble_parity=1)
    xf = syn.from_bits(x, in_dtype)  # library widening
    assert scale.shape == (rows // br, cols // bc)
    for i in range(rows // br):
        for j in range(cols // bc):
            blk = xf[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
            m = max(frexp_exponent_byte(float(v)) for v in blk.reshape(-1))
            e = max(1, m - EMAX[fmt])
            assert scale[i, j] == e, (i, j)
            y = blk * np.float32(math.ldexp(1.0, 127 - e))
            want = nearest_grid_codes(fmt, y.reshape(-1)).reshape(br, bc)
            if fmt == "e2m1":
                nib = np.array(_nibbles(data.reshape(-1), rows * cols)).reshape(rows, cols)
                got = nib[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
            else:
                got = data[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
            finite = np.isfinite(y)
            assert np.array_equal(got[finite], want[finite]), (i, j)


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_block_max_after_prescale_in_top_binade(fmt):
    # page 2, generateMxScales interpretation: when maxExp - EMAX >= 1 the block
    # maximum lands in [2^EMAX, 2^(EMAX+1)); never a NaN/Inf code from finite input
    x = syn.random_bits(128, 128, "bf16", seed=9, block_exp=(-60, 60))
    data, scale = orc.quantize(x, "bf16", fmt, lane_stride=0, nibble_parity=1)
    xf = syn.from_bits(x, "bf16").reshape(16, 8, 32, 4)
    e = scale.astype(np.float64)[:, None, :, None]
    bmax = np.abs(xf.astype(np.float64)).max(axis=(1, 3), keepdims=True) * np.exp2(127 - e)
    big = np.abs(xf).max(axis=(1, 3), keepdims=True) >= 2.0 ** (EMAX[fmt] - 126)
    assert np.all((bmax[big] >= 2.0 ** EMAX[fmt]) & (bmax[big] < 2.0 ** (EMAX[fmt] + 1)))
    if fmt == "e2m1":
        codes = np.array(_nibbles(data.reshape(-1), 128 * 128))
        assert np.all((codes & 7) <= 7)
    else:
        dec = orc.decode_array(fmt, data)
        assert np.all(np.isfinite(dec)) and np.all(np.abs(dec) <= MAXV[fmt])


@pytest.mark.parametrize("fmt", ALL_FMTS)
def test_dequantize_inverts_quantize_on_grid(fmt):
    # page 2: the prescale is the exact inverse of the dequant's
    # ldexpf(x, E8M0 - 127); values already on the grid round-trip exactly
    rng = np.random.default_rng(13)
    mags, _ = positive_grid(fmt)
    rows, cols = 32, 32
    vals = rng.choice(mags, size=(rows, cols)) * np.where(rng.random((rows, cols)) < 0.5, -1, 1)
    k = rng.integers(-20, 20, size=(rows // 8, 1, cols // 4, 1))
    v = vals.reshape(rows // 8, 8, cols // 4, 4)
    v[:, 0:1, :, 0:1] = mags[-1]  # anchor: the format maximum fixes E = 127 + k
    x = (v * np.exp2(k)).reshape(rows, cols)
    bits = syn.to_bits(x.astype(np.float32), "bf16")
    assert np.array_equal(syn.from_bits(bits, "bf16").astype(np.float64), x)
    data, scale = orc.quantize(bits, "bf16", fmt)
    assert np.all(scale == (127 + k).reshape(rows // 8, cols // 4))
    back = orc.dequantize(data, scale, rows, cols, fmt)
    assert np.array_equal(back, x)


def test_shape_errors():
    x = np.zeros((12, 8), np.uint16)
    with pytest.raises(orc.OracleError):
        orc.quantize(x, "bf16", "e4m3fn", geometry="8x4", dim=-2)  # 12 % 8
    with pytest.raises(orc.OracleError):
        orc.quantize(np.zeros((8, 6), np.uint16), "bf16", "e4m3fn")  # 6 % 4
    with pytest.raises(orc.OracleError):
        orc.quantize(np.zeros((2, 48), np.uint16), "bf16", "e4m3fn", geometry="1x32", dim=-1)


def test_empty_tensor():
    data, scale = orc.quantize(np.zeros((0, 32), np.uint16), "bf16", "e4m3fn",
                               geometry="1x32", dim=-1)
    assert data.size == 0 and scale.size == 0


def test_strided_input_uses_pitch():
    x = syn.random_bits(16, 64, "bf16", seed=2)
    d1, s1 = orc.quantize(x[:, :32], "bf16", "e4m3fn", geometry="1x32", dim=-1)
    d2, s2 = orc.quantize(x, "bf16", "e4m3fn", geometry="1x32", dim=-1, cols=32)
    assert np.array_equal(d1, d2) and np.array_equal(s1, s2)


# ------------------------------------------------------------ scaled matmul

def _codes_for(fmt, values):
    return np.array([orc.narrow(fmt, float(v)) for v in np.asarray(values).reshape(-1)],
                    np.uint8).reshape(np.shape(values))


@pytest.mark.parametrize("fmt", FP8)
def test_matmul_unit_scales_equal_integer_matmul(fmt):
    # all scales 127 (x1) and small-integer elements: the definition reduces
    # to an ordinary matmul, compared with torch.matmul in float64
    rng = np.random.default_rng(17)
    M, N, K = 5, 7, 96
    a_int = rng.integers(-8, 9, size=(M, K))
    b_int = rng.integers(-8, 9, size=(N, K))
    a, bt = _codes_for(fmt, a_int), _codes_for(fmt, b_int)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    c, s = orc.scaled_matmul_entries(a, bt, sa, sb, fmt, fmt, ms.reshape(-1), ns.reshape(-1))
    ref = torch.matmul(torch.tensor(a_int, dtype=torch.float64),
                       torch.tensor(b_int, dtype=torch.float64).T).numpy()
    assert np.array_equal(c.reshape(M, N), ref)
    assert np.array_equal(s.reshape(M, N), np.abs(a_int) @ np.abs(b_int).T)


def test_matmul_scale_shift_is_exact_power_of_two():
    rng = np.random.default_rng(19)
    M, N, K = 4, 6, 128
    a = rng.integers(0, 0x7F, size=(M, K)).astype(np.uint8)  # finite positive e4m3 codes
    bt = rng.integers(0x80, 0xFF, size=(N, K)).astype(np.uint8)
    sa = rng.integers(100, 150, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(100, 150, size=(N, K // 32)).astype(np.uint8)
    ms, ns = [v.reshape(-1) for v in np.meshgrid(np.arange(M), np.arange(N), indexing="ij")]
    c0, _ = orc.scaled_matmul_entries(a, bt, sa, sb, "e4m3fn", "e4m3fn", ms, ns)
    for d in (-3, 5):
        c1, _ = orc.scaled_matmul_entries(a, bt, (sa.astype(int) + d).astype(np.uint8), sb,
                                          "e4m3fn", "e4m3fn", ms, ns)
        assert np.array_equal(c1, c0 * 2.0 ** d)


@pytest.mark.parametrize("fmt", FP8)
def test_matmul_k32_exact_rationals(fmt):
    # one 32-element block: exact rational sum of the products, with element
    # values decoded by torch and scales as exact powers of two
    rng = np.random.default_rng(23)
    M, N, K = 3, 5, 32
    finite = [c for c in range(256) if np.isfinite(torch_decode_fp8(fmt, np.array([c], np.uint8)))[0]]
    a = rng.choice(finite, size=(M, K)).astype(np.uint8)
    bt = rng.choice(finite, size=(N, K)).astype(np.uint8)
    sa = rng.integers(90, 160, size=(M, 1)).astype(np.uint8)
    sb = rng.integers(90, 160, size=(N, 1)).astype(np.uint8)
    da, db = torch_decode_fp8(fmt, a), torch_decode_fp8(fmt, bt)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(da[m, k])) * Fraction(float(db[n, k])) for k in range(K))
            exact *= Fraction(2) ** (int(sa[m, 0]) - 127 + int(sb[n, 0]) - 127)
            c, s = orc.scaled_matmul_entries(a, bt, sa, sb, fmt, fmt, [m], [n])
            assert abs(Fraction(float(c[0])) - exact) <= Fraction(float(s[0])) * Fraction(2) ** -50


def test_matmul_orientation_nonsquare():
    # C[m, n] pairs row m of A with row n of Bt (both K-contiguous); a
    # transposed operand or scale index breaks this on a non-square case
    rng = np.random.default_rng(29)
    M, N, K = 4, 3, 64
    a = rng.integers(0, 0x7E, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 0x7E, size=(N, K)).astype(np.uint8)
    sa = rng.integers(120, 135, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8)
    da = torch_decode_fp8("e4m3fn", a) * np.exp2(np.repeat(sa.astype(float) - 127, 32, axis=1))
    db = torch_decode_fp8("e4m3fn", bt) * np.exp2(np.repeat(sb.astype(float) - 127, 32, axis=1))
    for m in range(M):
        for n in range(N):
            c, _ = orc.scaled_matmul_entries(a, bt, sa, sb, "e4m3fn", "e4m3fn", [m], [n])
            assert c[0] == pytest.approx(float(np.dot(da[m], db[n])), rel=1e-14)


def test_matmul_two_oracle_paths_agree():
    rng = np.random.default_rng(31)
    M, N, K = 16, 24, 256
    a = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0  # no NaN codes
    bt[(bt & 0x7F) == 0x7F] = 0
    sa = rng.integers(110, 140, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(110, 140, size=(N, K // 32)).astype(np.uint8)
    C, S = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    ms, ns = [v.reshape(-1) for v in np.meshgrid(np.arange(M), np.arange(N), indexing="ij")]
    c, s = orc.scaled_matmul_entries(a, bt, sa, sb, "e4m3fn", "e4m3fn", ms, ns)
    assert np.allclose(C.reshape(-1), c, rtol=0, atol=1e-12 * s.max())
    assert np.allclose(S.reshape(-1), s, rtol=1e-12)
