"""MX dequantize on the GPU (through the C-ABI) against the oracle.

Codes and scales come from the oracle's quantizer on the host.  f32 output
must equal the oracle's binary64 value exactly (every value is representable
in f32); bf16 output must equal that value rounded to nearest even (torch's
conversion)."""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc
from helpers import to_device_u8

pytestmark = pytest.mark.gpu

GEOMS = [("8x4", -2), ("8x4", -1), ("1x32", -1), ("1x32", -2)]
BLOCK = {("8x4", -2): (8, 4), ("8x4", -1): (4, 8), ("1x32", -1): (1, 32), ("1x32", -2): (32, 1)}


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


def _expect(values, out_dtype):
    import torch
    with np.errstate(over="ignore", invalid="ignore"):
        f32 = values.astype(np.float32)   # past the f32 range: Inf, as the kernel's multiply gives
    if out_dtype == "f32":
        return f32
    return torch.from_numpy(f32).to(torch.bfloat16).float().numpy()


def _check(got, want):
    assert got.shape == want.shape
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _shapes(geometry, dim):
    br, bc = BLOCK[(geometry, dim)]
    out = [(br * 6, max(bc, 8) * 19)]
    if bc <= 4:
        out.append((br * 5 + (0 if br > 1 else 2), 8 * 11 + 4))   # odd rows start unaligned; 12-element tail
        out.append((br * 3, 16 * 7 + 4))                           # 4-element tail
    return out


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["plain", "interleave"])
@pytest.mark.parametrize("geometry,dim", GEOMS)
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2", "e2m1"])
def test_dequantize_matches_oracle(mx, fmt, geometry, dim, layout, out_dtype):
    import torch
    for i, (rows, cols) in enumerate(_shapes(geometry, dim)):
        bits = syn.random_bits(rows, cols, "bf16", seed=40 + i, special_fraction=0.01, block_exp=(-40, 40),
                               block=BLOCK[(geometry, dim)])
        data, scale = orc.quantize(bits, "bf16", fmt, geometry=geometry, dim=dim, scale_layout=layout)
        want = _expect(orc.dequantize(data, scale, rows, cols, fmt, geometry=geometry, dim=dim,
                                      scale_layout=layout), out_dtype)
        got = mx.mx_dequantize(to_device_u8(data), to_device_u8(scale), rows, cols, fmt, out_dtype,
                               geometry=geometry, dim=dim, scale_layout=layout)
        torch.cuda.synchronize()
        _check(got.float().cpu().numpy(), want)


@pytest.mark.parametrize("stride", [0, 1, 2, 4])
@pytest.mark.parametrize("parity", [0, 1])
def test_dequantize_fp4_packing_variants(mx, stride, parity):
    import torch
    rows, cols = 40, 96
    bits = syn.random_bits(rows, cols, "bf16", seed=3, block_exp=(-10, 10))
    data, scale = orc.quantize(bits, "bf16", "e2m1", lane_stride=stride, nibble_parity=parity)
    want = _expect(orc.dequantize(data, scale, rows, cols, "e2m1", lane_stride=stride, nibble_parity=parity), "f32")
    got = mx.mx_dequantize(to_device_u8(data), to_device_u8(scale), rows, cols, "e2m1", "f32",
                           fp4_lane_stride=stride, fp4_nibble_parity=parity)
    torch.cuda.synchronize()
    _check(got.cpu().numpy(), want)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_dequantize_every_code_and_extreme_scales(mx, fmt, out_dtype):
    # every code with scales across the whole E8M0 range, 0 and 0xFF (NaN)
    # included; bf16 output reaches the bf16 subnormals and rounds there
    import torch
    rows, cols = 256, 256
    rng = np.random.default_rng(5)
    data = rng.integers(0, 256, size=(rows, cols)).astype(np.uint8)
    data[0, :] = np.arange(256, dtype=np.uint8)
    scale = rng.integers(0, 256, size=(rows, cols // 32)).astype(np.uint8)
    scale[1, :] = 0
    scale[2, :] = 255
    want = _expect(orc.dequantize(data, scale, rows, cols, fmt, geometry="1x32", dim=-1), out_dtype)
    got = mx.mx_dequantize(to_device_u8(data), to_device_u8(scale), rows, cols, fmt, out_dtype,
                           geometry="1x32", dim=-1)
    torch.cuda.synchronize()
    got = got.float().cpu().numpy()
    inf = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf)
    _check(np.where(inf, 0, got), np.where(inf, 0, want).astype(np.float32))


def test_dequantize_sf_layout(mx):
    import torch
    rows, cols = 200, 160
    bits = syn.random_bits(rows, cols, "bf16", seed=8, block_exp=(-20, 20), block=(1, 32))
    data, plain = orc.quantize(bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    sf = mx.mx_repack_scales(to_device_u8(plain), cols)
    want = _expect(orc.dequantize(data, plain, rows, cols, "e4m3fn", geometry="1x32", dim=-1), "bf16")
    got = mx.mx_dequantize(to_device_u8(data), sf, rows, cols, "e4m3fn", "bf16", geometry="1x32", dim=-1,
                           scale_layout="sf")
    torch.cuda.synchronize()
    _check(got.float().cpu().numpy(), want)


def test_quantize_then_dequantize_round_trip_on_grid(mx):
    # values already on the grid come back exactly (the page's prescale is the
    # inverse of the dequant's scale)
    import torch
    rows, cols = 64, 64
    rng = np.random.default_rng(9)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    v = rng.choice(grid, size=(rows, cols)) * np.where(rng.random((rows, cols)) < 0.5, -1, 1)
    v.reshape(rows // 8, 8, cols // 4, 4)[:, 0, :, 0] = 6.0  # anchor per block
    k = rng.integers(-30, 30, size=(rows // 8, 1, cols // 4, 1)).astype(np.float64)
    x = (v.reshape(rows // 8, 8, cols // 4, 4) * np.exp2(k)).reshape(rows, cols)
    bits = syn.to_bits(x.astype(np.float32), "bf16")
    xd = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    d, s = mx.mx_quantize(xd, "e2m1")
    back = mx.mx_dequantize(d, s, rows, cols, "e2m1", "f32")
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy().astype(np.float64), x)
