"""QuantizeMX on the GPU (through the C-ABI) against the CPU oracle, bit for
bit: data bytes and E8M0 scales, every geometry / layout / format / input
type, ragged widths, special values, sentinels around the outputs, and the
full-size sweep and FP4 workloads."""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc
from helpers import sf_pack, to_device_bits

pytestmark = pytest.mark.gpu

GEOMS = [("8x4", -2), ("8x4", -1), ("1x32", -1), ("1x32", -2)]
BLOCK = {("8x4", -2): (8, 4), ("8x4", -1): (4, 8), ("1x32", -1): (1, 32), ("1x32", -2): (32, 1)}


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


def _shapes(geometry, dim):
    br, bc = BLOCK[(geometry, dim)]
    wide = (br * 9, max(bc, 8) * 41)               # several warp tiles, cols % 8 == 0
    shapes = [wide]
    if bc <= 4:                                      # ragged width: cols % 8 == 4 (generic kernel)
        shapes.append((br * 5, 8 * 19 + 4))
    if br == 1:
        shapes.append((37, 32 * 7))                  # row count not a multiple of the 4-row group
    return shapes


def _run(mx, bits, in_dtype, fmt, geometry, dim, layout, stride=2, parity=0, emax_alt=False, fill=0xAB):
    import torch
    rows, cols = bits.shape
    x = to_device_bits(bits, in_dtype)
    _, srows, scols = mx.mx_quantize_sizes(rows, cols, in_dtype, fmt,
                                           mx.make_cfg(geometry, dim, layout, stride, parity, emax_alt))
    data_len = rows * cols // (2 if fmt == "e2m1" else 1)
    data = torch.full((data_len + 64,), 0xCD, dtype=torch.uint8, device="cuda")   # 64-byte canary
    scale = torch.full((srows * scols + 64,), fill, dtype=torch.uint8, device="cuda")
    mx.mx_quantize(x, fmt, geometry=geometry, dim=dim, scale_layout=layout, fp4_lane_stride=stride,
                   fp4_nibble_parity=parity, emax_alt=emax_alt, out_data=data, out_scale=scale)
    torch.cuda.synchronize()
    d, s = data.cpu().numpy(), scale.cpu().numpy()
    assert np.all(d[data_len:] == 0xCD), "data written past its end"
    assert np.all(s[srows * scols:] == fill), "scale written past its end"
    return d[:data_len], s[:srows * scols].reshape(srows, scols)


@pytest.mark.parametrize("layout", ["plain", "interleave"])
@pytest.mark.parametrize("geometry,dim", GEOMS)
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2", "e2m1"])
@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_quantize_matches_oracle(mx, in_dtype, fmt, geometry, dim, layout):
    for i, (rows, cols) in enumerate(_shapes(geometry, dim)):
        br, bc = BLOCK[(geometry, dim)]
        bits = syn.random_bits(rows, cols, in_dtype, seed=100 + i, special_fraction=0.01,
                               block_exp=(-40, 40) if in_dtype == "bf16" else (-14, 10), block=(br, bc))
        want_d, want_s = orc.quantize(bits, in_dtype, fmt, geometry=geometry, dim=dim,
                                      scale_layout=layout, scale_fill=0xAB)
        got_d, got_s = _run(mx, bits, in_dtype, fmt, geometry, dim, layout)
        assert np.array_equal(got_s, want_s), f"scales differ at {np.argwhere(got_s != want_s)[:5]}"
        bad = np.nonzero(got_d != want_d.reshape(-1))[0]
        assert bad.size == 0, f"{bad.size} data bytes differ, first at {bad[:5]}: " \
                              f"got {got_d[bad[:5]]} want {want_d.reshape(-1)[bad[:5]]}"


@pytest.mark.parametrize("stride", [0, 1, 2, 4])
@pytest.mark.parametrize("parity", [0, 1])
@pytest.mark.parametrize("geometry,dim", [("8x4", -2), ("1x32", -1), ("8x4", -1)])
def test_fp4_packing_variants(mx, stride, parity, geometry, dim):
    rows, cols = 64, 256
    bits = syn.random_bits(rows, cols, "bf16", seed=7, block_exp=(-10, 10), block=BLOCK[(geometry, dim)])
    want_d, want_s = orc.quantize(bits, "bf16", "e2m1", geometry=geometry, dim=dim,
                                  lane_stride=stride, nibble_parity=parity)
    got_d, got_s = _run(mx, bits, "bf16", "e2m1", geometry, dim, "plain", stride, parity)
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_d, want_d.reshape(-1))


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2", "e2m1"])
@pytest.mark.parametrize("geometry,dim", [("8x4", -2), ("1x32", -1)])
def test_emax_alternative_mode(mx, fmt, geometry, dim):
    bits = syn.random_bits(64, 128, "bf16", seed=9, block_exp=(-30, 30), block=BLOCK[(geometry, dim)])
    want_d, want_s = orc.quantize(bits, "bf16", fmt, geometry=geometry, dim=dim, emax_alt=True)
    got_d, got_s = _run(mx, bits, "bf16", fmt, geometry, dim, "plain", emax_alt=True)
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_d, want_d.reshape(-1))


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2", "e2m1"])
def test_special_value_blocks(mx, in_dtype, fmt):
    # every block made only of edge-case patterns: signed zeros, subnormals,
    # maxima, +-Inf, NaN
    rng = np.random.default_rng(3)
    pool = syn.special_values(in_dtype)
    bits = rng.choice(pool, size=(64, 64)).astype(np.uint16)
    for geometry, dim in GEOMS:
        want_d, want_s = orc.quantize(bits, in_dtype, fmt, geometry=geometry, dim=dim)
        got_d, got_s = _run(mx, bits, in_dtype, fmt, geometry, dim, "plain")
        assert np.array_equal(got_s, want_s), (geometry, dim)
        assert np.array_equal(got_d, want_d.reshape(-1)), (geometry, dim)


def test_hand_worked_blocks_on_gpu(mx, golden):
    for name, in_dtype, fmt, inputs, e_hex, codes_hex in golden("hand_worked_blocks.txt"):
        flat = np.zeros((1, 32), np.uint16)
        vals = [int(t, 16) for t in inputs.split()]
        flat[0, :len(vals)] = vals
        got_d, got_s = _run(mx, flat, in_dtype, fmt, "1x32", -1, "plain", stride=0, parity=1)
        assert got_s[0, 0] == int(e_hex, 16), name
        want = [int(t, 16) for t in codes_hex.split()]
        if fmt == "e2m1":
            codes = [(int(got_d[j // 2]) >> (4 * (j % 2))) & 0xF for j in range(32)]
        else:
            codes = list(got_d)
        assert codes[:len(want)] == want, name
        assert all(c == 0 for c in codes[len(want):]), name


def test_strided_and_folded_inputs(mx):
    import torch
    bits = syn.random_bits(64, 320, "bf16", seed=5, block_exp=(-8, 8))
    x = to_device_bits(bits, "bf16")
    view = x[:, :256]                                   # pitch 320 > width 256
    d, s = mx.mx_quantize(view, "e4m3fn", geometry="1x32", dim=-1)
    want_d, want_s = orc.quantize(bits, "bf16", "e4m3fn", geometry="1x32", dim=-1, cols=256)
    assert np.array_equal(d.cpu().numpy(), want_d) and np.array_equal(s.cpu().numpy(), want_s)
    x3 = to_device_bits(bits[:, :256].copy(), "bf16").reshape(4, 16, 256)   # rank 3 folds to [64, 256]
    d3, s3 = mx.mx_quantize(x3, "e4m3fn", geometry="8x4", dim=-2)
    want_d, want_s = orc.quantize(bits[:, :256].copy(), "bf16", "e4m3fn", geometry="8x4", dim=-2)
    assert np.array_equal(d3.cpu().numpy(), want_d) and np.array_equal(s3.cpu().numpy(), want_s)
    torch.cuda.synchronize()


def test_empty_input_launches_nothing(mx):
    import torch
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    d, s = mx.mx_quantize(x, "e4m3fn")
    assert d.numel() == 0 and s.numel() == 0


@pytest.mark.parametrize("rows,cols", [(256, 256), (200, 96), (130, 160)])
def test_sf_layout_output(mx, rows, cols):
    bits = syn.random_bits(rows, cols, "bf16", seed=11, block_exp=(-20, 20), block=(1, 32))
    _, plain = orc.quantize(bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    want = sf_pack(plain)
    got_d, got_s = _run(mx, bits, "bf16", "e4m3fn", "1x32", -1, "sf", fill=0x5A)
    assert np.array_equal(got_s.reshape(-1), want)
    want_d, _ = orc.quantize(bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    assert np.array_equal(got_d, want_d.reshape(-1))


def test_repack_matches_host_layout(mx):
    import torch
    rng = np.random.default_rng(1)
    for mn, k in [(128, 128), (300, 96), (1000, 2048), (7, 32)]:
        plain = rng.integers(1, 255, size=(mn, k // 32)).astype(np.uint8)
        sf = mx.mx_repack_scales(torch.from_numpy(plain).cuda(), k)
        assert np.array_equal(sf.cpu().numpy(), sf_pack(plain)), (mn, k)


# --------------------------------------------------------------- full size

@pytest.mark.parametrize("layout", ["plain", "interleave"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_sweep_full_size(mx, in_dtype, fmt, layout):
    """QuantizeMX sweep workload: [8192, 8192], 8x4 blocks, dim=-2, with the
    injected all-zero / subnormal / at-max / tie blocks; every byte checked."""
    bits = syn.sweep_input(8192, 8192, in_dtype, fmt, seed=0)
    want_d, want_s = orc.quantize(bits, in_dtype, fmt, geometry="8x4", dim=-2, scale_layout=layout,
                                  scale_fill=0xAB)
    got_d, got_s = _run(mx, bits, in_dtype, fmt, "8x4", -2, layout)
    assert got_s.shape == ((1024 if layout == "plain" else 8192), 2048)
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_d, want_d.reshape(-1))


def test_fp4_full_size(mx):
    """FP4 workload: [16384, 16384] bf16 -> e2m1, 8x4 blocks, packed nibbles
    (stride 2, parity 0), interleaved scales, 2% tie blocks."""
    bits = syn.fp4_input(16384, 16384, seed=0)
    want_d, want_s = orc.quantize(bits, "bf16", "e2m1", geometry="8x4", dim=-2, scale_layout="interleave",
                                  scale_fill=0xAB)
    got_d, got_s = _run(mx, bits, "bf16", "e2m1", "8x4", -2, "interleave")
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_d, want_d.reshape(-1))
