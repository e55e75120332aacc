"""Pair-kernel C stores paced over the next tile.

The CTA of each pair that issues the MMAs stores its accumulator rows in
8 KB steps while the next tile's K stages are issued, when a cluster runs
more than one tile and a tile has at least 16 K stages.  These shapes have
more 256 x 256 tiles than pair clusters (about 74 on a GB300) and K long
enough for the pacing, with ragged N, row pitches that allow 32-, 16- or
no-byte vector stores, batched problems and MXFP4.  Every element is
checked against the oracle with the ScaledMatmul tolerance
|C - C_ref| <= 1e-4 * sum_k |a_k b_k| (+ 1 bf16 ulp of C_ref for bf16)."""
import numpy as np
import pytest

import oracle as orc
from helpers import check_gemm, to_device_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


def fp8_operands(shape_a, shape_b, fmt, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 256, size=shape_a).astype(np.uint8)
    bt = rng.integers(0, 256, size=shape_b).astype(np.uint8)
    for x in (a, bt):
        bad = (x & 0x7F) == 0x7F if fmt == "e4m3fn" else (x & 0x7F) >= 0x7C
        x[bad] = 0x38
    sa = rng.integers(112, 142, size=shape_a[:-1] + (shape_a[-1] // 32,)).astype(np.uint8)
    sb = rng.integers(112, 142, size=shape_b[:-1] + (shape_b[-1] // 32,)).astype(np.uint8)
    return a, bt, sa, sb


def test_multi_tile_ragged_n_f32(mx):
    # 9 x 10 tiles, the last tile column 16 wide; 16 K stages per tile
    import torch
    M, N, K = 2304, 2320, 2048
    a, bt, sa, sb = fp8_operands((M, K), (N, K), "e4m3fn", seed=31)
    c = mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e4m3fn", "f32")
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch() == (2, 1)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(c.cpu().numpy(), c_ref, s_ref, "f32")


@pytest.mark.parametrize("N,pad", [(2304, 0), (2304, 8), (2311, 5)])
def test_multi_tile_bf16_row_pitches(mx, N, pad):
    # pitch N + pad: 32-byte aligned rows, 16-byte aligned rows, and rows no
    # vector store can take (odd N); nothing is written past column N
    import torch
    M, K = 2560, 2048
    a, bt, sa, sb = fp8_operands((M, K), (N, K), "e5m2", seed=N + pad)
    big = torch.full((M, N + pad), -5.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, :N]
    mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e5m2", "bf16",
                        out=out)
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch() == (2, 1)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e5m2")
    check_gemm(out.float().cpu().numpy(), c_ref, s_ref, "bf16")
    if pad:
        assert torch.all(big[:, N:] == -5.0)


def test_batched_dot_multi_tile(mx):
    # 3 problems x 36 tiles: clusters run tiles of consecutive problems
    import torch
    B, M, N, K = 3, 1536, 1536, 2048
    a, bt, sa, sb = fp8_operands((B, M, K), (B, N, K), "e4m3fn", seed=44)
    got = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e4m3fn",
                                 "bf16", lhs_batch=(0,), rhs_batch=(0,))
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch() == (2, 1)
    got = got.float().cpu().numpy()
    for i in range(B):
        c_ref, s_ref = orc.scaled_matmul(a[i], bt[i], sa[i], sb[i], "e4m3fn")
        check_gemm(got[i], c_ref, s_ref, "bf16")


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_mxfp4_multi_tile(mx, out_dtype):
    # 9 x 9 tiles, 16 K stages of 256 elements
    import torch
    M, N, K = 2304, 2304, 4096
    rng = np.random.default_rng(55)
    a = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sa = rng.integers(112, 142, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(N, K // 32)).astype(np.uint8)

    def pack(codes):
        rows, k = codes.shape
        return orc.pack_nibbles(codes.reshape(-1), lane_stride=1, nibble_parity=1).reshape(rows, k // 2)

    c = mx.mx_scaled_matmul(to_device_u8(pack(a)), to_device_u8(pack(bt)), to_device_u8(sa), to_device_u8(sb),
                            "e2m1", out_dtype, K=K)
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch() == (2, 1)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e2m1")
    check_gemm(c.float().cpu().numpy(), c_ref, s_ref, out_dtype)
