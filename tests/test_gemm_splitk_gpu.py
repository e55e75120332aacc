"""Split-K on the 1-SM ScaledMatmul kernel (few-tile problems: small M).

When a problem has too few 128 x 256 output tiles to fill the GPU, a cluster
of S CTAs shares each tile, each accumulating a slice of K; the slices' f32
partial sums are added in slice order through distributed shared memory.
Every result is checked against the oracle with the ScaledMatmul tolerance
|C - C_ref| <= 1e-4 * sum_k |a_k b_k| (+ 1 bf16 ulp of C_ref for bf16), and
the launch hook confirms the split that ran."""
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


def fp8_operands(M, N, K, fmt, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    for x in (a, bt):
        bad = (x & 0x7F) == 0x7F if fmt == "e4m3fn" else (x & 0x7F) >= 0x7C
        x[bad] = 0x38
    sa = rng.integers(112, 142, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(N, K // 32)).astype(np.uint8)
    return a, bt, sa, sb


def fp4_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sa = rng.integers(112, 142, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(N, K // 32)).astype(np.uint8)
    return a, bt, sa, sb


def pack(codes):
    rows, k = codes.shape
    return orc.pack_nibbles(codes.reshape(-1), lane_stride=1, nibble_parity=1).reshape(rows, k // 2)


def matmul(mx, a, bt, sa, sb, fmt, out_dtype):
    import torch
    if fmt == "e2m1":
        c = mx.mx_scaled_matmul(to_device_u8(pack(a)), to_device_u8(pack(bt)), to_device_u8(sa), to_device_u8(sb),
                                "e2m1", out_dtype, K=a.shape[1])
    else:
        c = mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), fmt,
                                out_dtype)
    torch.cuda.synchronize()
    return c


def expected_split(mx, M, N, K, fmt, batch=1):
    """The host's rule, restated: the largest S <= 8 with tiles x S CTAs on
    the SMs and at least 4 K stages per slice (cluster residency permitting)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = batch * -(-M // 128) * -(-N // 256)
    num_kb = -(-K // (256 if fmt == "e2m1" else 128))
    for s in range(8, 1, -1):
        if tiles * s <= sms and num_kb >= 4 * s:
            return s
    return 1


SHAPES = [(1, 256, 4096), (16, 1024, 2048), (100, 700, 1024), (128, 256, 8192), (64, 4096, 4096),
          (33, 2000, 1056), (128, 300, 768)]


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2", "e2m1"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_split_k_matches_oracle(mx, fmt, out_dtype, M, N, K):
    if fmt == "e2m1":
        a, bt, sa, sb = fp4_operands(M, N, K, seed=M + N + K)
    else:
        a, bt, sa, sb = fp8_operands(M, N, K, fmt, seed=M + N + K)
    c = matmul(mx, a, bt, sa, sb, fmt, out_dtype)
    kernel, split = mx.mx_debug_last_gemm_launch()
    assert kernel == 1
    want = expected_split(mx, M, N, K, fmt)
    # a cluster size the GPU cannot hold resident is skipped for a smaller one
    assert 1 < split <= want or want == 1, (split, want)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, fmt)
    check_gemm(c.float().cpu().numpy(), c_ref, s_ref, out_dtype)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e2m1"])
def test_split_and_unsplit_agree_with_oracle(mx, fmt):
    # the same problem with split-K and with it disabled: both within the
    # tolerance, and each run of the split kernel bit-identical to the last
    import torch
    M, N, K = 96, 512, 4096
    ops = fp4_operands(M, N, K, seed=3) if fmt == "e2m1" else fp8_operands(M, N, K, fmt, seed=3)
    c_ref, s_ref = orc.scaled_matmul(*ops, fmt)
    split1 = matmul(mx, *ops, fmt, "f32")
    assert mx.mx_debug_last_gemm_launch()[1] > 1
    split2 = matmul(mx, *ops, fmt, "f32")
    assert torch.equal(split1.view(torch.int32), split2.view(torch.int32))
    mx.mx_debug_set_gemm_variant(3)
    try:
        whole = matmul(mx, *ops, fmt, "f32")
        assert mx.mx_debug_last_gemm_launch() == (1, 1)
    finally:
        mx.mx_debug_set_gemm_variant(0)
    check_gemm(split1.cpu().numpy(), c_ref, s_ref, "f32")
    check_gemm(whole.cpu().numpy(), c_ref, s_ref, "f32")


def test_split_k_batched_dot(mx):
    # batch x small-M problems: the split covers every problem's tiles
    import torch
    rng = np.random.default_rng(12)
    B, M, N, K = 4, 40, 520, 2048
    a = rng.integers(0, 256, size=(B, M, K)).astype(np.uint8)
    bt = rng.integers(0, 256, size=(B, N, K)).astype(np.uint8)
    for x in (a, bt):
        x[(x & 0x7F) == 0x7F] = 0
    sa = rng.integers(112, 142, size=(B, M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(B, N, K // 32)).astype(np.uint8)
    got = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e4m3fn",
                                 "bf16", lhs_batch=(0,), rhs_batch=(0,))
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch()[1] > 1
    got = got.float().cpu().numpy()
    for i in range(B):
        c_ref, s_ref = orc.scaled_matmul(a[i], bt[i], sa[i], sb[i], "e4m3fn")
        check_gemm(got[i], c_ref, s_ref, "bf16")


def test_split_k_strided_output_rows(mx):
    # C written into a wider row pitch (ldc > N) and at an odd column count
    import torch
    M, N, K, ldc = 50, 250, 2048, 264
    a, bt, sa, sb = fp8_operands(M, N, K, "e4m3fn", seed=21)
    big = torch.full((M, ldc), -7.0, dtype=torch.float32, device="cuda")
    out = big[:, :N]
    mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e4m3fn", "f32",
                        out=out)
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch()[1] > 1
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(out.cpu().numpy(), c_ref, s_ref, "f32")
    assert torch.all(big[:, N:] == -7.0)   # nothing written past column N


@pytest.mark.parametrize("M", [16, 128])
def test_split_k_decode_shape_sampled(mx, M):
    # M x 8192 x 8192 (the small-M end of the ScaledMatmul workloads): every
    # row, sampled columns including both ends of every 256-column tile edge
    rng = np.random.default_rng(M)
    N = K = 8192
    a, bt, sa, sb = fp8_operands(M, N, K, "e4m3fn", seed=M)
    c = matmul(mx, a, bt, sa, sb, "e4m3fn", "bf16").float().cpu().numpy()
    assert mx.mx_debug_last_gemm_launch()[1] > 1
    cols = np.unique(np.concatenate([rng.choice(N, 96, replace=False), [0, 255, 256, 4095, 4096, N - 1]]))
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn", cols=cols)
    check_gemm(c[:, cols], c_ref, s_ref, "bf16")


def test_split_k_bounded_wait_times_out_without_fault(mx):
    """With loads suppressed, every CTA of every cluster gives up after 50 ms,
    records MX_ERR_TIMEOUT and still meets its cluster barriers; the context
    stays usable."""
    M, N, K = 64, 512, 4096
    a, bt, sa, sb = fp8_operands(M, N, K, "e4m3fn", seed=5)
    assert mx.mx_get_device_status() == 0
    mx.mx_debug_gemm_fault_injection(True, 50_000_000)
    try:
        matmul(mx, a, bt, sa, sb, "e4m3fn", "f32")
        assert mx.mx_debug_last_gemm_launch()[1] > 1
    finally:
        mx.mx_debug_gemm_fault_injection(False, 0)
    assert mx.mx_get_device_status() == mx.MX_ERR_TIMEOUT
    assert mx.mx_get_device_status() == 0
    c = matmul(mx, a, bt, sa, sb, "e4m3fn", "f32")
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(c.cpu().numpy(), c_ref, s_ref, "f32")


@pytest.mark.parametrize("fmt", ["e4m3fn", "e2m1"])
@pytest.mark.parametrize("M,N,K,kernel", [(1024, 1024, 4096, 1), (2048, 512, 4096, 1), (300, 1000, 4096, 1),
                                          (512, 4096, 2048, 2), (256, 8192, 1024, 2)])
def test_auto_choice_for_few_tile_problems(mx, fmt, M, N, K, kernel):
    # M > 128 whose 256 x 256 tiles fill at most a quarter of the pair
    # clusters runs on the 1-SM kernel with split-K; at half the clusters and
    # more, on the pair kernel.  Every element against the oracle.  FP4
    # stages hold 256 K elements, so FP4 runs at twice the K.
    if fmt == "e2m1":
        K *= 2
        a, bt, sa, sb = fp4_operands(M, N, K, seed=M + N + 1)
    else:
        a, bt, sa, sb = fp8_operands(M, N, K, fmt, seed=M + N + 1)
    c = matmul(mx, a, bt, sa, sb, fmt, "bf16")
    got_kernel, split = mx.mx_debug_last_gemm_launch()
    assert got_kernel == kernel
    assert split > 1 if kernel == 1 else split == 1
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, fmt)
    check_gemm(c.float().cpu().numpy(), c_ref, s_ref, "bf16")
