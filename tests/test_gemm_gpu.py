"""ScaledMatmul on the GPU (through the C-ABI) against the CPU oracle within
|C - C_ref| <= 1e-4 * sum_k |a_k b_k| (+ 1 bf16 ulp of C_ref for bf16
output).  Operands are quantized by the oracle on the host and copied to the
device, so no oracle input comes from the GPU; the pipeline tests also check
the GPU quantizer bit for bit."""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc
from helpers import check_gemm, sf_pack, to_device_bits, to_device_u8

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


@pytest.fixture(params=[1, 2, 3], ids=["1sm", "2sm", "1sm_nosplit"])
def variant(request, mx):
    """Run a test on the 1-SM kernel (split-K where the shape calls for it),
    on the 2-SM pair kernel and on the 1-SM kernel with split-K disabled."""
    mx.mx_debug_set_gemm_variant(request.param)
    yield request.param
    mx.mx_debug_set_gemm_variant(0)


def _random_operands(M, N, K, fmt, seed, scale_lo=112, scale_hi=142):
    rng = np.random.default_rng(seed)
    bad = {"e4m3fn": lambda c: (c & 0x7F) == 0x7F, "e5m2": lambda c: (c & 0x7F) >= 0x7C}[fmt]
    a = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    a[bad(a)] = 0x38
    bt[bad(bt)] = 0xB8
    sa = rng.integers(scale_lo, scale_hi, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(scale_lo, scale_hi, size=(N, K // 32)).astype(np.uint8)
    return a, bt, sa, sb


def _gpu_matmul(mx, a, bt, sa, sb, fmt, out_dtype, sf_layout=False):
    import torch
    sa_d = to_device_u8(sf_pack(sa) if sf_layout else sa)
    sb_d = to_device_u8(sf_pack(sb) if sf_layout else sb)
    c = mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), sa_d, sb_d, fmt, out_dtype,
                            scales_are_sf_layout=sf_layout, K=a.shape[1])
    torch.cuda.synchronize()
    return c.float().cpu().numpy()


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512), (384, 768, 1024),
                                   (200, 300, 96), (1, 1, 32), (130, 260, 160), (512, 256, 4096),
                                   (640, 1280, 256), (100, 700, 64)])
def test_matmul_matches_oracle(mx, variant, fmt, out_dtype, M, N, K):
    a, bt, sa, sb = _random_operands(M, N, K, fmt, seed=M * 7 + N + K)
    c = _gpu_matmul(mx, a, bt, sa, sb, fmt, out_dtype)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, fmt)
    check_gemm(c, c_ref, s_ref, out_dtype, TOL)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(2560, 2048, 256), (512, 1024, 256), (256, 200, 64), (768, 640, 384)])
def test_matmul_split_tail_round(mx, out_dtype, M, N, K):
    # the pair kernel runs a last round that fits in half the clusters as
    # 256 x 128 half tiles (80 tiles on 74-76 clusters; few-tile problems run
    # entirely as halves): every element against the oracle
    mx.mx_debug_set_gemm_variant(2)
    try:
        a, bt, sa, sb = _random_operands(M, N, K, "e4m3fn", seed=M + N + K)
        c = _gpu_matmul(mx, a, bt, sa, sb, "e4m3fn", out_dtype)
    finally:
        mx.mx_debug_set_gemm_variant(0)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(c, c_ref, s_ref, out_dtype, TOL)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 128), (4096, 8192, 256)])
def test_matmul_accumulator_handoff_many_short_tiles(mx, out_dtype, M, N, K):
    """Many pair tiles per cluster (3.5 and 7) of one or two K stages, so
    rank 0's stores are not paced and the accumulator changes hands every
    few microseconds: an MMA that overwrote the accumulator before rank 1's
    epilogue had read it would show in some tile.  Every element against
    the oracle."""
    mx.mx_debug_set_gemm_variant(2)
    try:
        a, bt, sa, sb = _random_operands(M, N, K, "e4m3fn", seed=M + N + K + 1)
        c = _gpu_matmul(mx, a, bt, sa, sb, "e4m3fn", out_dtype)
    finally:
        mx.mx_debug_set_gemm_variant(0)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(c, c_ref, s_ref, out_dtype, TOL)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_matmul_sf_layout_scales(mx, variant, fmt):
    M, N, K = 256, 512, 384
    a, bt, sa, sb = _random_operands(M, N, K, fmt, seed=3)
    c = _gpu_matmul(mx, a, bt, sa, sb, fmt, "f32", sf_layout=True)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, fmt)
    check_gemm(c, c_ref, s_ref, "f32", TOL)


def test_matmul_distinct_scales_per_block(mx, variant):
    # every (row, K-block) scale different and every product positive, so a
    # scale applied to the wrong row or K block shows up as a large error
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(4)
    a = np.full((M, K), 0x38, np.uint8)     # 1.0
    bt = np.full((N, K), 0x38, np.uint8)
    sa = rng.integers(100, 150, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(100, 150, size=(N, K // 32)).astype(np.uint8)
    c = _gpu_matmul(mx, a, bt, sa, sb, "e4m3fn", "f32")
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(c, c_ref, s_ref, "f32", TOL)


def test_matmul_strided_output(mx, variant):
    import torch
    M, N, K = 256, 256, 256
    a, bt, sa, sb = _random_operands(M, N, K, "e4m3fn", seed=8)
    big = torch.full((M, N + 64), -7.0, dtype=torch.float32, device="cuda")
    out = big[:, :N]
    mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e4m3fn", "f32",
                        out=out)
    torch.cuda.synchronize()
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(out.cpu().numpy(), c_ref, s_ref, "f32", TOL)
    assert torch.all(big[:, N:] == -7.0)


@pytest.mark.parametrize("out_dtype,pad,offset", [("bf16", 8, 8), ("f32", 4, 4), ("bf16", 8, 0)])
def test_matmul_rows_16_byte_not_32_byte_aligned(mx, variant, out_dtype, pad, offset):
    # rows 16-byte aligned but alternately 32-byte aligned (and a base 16
    # bytes past a 32-byte boundary): both vector store widths run
    import torch
    M, N, K = 256, 384, 256
    a, bt, sa, sb = _random_operands(M, N, K, "e5m2", seed=12)
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    big = torch.full((M, N + pad + offset), -3.0, dtype=dt, device="cuda")
    out = big[:, offset:offset + N]
    mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e5m2", out_dtype,
                        out=out)
    torch.cuda.synchronize()
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e5m2")
    check_gemm(out.float().cpu().numpy(), c_ref, s_ref, out_dtype, TOL)
    assert torch.all(big[:, :offset] == -3.0) and torch.all(big[:, offset + N:] == -3.0)


def test_pipeline_256(mx):
    """MX-FP8 pipeline at M=N=K=256, seed 0: A and Bt (bf16, N(0,1) * 2^U(-20,20)
    per 32-block) quantized along K to e4m3fn on the GPU, then ScaledMatmul to
    f32.  The GPU quantizer must equal the oracle's bit for bit, and C must be
    within tolerance of the oracle pipeline."""
    import torch
    a_bits, b_bits = syn.pipeline_operands(256, 256, 256, seed=0)
    qa, sa = orc.quantize(a_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    qb, sb = orc.quantize(b_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    ga, gsa = mx.mx_quantize(to_device_bits(a_bits, "bf16"), "e4m3fn", geometry="1x32", dim=-1)
    gb, gsb = mx.mx_quantize(to_device_bits(b_bits, "bf16"), "e4m3fn", geometry="1x32", dim=-1)
    c = mx.mx_scaled_matmul(ga, gb, gsa, gsb, "e4m3fn", "f32")
    torch.cuda.synchronize()
    assert np.array_equal(ga.cpu().numpy(), qa) and np.array_equal(gsa.cpu().numpy(), sa)
    assert np.array_equal(gb.cpu().numpy(), qb) and np.array_equal(gsb.cpu().numpy(), sb)
    c_ref, s_ref = orc.scaled_matmul(qa, qb, sa, sb, "e4m3fn")
    check_gemm(c.cpu().numpy(), c_ref, s_ref, "f32", TOL)


def _sample_rows_cols(M, N, n=128, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(M, n, replace=False), [0, M - 1, 127, 128]]))
    cols = np.unique(np.concatenate([rng.choice(N, n, replace=False), [0, N - 1, 255, 256]]))
    return rows, cols


@pytest.mark.parametrize("fmt,out_dtype", [("e4m3fn", "bf16"), ("e5m2", "f32")])
def test_matmul_8192_sampled(mx, fmt, out_dtype):
    """ScaledMatmul at M=N=K=8192 (operands: QuantizeMX along K of bf16
    N(0,1) * 2^U(-8,8) per row), checked on 128+ full rows and 128+ full
    columns, covering tile boundaries."""
    import torch
    M = N = K = 8192
    a_bits, b_bits = syn.gemm_operands(M, N, K, seed=0)
    qa, sa = orc.quantize(a_bits, "bf16", fmt, geometry="1x32", dim=-1)
    qb, sb = orc.quantize(b_bits, "bf16", fmt, geometry="1x32", dim=-1)
    c = mx.mx_scaled_matmul(to_device_u8(qa), to_device_u8(qb), to_device_u8(sa), to_device_u8(sb), fmt,
                            out_dtype)
    torch.cuda.synchronize()
    c = c.float().cpu().numpy()
    rows, cols = _sample_rows_cols(M, N)
    c_ref, s_ref = orc.scaled_matmul(qa, qb, sa, sb, fmt, rows=rows)
    check_gemm(c[rows], c_ref, s_ref, out_dtype, TOL)
    c_ref, s_ref = orc.scaled_matmul(qa, qb, sa, sb, fmt, cols=cols)
    check_gemm(c[:, cols], c_ref, s_ref, out_dtype, TOL)


def test_fused_small(mx):
    import torch
    M, N, K = 384, 512, 512
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=2)
    qw, sw = orc.quantize(w_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    qx, sx = orc.quantize(x_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    c = mx.mx_fused_quantize_matmul(to_device_bits(x_bits, "bf16"), to_device_u8(qw), to_device_u8(sf_pack(sw)),
                                    "e4m3fn", "bf16")
    torch.cuda.synchronize()
    c_ref, s_ref = orc.scaled_matmul(qx, qw, sx, sw, "e4m3fn")
    check_gemm(c.float().cpu().numpy(), c_ref, s_ref, "bf16", TOL)


def test_fused_full_size_sampled(mx):
    """Fused activation quantize + ScaledMatmul: X[16384, 8192] bf16 (0.1%
    outliers x100) quantized along K to e4m3fn, times a pre-quantized e4m3fn
    weight W[8192, 28672] (N(0, 0.02)), bf16 out [16384, 28672]."""
    import torch
    M, N, K = 16384, 28672, 8192
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=0)
    qw, sw = orc.quantize(w_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    qx, sx = orc.quantize(x_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
    c = mx.mx_fused_quantize_matmul(to_device_bits(x_bits, "bf16"), to_device_u8(qw), to_device_u8(sf_pack(sw)),
                                    "e4m3fn", "bf16")
    torch.cuda.synchronize()
    rows, cols = _sample_rows_cols(M, N, n=96)
    c_rows = c[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    c_ref, s_ref = orc.scaled_matmul(qx, qw, sx, sw, "e4m3fn", rows=rows)
    check_gemm(c_rows, c_ref, s_ref, "bf16", TOL)
    c_cols = c[:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    c_ref, s_ref = orc.scaled_matmul(qx, qw, sx, sw, "e4m3fn", cols=cols)
    check_gemm(c_cols, c_ref, s_ref, "bf16", TOL)


def test_bounded_wait_times_out_without_fault(mx, variant):
    """With loads suppressed, every wait of the GEMM runs out after 50 ms; the
    kernel records MX_ERR_TIMEOUT, frees its tensor memory and returns, and the
    context stays usable."""
    import torch
    a, bt, sa, sb = _random_operands(256, 256, 256, "e4m3fn", seed=5)
    assert mx.mx_get_device_status() == 0
    mx.mx_debug_gemm_fault_injection(True, 50_000_000)
    try:
        _gpu_matmul(mx, a, bt, sa, sb, "e4m3fn", "f32")
    finally:
        mx.mx_debug_gemm_fault_injection(False, 0)
    assert mx.mx_get_device_status() == mx.MX_ERR_TIMEOUT
    assert mx.mx_get_device_status() == 0           # read clears it
    c = _gpu_matmul(mx, a, bt, sa, sb, "e4m3fn", "f32")   # the context still works
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn")
    check_gemm(c, c_ref, s_ref, "f32", TOL)
    torch.cuda.synchronize()
