"""Maximum sizes: tensors past 2^31 elements and 2^32 bytes, where 32-bit
index arithmetic anywhere in a kernel or in the host's size math would wrap.

Inputs are drawn on the device by torch's seeded generator (none comes from
this library's kernels); the oracle checks sampled row groups at the start,
the middle and the end of each tensor, read back to the host:
- QuantizeMX bf16 [40960, 65536] (2.7e9 elements) -> e4m3fn, 8x4 blocks along
  dim -2 and 1x32 blocks along dim -1: codes and scales bit-exact;
- dequantize e5m2 codes [40960, 65536] with 1x32 scales -> bf16: bit-exact;
- ScaledMatmul 65536 x 65536 x 256 -> bf16 (C holds 4.3e9 elements): within
  |C - C_ref| <= 1e-4 * sum_k |a_k b_k| + 1 bf16 ulp on sampled rows.
Each test holds at most about 17 GB on the device."""
import numpy as np
import pytest

import oracle as orc
from helpers import check_gemm

pytestmark = pytest.mark.gpu

R, C = 40960, 65536          # 2,684,354,560 elements
GROUPS = [0, R // 2 - 8, R - 8]


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


@pytest.fixture
def free_after():
    import torch
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _bf16_input(torch, seed):
    """N(0,1) x 2^U(-30,30) per row, bf16, on the device."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((R, C), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    e = torch.randint(-30, 31, (R, 1), generator=g, device="cuda", dtype=torch.int32)
    x.mul_(torch.pow(2.0, e.float()).to(torch.bfloat16))
    return x


def _rows_bits(torch, x, r0, n):
    return x[r0:r0 + n].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_quantize_8x4_past_2_31_elements(mx, free_after):
    import torch
    x = _bf16_input(torch, seed=1)
    q, s = mx.mx_quantize(x, "e4m3fn", geometry="8x4", dim=-2)
    torch.cuda.synchronize()
    assert tuple(q.shape) == (R, C) and tuple(s.shape) == (R // 8, C // 4)
    for r0 in GROUPS:
        want_q, want_s = orc.quantize(_rows_bits(torch, x, r0, 8), "bf16", "e4m3fn", geometry="8x4", dim=-2)
        assert np.array_equal(q[r0:r0 + 8].cpu().numpy(), want_q), r0
        assert np.array_equal(s[r0 // 8:r0 // 8 + 1].cpu().numpy(), want_s), r0


def test_quantize_1x32_past_2_31_elements(mx, free_after):
    import torch
    x = _bf16_input(torch, seed=2)
    q, s = mx.mx_quantize(x, "e4m3fn", geometry="1x32", dim=-1)
    torch.cuda.synchronize()
    assert tuple(s.shape) == (R, C // 32)
    for r0 in GROUPS + [R - 1]:
        want_q, want_s = orc.quantize(_rows_bits(torch, x, r0, 1), "bf16", "e4m3fn", geometry="1x32", dim=-1)
        assert np.array_equal(q[r0:r0 + 1].cpu().numpy(), want_q), r0
        assert np.array_equal(s[r0:r0 + 1].cpu().numpy(), want_s), r0


def test_dequantize_past_2_31_elements(mx, free_after):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    codes = torch.randint(0, 256, (R, C), generator=g, device="cuda", dtype=torch.uint8)
    scales = torch.randint(100, 155, (R, C // 32), generator=g, device="cuda", dtype=torch.uint8)
    out = mx.mx_dequantize(codes, scales, R, C, "e5m2", "bf16", geometry="1x32", dim=-1)
    torch.cuda.synchronize()
    for r0 in GROUPS + [R - 1]:
        want = orc.dequantize(codes[r0:r0 + 1].cpu().numpy(), scales[r0:r0 + 1].cpu().numpy(), 1, C, "e5m2",
                              geometry="1x32", dim=-1)
        with np.errstate(over="ignore", invalid="ignore"):
            want = torch.from_numpy(want.astype(np.float32)).to(torch.bfloat16).float().numpy()
        got = out[r0:r0 + 1].float().cpu().numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), r0
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), r0


def test_scaled_matmul_output_past_2_32_elements(mx, free_after):
    import torch
    M = N = 65536
    K = 256
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    a = torch.randint(0, 0x7F, (M, K), generator=g, device="cuda", dtype=torch.uint8)   # finite e4m3fn
    bt = torch.randint(0, 0x7F, (N, K), generator=g, device="cuda", dtype=torch.uint8)
    bt[N // 2:] |= 0x80                                                                  # negative half
    sa = torch.randint(120, 135, (M, K // 32), generator=g, device="cuda", dtype=torch.uint8)
    sb = torch.randint(120, 135, (N, K // 32), generator=g, device="cuda", dtype=torch.uint8)
    c = mx.mx_scaled_matmul(a, bt, sa, sb, "e4m3fn", "bf16")
    torch.cuda.synchronize()
    assert c.numel() == M * N
    bt_h, sb_h = bt.cpu().numpy(), sb.cpu().numpy()
    rows = np.array([0, 1, 255, 256, M // 2 + 3, M - 129, M - 1])
    cols = np.concatenate([np.arange(0, 64), np.arange(N // 2 - 32, N // 2 + 32), np.arange(N - 64, N)])
    a_h, sa_h = a[rows].cpu().numpy(), sa[rows].cpu().numpy()
    c_ref, s_ref = orc.scaled_matmul(a_h, bt_h, sa_h, sb_h, "e4m3fn", cols=cols)
    got = c[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    check_gemm(got, c_ref, s_ref, "bf16")
