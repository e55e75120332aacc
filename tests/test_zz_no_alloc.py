"""mx_scaled_matmul_noalloc: the ScaledMatmul entry point for callers that
cannot allocate device memory (a plugin whose host runtime owns all device
memory and offers no allocator, or a path that must not call cudaMalloc).

It keeps its scratch in the library's fixed 4 MiB device array instead of a
caller workspace.  Its output is checked against the CPU oracle within the
matmul tolerance, on two calls in a row so the shared array is reused, and
at the size limit of the array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle as orc
from helpers import check_gemm, to_device_u8

MX_ERR_WORKSPACE = 7


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    # codes below 0x7C are finite in both e4m3fn and e5m2
    a = rng.integers(0, 0x7C, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0x80, 0xFC, size=(N, K)).astype(np.uint8)
    sa = rng.integers(112, 142, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(N, K // 32)).astype(np.uint8)
    return a, bt, sa, sb


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_consecutive_calls():
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import mx_fp8_microscaling_gb300 as mx

    for call, (M, N, K, fmt, out) in enumerate([(384, 512, 640, "e4m3fn", "f32"),
                                                 (256, 768, 1024, "e5m2", "bf16")]):
        a, bt, sa, sb = _operands(M, N, K, seed=call)
        da, dbt, dsa, dsb = (to_device_u8(v) for v in (a, bt, sa, sb))
        no_alloc = mx.mx_scaled_matmul_noalloc(da, dbt, dsa, dsb, fmt, out)
        with_ws = mx.mx_scaled_matmul(da, dbt, dsa, dsb, fmt, out)
        torch.cuda.synchronize()
        c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, fmt)
        check_gemm(no_alloc.float().cpu().numpy(), c_ref, s_ref, out)
        check_gemm(with_ws.float().cpu().numpy(), c_ref, s_ref, out)
    assert mx.mx_get_device_status() == 0


@pytest.mark.gpu
def test_noalloc_at_the_scratch_limit():
    """M = N = K = 8192 needs exactly the 4 MiB of repacked scales the array
    holds; sampled rows and columns against the oracle."""
    import torch
    import mx_fp8_microscaling_gb300 as mx

    M = N = K = 8192
    a, bt, sa, sb = _operands(M, N, K, seed=7)
    c = mx.mx_scaled_matmul_noalloc(*(to_device_u8(v) for v in (a, bt, sa, sb)), "e4m3fn", "bf16")
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    # the first and last row / column of tiles and random ones between
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], rng.integers(0, M, 26)]))
    cols = np.unique(np.concatenate([[0, 255, 256, N - 1], rng.integers(0, N, 28)]))
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn", rows=rows)
    check_gemm(c[torch.from_numpy(rows).cuda()].float().cpu().numpy(), c_ref, s_ref, "bf16")
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e4m3fn", cols=cols)
    check_gemm(c[:, torch.from_numpy(cols).cuda()].float().cpu().numpy(), c_ref, s_ref, "bf16")
    assert mx.mx_get_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(16384, 16384, 8192),   # twice the array
                                   (8193, 8192, 8192),     # one 128-row scale tile over
                                   (8192, 8192, 8224)])    # one 128-column scale tile over
def test_noalloc_rejects_problems_beyond_its_scratch(M, N, K):
    """Refused with MX_ERR_WORKSPACE before anything is read or launched (a
    host-side check: runs without a GPU)."""
    import mx_fp8_microscaling_gb300 as mx
    fake = ctypes.c_void_p(0x10000)
    st = mx.raw_library().mx_scaled_matmul_noalloc(fake, fake, fake, fake, mx.DTYPES["e4m3fn"], M, N, K,
                                                   mx.DTYPES["f32"], fake, N, None)
    assert st == MX_ERR_WORKSPACE
