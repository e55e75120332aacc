"""mx_scaled_matmul_noalloc: the ScaledMatmul entry point for callers that
cannot allocate device memory (a plugin whose host runtime owns all device
memory and offers no allocator, or a path that must not call cudaMalloc).

It keeps its scratch in the library's fixed 4 MiB device array instead of a
caller workspace.  Its output must agree with mx_scaled_matmul (which takes a
workspace) within the matmul tolerance, on two calls in a row so the shared
array is reused.  This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle as orc
from helpers import check_gemm, to_device_u8

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    # codes below 0x7C are finite in both e4m3fn and e5m2
    a = rng.integers(0, 0x7C, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0x80, 0xFC, size=(N, K)).astype(np.uint8)
    sa = rng.integers(112, 142, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(N, K // 32)).astype(np.uint8)
    return a, bt, sa, sb


def test_noalloc_matches_workspace_entry_point():
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import mx_fp8_microscaling_gb300 as mx

    for call, (M, N, K, fmt, out) in enumerate([(384, 512, 640, "e4m3fn", "f32"),
                                                 (256, 768, 1024, "e5m2", "bf16")]):
        a, bt, sa, sb = _operands(M, N, K, seed=call)
        da, dbt, dsa, dsb = (to_device_u8(v) for v in (a, bt, sa, sb))
        with_ws = mx.mx_scaled_matmul(da, dbt, dsa, dsb, fmt, out)
        no_alloc = mx.mx_scaled_matmul_noalloc(da, dbt, dsa, dsb, fmt, out)
        torch.cuda.synchronize()
        _, s_ref = orc.scaled_matmul(a, bt, sa, sb, fmt)
        ref = with_ws.float().cpu().numpy().astype(np.float64)
        check_gemm(no_alloc.float().cpu().numpy(), ref, s_ref, out)
    assert mx.mx_get_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    import ctypes

    import mx_fp8_microscaling_gb300 as mx
    # 16384 x 16384 x 8192 needs 2 x 4 MiB of repacked scales, over the 4 MiB
    # array: refused before anything is read or launched
    fake = ctypes.c_void_p(0x10000)
    st = mx.raw_library().mx_scaled_matmul_noalloc(fake, fake, fake, fake, mx.DTYPES["e4m3fn"], 16384, 16384,
                                                   8192, mx.DTYPES["f32"], fake, 16384, None)
    assert st == 7  # MX_ERR_WORKSPACE
