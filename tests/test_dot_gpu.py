"""General block-scaled dot (batch / contracting dimension numbers) on the GPU
against the oracle's block_scaled_dot.

Codes are random finite FP8 codes and scales random E8M0 values; the kernel
result must satisfy |C - C_ref| <= 1e-4 * sum_k |a_k b_k| (+ 1 bf16 ulp of
C_ref for bf16 output) on every element."""
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


def operand(rng, shape, axis, fmt):
    codes = rng.integers(0, 256, size=shape).astype(np.uint8)
    bad = (codes & 0x7F) == 0x7F if fmt == "e4m3fn" else (codes & 0x7F) >= 0x7C
    codes[bad] = 0   # no NaN / Inf codes
    sshape = list(shape)
    sshape[axis] //= 32
    scale = rng.integers(112, 142, size=sshape).astype(np.uint8)
    return codes, scale


def run(mx, lshape, rshape, lb, rb, lc, rc, fmt, out_dtype, seed):
    import torch
    rng = np.random.default_rng(seed)
    lhs, ls = operand(rng, lshape, lc, fmt)
    rhs, rs = operand(rng, rshape, rc, fmt)
    want, s = orc.block_scaled_dot(lhs, rhs, ls, rs, fmt, lhs_batch=lb, rhs_batch=rb, lhs_contract=(lc,),
                                   rhs_contract=(rc,))
    got = mx.mx_block_scaled_dot(to_device_u8(lhs), to_device_u8(rhs), to_device_u8(ls), to_device_u8(rs), fmt,
                                 out_dtype, lhs_batch=lb, rhs_batch=rb, lhs_contract=(lc,), rhs_contract=(rc,))
    torch.cuda.synchronize()
    assert tuple(got.shape) == want.shape
    check_gemm(got.float().cpu().numpy(), want, s, out_dtype)


# (lhs shape, rhs shape, lhs batch, rhs batch, lhs contract, rhs contract)
CASES = {
    "canonical_pair_kernel": ((3, 200, 256), (3, 300, 256), (0,), (0,), 2, 2),
    "rhs_k_by_n": ((2, 64, 96), (2, 96, 136), (0,), (0,), 2, 1),
    # 16-byte aligned rows, both tile axes cut by the edge at multiples of 16
    # bytes (N = 208 = 128 + 80, K = 160 = 128 + 32): the transposing copy's
    # partial tiles on its shared-memory path
    "rhs_k_by_n_partial_tiles": ((2, 64, 160), (2, 160, 208), (0,), (0,), 2, 1),
    "batch_in_middle": ((130, 2, 64), (2, 72, 64), (1,), (0,), 2, 2),
    "two_batch_dims_reordered": ((2, 3, 40, 64), (3, 2, 64, 48), (0, 1), (1, 0), 3, 2),
    "several_free_dims": ((2, 5, 7, 64), (64, 3, 40), (), (), 3, 0),
    "lhs_k_major_axis0": ((128, 96), (160, 128), (), (), 0, 1),
    "both_k_leading": ((64, 4, 150), (64, 4, 33), (1,), (1,), 0, 0),
}


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_block_scaled_dot_matches_oracle(mx, name, fmt, out_dtype):
    lshape, rshape, lb, rb, lc, rc = CASES[name]
    run(mx, lshape, rshape, lb, rb, lc, rc, fmt, out_dtype, seed=sorted(CASES).index(name))


def test_batch_of_one_equals_scaled_matmul(mx):
    # [1, M, K] x [1, N, K]: the same kernel and bits as mx_scaled_matmul
    import torch
    rng = np.random.default_rng(3)
    M, N, K = 300, 260, 512
    a, sa = operand(rng, (M, K), 1, "e4m3fn")
    bt, sb = operand(rng, (N, K), 1, "e4m3fn")
    ref = mx.mx_scaled_matmul(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e4m3fn",
                              "f32")
    got = mx.mx_block_scaled_dot(to_device_u8(a[None]), to_device_u8(bt[None]), to_device_u8(sa[None]),
                                 to_device_u8(sb[None]), "e4m3fn", "f32", lhs_batch=(0,), rhs_batch=(0,))
    torch.cuda.synchronize()
    assert torch.equal(got[0].view(torch.int32), ref.view(torch.int32))


def test_batches_are_independent(mx):
    # each problem of a batch equals the same problem run alone (bit for bit:
    # same tiles, same accumulation order)
    import torch
    rng = np.random.default_rng(5)
    B, M, N, K = 5, 140, 200, 320
    a, sa = operand(rng, (B, M, K), 2, "e5m2")
    bt, sb = operand(rng, (B, N, K), 2, "e5m2")
    got = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(bt), to_device_u8(sa), to_device_u8(sb), "e5m2",
                                 "bf16", lhs_batch=(0,), rhs_batch=(0,))
    for b in range(B):
        one = mx.mx_scaled_matmul(to_device_u8(a[b]), to_device_u8(bt[b]), to_device_u8(sa[b]), to_device_u8(sb[b]),
                                  "e5m2", "bf16")
        torch.cuda.synchronize()
        assert torch.equal(got[b].view(torch.int16), one.view(torch.int16)), b


def test_empty_batch_and_empty_free_dims(mx):
    import torch
    for lshape, rshape in [((0, 8, 64), (0, 16, 64)), ((2, 0, 64), (2, 16, 64)), ((2, 8, 64), (2, 0, 64))]:
        lhs = torch.zeros(lshape, dtype=torch.uint8, device="cuda")
        rhs = torch.zeros(rshape, dtype=torch.uint8, device="cuda")
        ls = torch.zeros(lshape[:-1] + (2,), dtype=torch.uint8, device="cuda")
        rs = torch.zeros(rshape[:-1] + (2,), dtype=torch.uint8, device="cuda")
        out = mx.mx_block_scaled_dot(lhs, rhs, ls, rs, "e4m3fn", "f32", lhs_batch=(0,), rhs_batch=(0,))
        torch.cuda.synchronize()
        assert tuple(out.shape) == (lshape[0], lshape[1], rshape[1])


def test_large_batched_sampled(mx):
    # 8 problems of 1024 x 1024 x 1024 (rhs stored [B, K, N]: the transposing
    # copy runs at full size); the oracle checks sampled rows and columns
    import torch
    rng = np.random.default_rng(9)
    B, M, N, K = 8, 1024, 1024, 1024
    a, sa = operand(rng, (B, M, K), 2, "e4m3fn")
    b, sb = operand(rng, (B, K, N), 1, "e4m3fn")
    got = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(b), to_device_u8(sa), to_device_u8(sb), "e4m3fn",
                                 "bf16", lhs_batch=(0,), rhs_batch=(0,), lhs_contract=(2,), rhs_contract=(1,))
    torch.cuda.synchronize()
    got = got.float().cpu().numpy()
    rows = rng.choice(M, 24, replace=False)
    cols = rng.choice(N, 24, replace=False)
    for bb in (0, 3, 7):
        bt = np.ascontiguousarray(b[bb].T)
        sbt = np.ascontiguousarray(sb[bb].T)
        C, S = orc.scaled_matmul(a[bb], bt, sa[bb], sbt, "e4m3fn", rows=rows)
        check_gemm(got[bb][rows], C, S, "bf16")
        C, S = orc.scaled_matmul(a[bb], bt, sa[bb], sbt, "e4m3fn", cols=cols)
        check_gemm(got[bb][:, cols], C, S, "bf16")
