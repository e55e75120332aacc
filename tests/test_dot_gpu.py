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


# ---------------------------------------------------------------- MN-major operands
#
# An FP8 operand stored [batch, K, rows] (the contracting axis before the free
# axes) is read in place as MN-major tiles, with no transposing copy, when its
# rows are a multiple of 16 bytes, by either GEMM kernel.  Each case runs
# under a forced kernel (small shapes) or the automatic choice (large ones),
# checks which operands were read in place, and compares every element with
# the oracle.

def run_major(mx, lshape, rshape, lb, rb, lc, rc, fmt, out_dtype, seed, variant=2):
    import torch
    rng = np.random.default_rng(seed)
    lhs, ls = operand(rng, lshape, lc, fmt)
    rhs, rs = operand(rng, rshape, rc, fmt)
    want, s = orc.block_scaled_dot(lhs, rhs, ls, rs, fmt, lhs_batch=lb, rhs_batch=rb, lhs_contract=(lc,),
                                   rhs_contract=(rc,))
    mx.mx_debug_set_gemm_variant(variant)
    try:
        got = mx.mx_block_scaled_dot(to_device_u8(lhs), to_device_u8(rhs), to_device_u8(ls), to_device_u8(rs), fmt,
                                     out_dtype, lhs_batch=lb, rhs_batch=rb, lhs_contract=(lc,), rhs_contract=(rc,))
        torch.cuda.synchronize()
    finally:
        mx.mx_debug_set_gemm_variant(0)
    check_gemm(got.float().cpu().numpy(), want, s, out_dtype)
    return got, mx.mx_debug_last_gemm_launch(), mx.mx_debug_last_gemm_operands()


MAJOR_CASES = {
    # name: (lhs shape, rhs shape, lb, rb, lc, rc, expected (a_mn, b_mn))
    "rhs_kn": ((2, 256, 512), (2, 512, 384), (0,), (0,), 2, 1, (0, 1)),
    # N = 208 = 128 + 80 and K = 160 = 128 + 32: both edges of the MN-major
    # tile read zeros past the operand
    "rhs_kn_ragged": ((2, 200, 160), (2, 160, 208), (0,), (0,), 2, 1, (0, 1)),
    "rhs_kn_short_k": ((1, 300, 96), (1, 96, 48), (0,), (0,), 2, 1, (0, 1)),
    "lhs_km": ((3, 512, 272), (3, 136, 512), (0,), (0,), 1, 2, (1, 0)),
    "both_mn": ((2, 384, 400), (2, 384, 144), (0,), (0,), 1, 1, (1, 1)),
    "no_batch_both_mn": ((288, 336), (288, 528), (), (), 0, 0, (1, 1)),
    "two_batch_dims_both_mn": ((2, 3, 256, 160), (2, 3, 256, 96), (0, 1), (0, 1), 2, 2, (1, 1)),
    "two_batch_dims_rhs_kn": ((2, 3, 160, 256), (2, 3, 256, 96), (0, 1), (0, 1), 3, 2, (0, 1)),
    "two_free_dims_rhs_kn": ((2, 160, 256), (2, 256, 3, 32), (0,), (0,), 2, 1, (0, 1)),
    # rows not a multiple of 16 bytes: copied into [batch, rows, K] instead
    "rhs_kn_odd_rows": ((2, 256, 256), (2, 256, 200), (0,), (0,), 2, 1, (0, 0)),
    "rhs_kn_rows_8": ((2, 256, 256), (2, 256, 8), (0,), (0,), 2, 1, (0, 0)),
}


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("name", sorted(MAJOR_CASES))
def test_mn_major_operands_match_oracle(mx, name, fmt, out_dtype):
    lshape, rshape, lb, rb, lc, rc, majors = MAJOR_CASES[name]
    _, launch, got_majors = run_major(mx, lshape, rshape, lb, rb, lc, rc, fmt, out_dtype,
                                      seed=100 + sorted(MAJOR_CASES).index(name))
    assert launch[0] == 2
    assert got_majors == majors


def test_mn_major_equals_copied_operand_bitwise(mx):
    # the same products from the same codes and scales: reading [B, K, N] in
    # place gives the bits of the [B, N, K] copy
    import torch
    rng = np.random.default_rng(41)
    B, M, N, K = 3, 384, 272, 640
    a, sa = operand(rng, (B, M, K), 2, "e4m3fn")
    b_kn, sb_kn = operand(rng, (B, K, N), 1, "e4m3fn")
    b_nk = np.ascontiguousarray(b_kn.transpose(0, 2, 1))
    sb_nk = np.ascontiguousarray(sb_kn.transpose(0, 2, 1))
    mx.mx_debug_set_gemm_variant(2)
    try:
        in_place = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(b_kn), to_device_u8(sa), to_device_u8(sb_kn),
                                          "e4m3fn", "f32", lhs_batch=(0,), rhs_batch=(0,), rhs_contract=(1,))
        assert mx.mx_debug_last_gemm_operands() == (0, 1)
        copied = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(b_nk), to_device_u8(sa), to_device_u8(sb_nk),
                                        "e4m3fn", "f32", lhs_batch=(0,), rhs_batch=(0,))
        assert mx.mx_debug_last_gemm_operands() == (0, 0)
        torch.cuda.synchronize()
    finally:
        mx.mx_debug_set_gemm_variant(0)
    assert torch.equal(in_place.view(torch.int32), copied.view(torch.int32))


ONE_SM_CASES = {
    # M <= 128: the 1-SM kernel, split K over a cluster where the shape
    # calls for it; its MN-major B tile is two 128-row atom columns
    "rhs_kn_split": ((2, 64, 2048), (2, 2048, 512), (0,), (0,), 2, 1, (0, 1)),
    "rhs_kn_ragged_n": ((3, 100, 1024), (3, 1024, 208), (0,), (0,), 2, 1, (0, 1)),
    "lhs_km": ((2, 1024, 48), (2, 300, 1024), (0,), (0,), 1, 2, (1, 0)),
    "both_mn_k_tail": ((1, 160, 128), (1, 160, 400), (0,), (0,), 1, 1, (1, 1)),
}


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "no_split"])
@pytest.mark.parametrize("name", sorted(ONE_SM_CASES))
def test_mn_major_on_the_one_sm_kernel(mx, name, variant, out_dtype):
    lshape, rshape, lb, rb, lc, rc, majors = ONE_SM_CASES[name]
    _, launch, got = run_major(mx, lshape, rshape, lb, rb, lc, rc, "e4m3fn", out_dtype,
                               seed=200 + sorted(ONE_SM_CASES).index(name), variant=variant)
    assert launch[0] == 1
    assert launch[1] == 1 if variant == 3 else launch[1] >= 1
    assert got == majors


def test_mn_major_one_sm_split_equals_copied_operand_bitwise(mx):
    # the split-K slices add the same partial products in the same order
    # whichever way B is stored
    import torch
    rng = np.random.default_rng(43)
    B, M, N, K = 2, 96, 768, 4096
    a, sa = operand(rng, (B, M, K), 2, "e5m2")
    b_kn, sb_kn = operand(rng, (B, K, N), 1, "e5m2")
    b_nk = np.ascontiguousarray(b_kn.transpose(0, 2, 1))
    sb_nk = np.ascontiguousarray(sb_kn.transpose(0, 2, 1))
    in_place = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(b_kn), to_device_u8(sa), to_device_u8(sb_kn),
                                      "e5m2", "f32", lhs_batch=(0,), rhs_batch=(0,), rhs_contract=(1,))
    assert mx.mx_debug_last_gemm_operands() == (0, 1)
    kernel, split = mx.mx_debug_last_gemm_launch()
    assert kernel == 1 and split > 1
    copied = mx.mx_block_scaled_dot(to_device_u8(a), to_device_u8(b_nk), to_device_u8(sa), to_device_u8(sb_nk),
                                    "e5m2", "f32", lhs_batch=(0,), rhs_batch=(0,))
    assert mx.mx_debug_last_gemm_operands() == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(in_place.view(torch.int32), copied.view(torch.int32))
    want, s = orc.block_scaled_dot(a, b_kn, sa, sb_kn, "e5m2", lhs_batch=(0,), rhs_batch=(0,), rhs_contract=(1,))
    check_gemm(in_place.cpu().numpy(), want, s, "f32")


def test_mn_major_full_tiles_sampled(mx):
    # 8 x 1024^3 with rhs [B, K, N] and lhs [B, K, M]: enough 256 x 256 tiles
    # for whole rounds (no split tail) on the automatic choice; sampled rows
    # and columns of three problems against the oracle
    import torch
    rng = np.random.default_rng(19)
    B, M, N, K = 8, 1024, 1024, 1024
    a_km, sa_km = operand(rng, (B, K, M), 1, "e4m3fn")
    b_kn, sb_kn = operand(rng, (B, K, N), 1, "e4m3fn")
    got = mx.mx_block_scaled_dot(to_device_u8(a_km), to_device_u8(b_kn), to_device_u8(sa_km), to_device_u8(sb_kn),
                                 "e4m3fn", "bf16", lhs_batch=(0,), rhs_batch=(0,), lhs_contract=(1,),
                                 rhs_contract=(1,))
    torch.cuda.synchronize()
    assert mx.mx_debug_last_gemm_launch()[0] == 2
    assert mx.mx_debug_last_gemm_operands() == (1, 1)
    got = got.float().cpu().numpy()
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], rng.choice(M, 18, replace=False)]))
    cols = np.unique(np.concatenate([[0, 127, 128, 255, 256, N - 1], rng.choice(N, 18, replace=False)]))
    for bb in (0, 5, 7):
        a = np.ascontiguousarray(a_km[bb].T)
        sa = np.ascontiguousarray(sa_km[bb].T)
        bt = np.ascontiguousarray(b_kn[bb].T)
        sbt = np.ascontiguousarray(sb_kn[bb].T)
        C, S = orc.scaled_matmul(a, bt, sa, sbt, "e4m3fn", rows=rows)
        check_gemm(got[bb][rows], C, S, "bf16")
        C, S = orc.scaled_matmul(a, bt, sa, sbt, "e4m3fn", cols=cols)
        check_gemm(got[bb][:, cols], C, S, "bf16")
