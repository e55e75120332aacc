"""MXFP4 ScaledMatmul (packed e2m1 operands, one E8M0 per 32 along K) on the
GPU against the oracle, |C - C_ref| <= 1e-4 * sum_k |a_k b_k| (+ 1 bf16 ulp
of C_ref for bf16 output).

Operands are random e2m1 codes packed on the host with the oracle's nibble
packing in the tensor-core order (lane stride 1 = identity, parity 1: element
2i in the low nibble); the oracle sees the unpacked codes."""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc
from helpers import check_gemm, to_device_bits, to_device_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


@pytest.fixture(params=[1, 2], ids=["1sm", "2sm"])
def variant(request, mx):
    mx.mx_debug_set_gemm_variant(request.param)
    yield request.param
    mx.mx_debug_set_gemm_variant(0)


def pack(codes):
    rows, k = codes.shape
    return orc.pack_nibbles(codes.reshape(-1), lane_stride=1, nibble_parity=1).reshape(rows, k // 2)


def operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sa = rng.integers(112, 142, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(N, K // 32)).astype(np.uint8)
    return a, bt, sa, sb


def gpu_matmul(mx, a, bt, sa, sb, out_dtype):
    import torch
    c = mx.mx_scaled_matmul(to_device_u8(pack(a)), to_device_u8(pack(bt)), to_device_u8(sa), to_device_u8(sb),
                            "e2m1", out_dtype, K=a.shape[1])
    torch.cuda.synchronize()
    return c.float().cpu().numpy()


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (300, 260, 512), (256, 256, 32),
                                   (200, 136, 160), (130, 260, 384), (1, 1, 64), (512, 256, 4096),
                                   (100, 700, 96)])
def test_fp4_matmul_matches_oracle(mx, variant, out_dtype, M, N, K):
    a, bt, sa, sb = operands(M, N, K, seed=M * 5 + N + K)
    c = gpu_matmul(mx, a, bt, sa, sb, out_dtype)
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e2m1")
    check_gemm(c, c_ref, s_ref, out_dtype)


def test_fp4_distinct_scales_per_block(mx, variant):
    # every (row, K-block) scale different and every product positive, so a
    # scale taken from the wrong row, K block or half of a scale column shows
    M, N, K = 256, 256, 1024
    rng = np.random.default_rng(4)
    a = rng.integers(1, 8, size=(M, K)).astype(np.uint8)
    bt = rng.integers(1, 8, size=(N, K)).astype(np.uint8)
    sa = (100 + (np.arange(M)[:, None] * 3 + np.arange(K // 32)[None, :] * 7) % 50).astype(np.uint8)
    sb = (100 + (np.arange(N)[:, None] * 5 + np.arange(K // 32)[None, :] * 11) % 50).astype(np.uint8)
    c = gpu_matmul(mx, a, bt, sa, sb, "f32")
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e2m1")
    check_gemm(c, c_ref, s_ref, "f32")


def test_fp4_pipeline_quantize_then_matmul(mx, variant):
    # bf16 operands quantized on the GPU to e2m1 in the tensor-core packing,
    # checked bit for bit against the oracle's quantizer, then multiplied
    import torch
    M, N, K = 256, 384, 512
    a_bits, b_bits = syn.gemm_operands(M, N, K, seed=2)
    cfg = dict(geometry="1x32", dim=-1, fp4_lane_stride=1, fp4_nibble_parity=1)
    qa, sa = mx.mx_quantize(to_device_bits(a_bits, "bf16"), "e2m1", **cfg)
    qb, sb = mx.mx_quantize(to_device_bits(b_bits, "bf16"), "e2m1", **cfg)
    oa, osa = orc.quantize(a_bits, "bf16", "e2m1", geometry="1x32", dim=-1, lane_stride=1, nibble_parity=1)
    ob, osb = orc.quantize(b_bits, "bf16", "e2m1", geometry="1x32", dim=-1, lane_stride=1, nibble_parity=1)
    torch.cuda.synchronize()
    assert np.array_equal(qa.cpu().numpy().reshape(oa.shape), oa)
    assert np.array_equal(sa.cpu().numpy().reshape(osa.shape), osa)
    c = mx.mx_scaled_matmul(qa.view(M, K // 2), qb.view(N, K // 2), sa.view(M, K // 32), sb.view(N, K // 32),
                            "e2m1", "f32")
    torch.cuda.synchronize()
    unpack = lambda q: np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)  # noqa: E731
    c_ref, s_ref = orc.scaled_matmul(unpack(oa), unpack(ob), osa, osb, "e2m1")
    check_gemm(c.cpu().numpy(), c_ref, s_ref, "f32")


def test_fp4_fused_equals_unfused(mx):
    import torch
    M, N, K = 512, 768, 1024
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=1)
    x = to_device_bits(x_bits, "bf16")
    cfg = dict(geometry="1x32", dim=-1, fp4_lane_stride=1, fp4_nibble_parity=1)
    wq, ws = mx.mx_quantize(to_device_bits(w_bits, "bf16"), "e2m1", scale_layout="sf", **cfg)
    fused = mx.mx_fused_quantize_matmul(x, wq.view(N, K // 2), ws, "e2m1", "bf16")
    xq, xs = mx.mx_quantize(x, "e2m1", scale_layout="sf", **cfg)
    ref = mx.mx_scaled_matmul(xq.view(M, K // 2), wq.view(N, K // 2), xs, ws, "e2m1", "bf16",
                              scales_are_sf_layout=True)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), ref.view(torch.int16))


def test_fp4_batched_dot(mx):
    import torch
    rng = np.random.default_rng(6)
    B, M, N, K = 3, 200, 136, 256
    a = rng.integers(0, 16, size=(B, M, K)).astype(np.uint8)
    bt = rng.integers(0, 16, size=(B, N, K)).astype(np.uint8)
    sa = rng.integers(112, 142, size=(B, M, K // 32)).astype(np.uint8)
    sb = rng.integers(112, 142, size=(B, N, K // 32)).astype(np.uint8)
    pa = np.stack([pack(a[i]) for i in range(B)])
    pb = np.stack([pack(bt[i]) for i in range(B)])
    got = mx.mx_block_scaled_dot(to_device_u8(pa), to_device_u8(pb), to_device_u8(sa), to_device_u8(sb), "e2m1",
                                 "f32", lhs_batch=(0,), rhs_batch=(0,))
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    for i in range(B):
        c_ref, s_ref = orc.scaled_matmul(a[i], bt[i], sa[i], sb[i], "e2m1")
        check_gemm(got[i], c_ref, s_ref, "f32")


def test_fp4_8192_sampled(mx):
    import torch
    M = N = K = 8192
    rng = np.random.default_rng(8)
    a = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    bt = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sa = rng.integers(118, 136, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(118, 136, size=(N, K // 32)).astype(np.uint8)
    c = mx.mx_scaled_matmul(to_device_u8(pack(a)), to_device_u8(pack(bt)), to_device_u8(sa), to_device_u8(sb),
                            "e2m1", "bf16")
    torch.cuda.synchronize()
    c = c.float().cpu().numpy()
    rows = np.unique(np.concatenate([rng.choice(M, 48, replace=False), [0, 255, 256, M - 1]]))
    cols = np.unique(np.concatenate([rng.choice(N, 48, replace=False), [0, 255, 256, N - 1]]))
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e2m1", rows=rows)
    check_gemm(c[rows], c_ref, s_ref, "bf16")
    c_ref, s_ref = orc.scaled_matmul(a, bt, sa, sb, "e2m1", cols=cols)
    check_gemm(c[:, cols], c_ref, s_ref, "bf16")
